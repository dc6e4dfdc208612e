// Lossless verification of a proposed block: the standard speculative-sampling
// rule (Leviathan et al. 2023; Chen et al. 2023), the consumer of the walk's q.
//
// verify_stats_kernel, one CTA per target position: one coalesced pass over
// the position's logits (16-byte vectors), in contiguous chunks of kVChunk
// elements; for each chunk the online-softmax partial in base 2 of
// x = logit * log2(e) / T' (chunk maximum m_c and s_c = sum 2^(x - m_c)) for
// the positions of sampled requests, or the chunk's argmax of the raw logits
// for greedy requests (each needs only its own statistic).  The pass is the
// whole HBM cost of the verification, and per element it is one multiply,
// one hardware exp2 and a few compares and adds: a divide and a natural-base
// expf per element made the first version arithmetic-bound at a sixth of HBM
// bandwidth.
//
// verify_decide_kernel, one CTA per request: combines the chunk partials into
// each position's maximum, normaliser and argmax (fixed order), takes the
// accept decisions slot by slot from values gathered in parallel, and draws
// the emitted token.  The residual draw max(0, p - qt) needs the cumulative
// mass by vocab index: the chunk partials give it per chunk without a second
// pass over the row (minus min(p, q) of the candidates in each chunk), and
// only the chunk holding the crossing is scanned element by element.
#include "common.cuh"

namespace dflash2 {
namespace {

constexpr int kVChunk = 4096;  // vocab elements per chunk (whole 16-byte vectors)
constexpr int kVThreads = 256;
constexpr int64_t kVMaxVocab = (int64_t)kVChunk * kVThreads;  // one decide thread per chunk
constexpr int kVMaxK = 128;
constexpr int kVMaxSlots = 64;  // slots * top_k <= 8192 entries staged in shared memory

struct ChunkStat {
    float m;    // sampled rows: max of x = logit * log2(e) / T' (-inf when empty)
    float s;    // sampled rows: sum of 2^(x - m)
    float v;    // greedy rows: max raw logit
    int32_t i;  // greedy rows: smallest index reaching v
};

// 2^x by the hardware approximation (relative error about 2^-22, flushing
// subnormal results to zero).  Every probability of the verification goes
// through it, so the chunk partials and the per-element values agree.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void combine_ms(float &m, float &s, float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) {
        m = m2;
        s = s2;
        return;
    }
    const float mm = fmaxf(m, m2);
    s = s * ex2(m - mm) + s2 * ex2(m2 - mm);
    m = mm;
}
__device__ __forceinline__ void combine_arg(float &v, int32_t &i, float v2, int32_t i2) {
    if (v2 > v || (v2 == v && i2 < i)) {
        v = v2;
        i = i2;
    }
}

template <typename T> __device__ __forceinline__ float ld_f(const T *p);
template <> __device__ __forceinline__ float ld_f<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}

// Folds n values into a lane's running softmax partial: the block maximum
// first, one rescale at most, then the terms.
template <int N>
__device__ __forceinline__ void fold_soft(const float (&l)[N], float c, float &m, float &s) {
    float x[N];
    float bm = -INFINITY;
#pragma unroll
    for (int q = 0; q < N; ++q) {
        x[q] = l[q] * c;
        bm = fmaxf(bm, x[q]);
    }
    if (bm == -INFINITY) return;
    if (bm > m) {
        s = m == -INFINITY ? 0.0f : s * ex2(m - bm);
        m = bm;
    }
#pragma unroll
    for (int q = 0; q < N; ++q) s += ex2(x[q] - m);
}

// Folds n values (indices idx0, idx0 + 1, ...) into a lane's running argmax;
// strict comparison keeps the first index of the lane's maximum.
template <int N>
__device__ __forceinline__ void fold_arg(const float (&l)[N], int32_t idx0, float &v, int32_t &i) {
#pragma unroll
    for (int q = 0; q < N; ++q)
        if (l[q] > v) {
            v = l[q];
            i = idx0 + q;
        }
}

template <typename T, int N>
__device__ __forceinline__ void unpack(const uint4 &u, float (&l)[N]) {
    const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
    for (int q = 0; q < N; ++q) l[q] = ld_f(e + q);
}

template <typename T, bool GREEDY>
__device__ __forceinline__ void stats_chunk(const T *lr, int64_t c0, int64_t c1, bool vec, float c,
                                            int lane, ChunkStat &out) {
    constexpr int kVec = 16 / sizeof(T);
    float m = -INFINITY, s = 0.0f, v = -INFINITY;
    int32_t i = INT32_MAX;
    if (vec) {
        // chunk starts and vocab are multiples of kVec: whole 16-byte vectors
        const uint4 *p4 = reinterpret_cast<const uint4 *>(lr + c0);
        const int nv = (int)((c1 - c0) / kVec);
        int j = lane;
        for (; j + 96 < nv; j += 128) {  // four loads in flight per lane
            uint4 u[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) u[t] = __ldg(p4 + j + 32 * t);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                float l[kVec];
                unpack<T>(u[t], l);
                if (GREEDY) fold_arg(l, (int32_t)(c0 + (int64_t)(j + 32 * t) * kVec), v, i);
                else fold_soft(l, c, m, s);
            }
        }
        for (; j < nv; j += 32) {
            float l[kVec];
            unpack<T>(__ldg(p4 + j), l);
            if (GREEDY) fold_arg(l, (int32_t)(c0 + (int64_t)j * kVec), v, i);
            else fold_soft(l, c, m, s);
        }
    } else {
        for (int64_t y = c0 + lane; y < c1; y += 32) {
            const float l[1] = {ld_f(lr + y)};
            if (GREEDY) fold_arg(l, (int32_t)y, v, i);
            else fold_soft(l, c, m, s);
        }
    }
    // lanes hold interleaved indices: combine by value, smallest index on ties
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        if (GREEDY) {
            const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, o);
            const int32_t i2 = __shfl_xor_sync(0xFFFFFFFFu, i, o);
            combine_arg(v, i, v2, i2);
        } else {
            const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
            const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
            combine_ms(m, s, m2, s2);
        }
    }
    out = ChunkStat{m, s, v, i};
}

template <typename T>
__global__ void __launch_bounds__(kVThreads)
    verify_stats_kernel(const T *__restrict__ logits, int64_t vocab, int32_t n_chunks,
                        int32_t slots1, const float *__restrict__ temperatures,
                        const uint8_t *__restrict__ greedy, bool vec, ChunkStat *stats) {
    grid_dep_wait();
    const int64_t row = blockIdx.x;  // one target position; blockIdx.y splits its chunks
    const int b = (int)(row / slots1);
    const bool is_greedy = greedy[b] != 0;
    const float c = 1.4426950408889634f / fmaxf(temperatures[b], 1e-5f);  // log2(e) / T'
    const T *lr = logits + row * vocab;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the position's chunks are spread over the warps of gridDim.y CTAs
    const int gw = blockIdx.y * (kVThreads / 32) + warp;
    const int nw = gridDim.y * (kVThreads / 32);
    for (int ch = gw; ch < n_chunks; ch += nw) {
        const int64_t c0 = (int64_t)ch * kVChunk;
        const int64_t c1 = min(vocab, c0 + kVChunk);
        ChunkStat st;
        if (is_greedy) stats_chunk<T, true>(lr, c0, c1, vec, c, lane, st);
        else stats_chunk<T, false>(lr, c0, c1, vec, c, lane, st);
        if (lane == 0) stats[row * n_chunks + ch] = st;
    }
}

struct DecideShared {
    float m[kVMaxSlots + 1], z[kVMaxSlots + 1];
    int32_t am[kVMaxSlots + 1];
    int32_t kpos[kVMaxSlots];
    int64_t dr[kVMaxSlots];
    float lx[kVMaxSlots], qx[kVMaxSlots];
    int64_t cy[kVMaxK];     // candidate target ids of the final position
    float cmin[kVMaxK];     // min(p, q) of those candidates
    float corr[kVChunk];    // min(p, q) at the crossing chunk's candidate positions
    float part[kVThreads];
    int32_t pidx[kVThreads];
    int32_t final_pos, accepted, bad, chunk_star, t_star, fallback;
    float rem, rem2;
    int64_t emit;
};

// Warp 0 of the block: the first index t in [0, n) (n <= 256) where the
// running sum of vals passes `target` (entries <= 0 skipped), and the mass
// still to pass inside it.  Each lane sums 8 consecutive entries, a shuffle
// scan gives the lanes' prefixes, and the first lane whose prefix passes walks
// its entries.  With no crossing (rounding at the very top) it returns the
// last positive entry.  Fixed order: deterministic.
__device__ __forceinline__ void warp_find_crossing(const float *vals, int n, float target, int lane,
                                                   int32_t *t_out, float *rem_out) {
    float loc[8];
    float tot = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int t = lane * 8 + j;
        loc[j] = t < n ? fmaxf(vals[t], 0.0f) : 0.0f;
        tot += loc[j];
    }
    float inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += y;
    }
    const float exc = inc - tot;
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, tot > 0.0f && inc > target);
    const uint32_t pos = __ballot_sync(0xFFFFFFFFu, tot > 0.0f);
    const int lead = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    if (lead < 0) {
        if (lane == 0) {
            *t_out = -1;
            *rem_out = 0.0f;
        }
        return;
    }
    if (lane == lead) {
        float acc = exc;
        int32_t ts = -1;
        for (int j = 0; j < 8; ++j) {
            if (loc[j] > 0.0f) {
                ts = lane * 8 + j;
                if (acc + loc[j] > target) break;
                acc += loc[j];
            }
        }
        *t_out = ts;
        *rem_out = target - acc;
    }
}

// p(y) of the final position in the same base-2 form as the partials.
template <typename T>
__device__ __forceinline__ float prob(const T *lr, int64_t y, float c, float m, float z) {
    return ex2(ld_f(lr + y) * c - m) / z;
}

template <typename T>
__global__ void __launch_bounds__(kVThreads)
    verify_decide_kernel(const T *__restrict__ logits, int64_t vocab, int32_t n_chunks,
                         int32_t slots, int32_t k, const ChunkStat *__restrict__ stats,
                         const float *__restrict__ temperatures, const uint8_t *__restrict__ greedy,
                         const int64_t *__restrict__ draft, const int64_t *__restrict__ cand,
                         const float *__restrict__ q, const float *__restrict__ r,
                         int64_t *accept_len, int64_t *out_tokens, int32_t *err) {
    grid_dep_wait();
    __shared__ DecideShared sh;
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const int slots1 = slots + 1;
    const float c = 1.4426950408889634f / fmaxf(temperatures[b], 1e-5f);  // log2(e) / T'
    const bool is_greedy = greedy[b] != 0;

    // (1) per position: maximum, normaliser and argmax from the chunk partials,
    // one warp per position (lanes load chunks in parallel, a fixed shuffle tree
    // combines them)
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int pos = warp; pos < slots1; pos += kVThreads / 32) {
            const ChunkStat *cs = stats + ((int64_t)b * slots1 + pos) * n_chunks;
            float m = -INFINITY, s = 0.0f, v = -INFINITY;
            int32_t i = INT32_MAX;
            for (int ch = lane; ch < n_chunks; ch += 32) {
                const ChunkStat x = cs[ch];
                combine_ms(m, s, x.m, x.s);
                combine_arg(v, i, x.v, x.i);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
                const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
                const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, o);
                const int32_t i2 = __shfl_xor_sync(0xFFFFFFFFu, i, o);
                combine_ms(m, s, m2, s2);
                combine_arg(v, i, v2, i2);
            }
            if (lane == 0) {
                sh.m[pos] = m;
                sh.z[pos] = s;
                sh.am[pos] = i;
            }
        }
    }
    if (tid < slots) sh.kpos[tid] = k;  // k = not found
    if (tid == 0) sh.bad = 0;
    __syncthreads();
    // (2) every slot's draft, candidates and q in shared memory (one round of
    // loads, independent of the decisions), then which candidate each draft is
    // (ids are distinct within a slot)
    extern __shared__ __align__(16) uint8_t dyn[];
    const int sk = slots * k;
    int64_t *s_cand = reinterpret_cast<int64_t *>(dyn);
    float *s_q = reinterpret_cast<float *>(s_cand + sk);
    float *s_lc = s_q + sk;  // sampled rows: the logit at every candidate
    for (int idx = tid; idx < sk; idx += kVThreads) {
        s_cand[idx] = cand[(int64_t)b * sk + idx];
        s_q[idx] = q[(int64_t)b * sk + idx];
    }
    if (tid < slots) sh.dr[tid] = draft[(int64_t)b * slots + tid];
    __syncthreads();
    for (int idx = tid; idx < sk; idx += kVThreads) {
        const int s = idx / k, j = idx - s * k;
        const int64_t y = s_cand[idx];
        if (y == sh.dr[s]) atomicMin(&sh.kpos[s], j);
        // the second round of loads: logits at the candidates (sampled rows)
        if (!is_greedy)
            s_lc[idx] = (y >= 0 && y < vocab) ? ld_f(logits + ((int64_t)b * slots1 + s) * vocab + y)
                                               : -INFINITY;
    }
    __syncthreads();
    if (tid < slots) {
        const int64_t x = sh.dr[tid];
        const int kp = sh.kpos[tid];
        if (kp >= k || x < 0 || x >= vocab) {
            sh.bad = 1;
            sh.lx[tid] = 0.0f;
            sh.qx[tid] = 0.0f;
        } else {
            sh.lx[tid] = is_greedy ? 0.0f : s_lc[tid * k + kp];
            sh.qx[tid] = s_q[tid * k + kp];
        }
    }
    __syncthreads();
    // (3) accept decisions, slot by slot
    if (tid == 0) {
        int s = 0;
        bool rejected = false;
        for (; s < slots; ++s) {
            bool acc;
            if (is_greedy) {
                acc = (int64_t)sh.am[s] == sh.dr[s];
            } else {
                const float px = ex2(sh.lx[s] * c - sh.m[s]) / sh.z[s];
                acc = r[(int64_t)b * slots1 + s] * sh.qx[s] < px;
            }
            if (!acc) {
                rejected = true;
                break;
            }
        }
        sh.accepted = s;
        sh.final_pos = rejected ? s : slots;
        sh.emit = -1;
    }
    __syncthreads();
    const int f = sh.final_pos;
    if (sh.bad) {
        for (int j = tid; j < slots1; j += kVThreads) out_tokens[(int64_t)b * slots1 + j] = -1;
        if (tid == 0) {
            accept_len[b] = 0;
            if (err) atomicOr(err, DFLASH2_DEVERR_ID_RANGE);
        }
        return;
    }
    const T *lr = logits + ((int64_t)b * slots1 + f) * vocab;
    if (!is_greedy) {
        const float mf = sh.m[f], zf = sh.z[f];
        const int kk = f < slots ? k : 0;  // a rejection: residual max(0, p - qt)
        // (4) min(p, q) of the final position's candidates
        if (tid < kk) {
            const int64_t y = s_cand[f * k + tid];
            const float ly = s_lc[f * k + tid];
            const float py = ly == -INFINITY ? 0.0f : ex2(ly * c - mf) / zf;
            sh.cy[tid] = y;
            sh.cmin[tid] = fminf(py, s_q[f * k + tid]);
        }
        __syncthreads();
        // (5) residual mass per chunk from the partials (one thread per chunk,
        // candidates in index order), then thread 0 finds the chunk where the
        // cumulative residual passes u * total
        if (tid < n_chunks) {
            const ChunkStat x = stats[((int64_t)b * slots1 + f) * n_chunks + tid];
            float rc = x.m == -INFINITY ? 0.0f : x.s * ex2(x.m - mf) / zf;
            for (int j = 0; j < kk; ++j)
                if (sh.cy[j] >= 0 && sh.cy[j] / kVChunk == tid) rc -= sh.cmin[j];
            sh.part[tid] = fmaxf(rc, 0.0f);
        }
        __syncthreads();
        if (tid < 32) {
            float tot = 0.0f;
            for (int ch = tid; ch < n_chunks; ch += 32) tot += sh.part[ch];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
            tot = __shfl_sync(0xFFFFFFFFu, tot, 0);  // one value for every lane
            const float target = r[(int64_t)b * slots1 + slots] * tot;
            warp_find_crossing(sh.part, n_chunks, target, tid, &sh.chunk_star, &sh.rem);
        }
        __syncthreads();
        // no residual mass at all cannot follow a rejection in exact arithmetic;
        // should rounding produce it, emit the most likely token
        if (tid == 0) sh.fallback = sh.chunk_star < 0;
        __syncthreads();
        for (int e = tid; e < kVChunk; e += kVThreads) sh.corr[e] = 0.0f;
        __syncthreads();
        const int cstar = sh.chunk_star;
        if (cstar >= 0) {
            const int64_t c0 = (int64_t)cstar * kVChunk;
            const int len = (int)(min(vocab, c0 + kVChunk) - c0);
            if (tid < kk && sh.cy[tid] >= c0 && sh.cy[tid] < c0 + len)
                sh.corr[sh.cy[tid] - c0] = sh.cmin[tid];  // distinct ids: no two writers
            __syncthreads();
            // (6) the chunk's residual values in shared memory: coalesced loads,
            // then contiguous segments of kSeg per thread
            float pe[kVChunk / kVThreads];  // all loads issued before any use
#pragma unroll
            for (int it = 0; it < kVChunk / kVThreads; ++it) {
                const int e = tid + it * kVThreads;
                pe[it] = e < len ? ld_f(lr + c0 + e) : -INFINITY;
            }
#pragma unroll
            for (int it = 0; it < kVChunk / kVThreads; ++it) {
                const int e = tid + it * kVThreads;
                const float pv = pe[it] == -INFINITY ? 0.0f : ex2(pe[it] * c - mf) / zf;
                sh.corr[e] = fmaxf(pv - sh.corr[e], 0.0f);  // p - min(p, q) >= 0
            }
            __syncthreads();
            constexpr int kSeg = kVChunk / kVThreads;
            float mine = 0.0f;
#pragma unroll
            for (int e = 0; e < kSeg; ++e) mine += sh.corr[tid * kSeg + e];
            sh.part[tid] = mine;
            __syncthreads();
            if (tid < 32) warp_find_crossing(sh.part, kVThreads, sh.rem, tid, &sh.t_star, &sh.rem2);
            __syncthreads();
            if (tid == 0 && sh.t_star < 0) sh.fallback = 1;  // rounding left the chunk empty
            __syncthreads();
            if (tid == sh.t_star) {
                const float rem = sh.rem2;
                float acc = 0.0f;
                int64_t pick = -1;
                for (int e = tid * kSeg; e < tid * kSeg + kSeg; ++e) {
                    const float res = sh.corr[e];
                    if (res > 0.0f) {
                        pick = c0 + e;
                        if (acc + res > rem) break;
                        acc += res;
                    }
                }
                sh.emit = pick;
            }
        }
        __syncthreads();
        if (sh.fallback) {
            // the most likely token of the position: the largest logit (smallest
            // index on ties) inside the chunk with the largest partial maximum
            if (tid == 0) {
                const ChunkStat *cs = stats + ((int64_t)b * slots1 + f) * n_chunks;
                int best = 0;
                for (int ch = 1; ch < n_chunks; ++ch)
                    if (cs[ch].m > cs[best].m) best = ch;
                sh.chunk_star = best;
            }
            __syncthreads();
            const int64_t c0 = (int64_t)sh.chunk_star * kVChunk;
            const int64_t c1 = min(vocab, c0 + kVChunk);
            float v = -INFINITY;
            int32_t i = INT32_MAX;
            for (int64_t y = c0 + tid; y < c1; y += kVThreads) {
                const float l = ld_f(lr + y);
                if (l > v) {
                    v = l;
                    i = (int32_t)y;
                }
            }
            sh.part[tid] = v;
            sh.pidx[tid] = i;
            __syncthreads();
            if (tid == 0) {
                for (int t = 1; t < kVThreads; ++t) combine_arg(v, i, sh.part[t], sh.pidx[t]);
                sh.emit = i;
            }
        }
        __syncthreads();
    } else if (tid == 0) {
        sh.emit = sh.am[f];
    }
    __syncthreads();
    // (7) outputs
    const int na = sh.accepted;
    for (int j = tid; j < slots1; j += kVThreads) {
        int64_t v = -1;
        if (j < na) v = sh.dr[j];
        else if (j == na) v = sh.emit;
        out_tokens[(int64_t)b * slots1 + j] = v;
    }
    if (tid == 0) accept_len[b] = na;
}

inline int32_t verify_chunks(int64_t vocab) { return (int32_t)((vocab + kVChunk - 1) / kVChunk); }

bool g_verify_attr[64];

}  // namespace
}  // namespace dflash2

using namespace dflash2;

extern "C" size_t dflash2_verify_workspace_size(int32_t batch, int32_t slots, int64_t vocab) {
    if (batch <= 0 || slots < 0 || vocab <= 0 || vocab > kVMaxVocab) return 0;
    return (size_t)batch * (slots + 1) * verify_chunks(vocab) * sizeof(ChunkStat);
}

extern "C" dflash2_status dflash2_verify(const void *target_logits, int64_t vocab,
                                         const float *temperatures, const uint8_t *greedy,
                                         const int64_t *draft, const int64_t *cand,
                                         const float *q, const float *uniforms, int32_t batch,
                                         int32_t slots, int32_t top_k, int32_t dtype,
                                         int64_t *accept_len, int64_t *out_tokens,
                                         void *workspace, size_t ws_bytes, int32_t *err_word,
                                         void *stream) {
    if (dtype != DFLASH2_F32 && dtype != DFLASH2_BF16) return DFLASH2_ERR_UNSUPPORTED_DTYPE;
    if (batch < 0 || slots < 0 || slots > kVMaxSlots || top_k <= 0 || top_k > kVMaxK ||
        vocab <= 0 || vocab > kVMaxVocab)
        return DFLASH2_ERR_INVALID_ARG;
    if (batch == 0) return DFLASH2_OK;
    if (!target_logits || !temperatures || !greedy || !uniforms || !accept_len || !out_tokens ||
        (slots > 0 && (!draft || !cand || !q)))
        return DFLASH2_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < dflash2_verify_workspace_size(batch, slots, vocab))
        return DFLASH2_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(accept_len) | reinterpret_cast<uintptr_t>(out_tokens) |
         reinterpret_cast<uintptr_t>(draft) | reinterpret_cast<uintptr_t>(cand)) % 8 != 0 ||
        (reinterpret_cast<uintptr_t>(temperatures) | reinterpret_cast<uintptr_t>(q) |
         reinterpret_cast<uintptr_t>(uniforms)) % 4 != 0)
        return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    dflash2_status s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int32_t n_chunks = verify_chunks(vocab);
    const size_t esz = dtype == DFLASH2_BF16 ? 2 : 4;
    // whole 16-byte vectors in every row and chunk
    const bool vec = reinterpret_cast<uintptr_t>(target_logits) % 16 == 0 &&
                     (vocab * (int64_t)esz) % 16 == 0;
    const int64_t rows = (int64_t)batch * (slots + 1);
    ChunkStat *stats = static_cast<ChunkStat *>(workspace);
    // enough CTAs to keep every SM's loads in flight: split a position's chunks
    // over up to 4 CTAs while positions alone fill fewer than 8 CTAs per SM
    int splits = 1;
    while (splits < 4 && rows * splits < (int64_t)di.sm_count * 8 &&
           (int64_t)(splits * 2) * (kVThreads / 32) <= n_chunks)
        splits *= 2;
    const dim3 sgrid((unsigned)rows, (unsigned)splits);
    const size_t dsm = (size_t)slots * top_k * (8 + 4 + 4);  // staged candidates, q, logits
    if (di.device >= 0 && di.device < 64 && !g_verify_attr[di.device]) {
        if (cudaFuncSetAttribute(verify_decide_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024) !=
                cudaSuccess ||
            cudaFuncSetAttribute(verify_decide_kernel<float>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024) !=
                cudaSuccess) {
            cudaGetLastError();
            return DFLASH2_ERR_CUDA;
        }
        g_verify_attr[di.device] = true;
    }
    if (dtype == DFLASH2_BF16) {
        const auto *lg = static_cast<const __nv_bfloat16 *>(target_logits);
        launch_k(verify_stats_kernel<__nv_bfloat16>, sgrid, kVThreads, 0, st, lg, vocab, n_chunks,
            slots + 1, temperatures, greedy, vec, stats);
        launch_k(verify_decide_kernel<__nv_bfloat16>, (unsigned)batch, kVThreads, dsm, st, lg,
            vocab, n_chunks, slots, top_k, stats, temperatures, greedy, draft, cand, q,
            uniforms, accept_len, out_tokens, err_word);
    } else {
        const auto *lg = static_cast<const float *>(target_logits);
        launch_k(verify_stats_kernel<float>, sgrid, kVThreads, 0, st, lg, vocab, n_chunks,
            slots + 1, temperatures, greedy, vec, stats);
        launch_k(verify_decide_kernel<float>, (unsigned)batch, kVThreads, dsm, st, lg, vocab,
            n_chunks, slots, top_k, stats, temperatures, greedy, draft, cand, q,
            uniforms, accept_len, out_tokens, err_word);
    }
    return launch_status();
}
