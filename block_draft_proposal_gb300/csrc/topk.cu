// Unary candidates: lm_head GEMM + softcap transform + padded-vocab mask +
// per-row top-K (sglang DFlash2 PR: compute_candidates, _transform_unary_logits,
// _radix_topk; vLLM DSpark padded-vocab review: mask [target_vocab, draft_vocab)).
//
// bf16 pipeline (four launches, no full logit matrix in HBM):
//   1. pilot GEMM: the raw logits of weight units spread over the vocab
//      (about a sixteenth of it, 8192 rows at most) are written to the
//      workspace;
//   2. pilot select: per row, the pilot's keys are formed with the same
//      transform as the filter epilogue; the K-th largest of the per-thread
//      maxima is at most the pilot's K-th best (u, id) key, itself at most the
//      row's true K-th best key (the K-th best of a subset), so it is a safe
//      threshold; every pilot key that reaches it seeds the candidate list;
//   3. filter GEMM over the remaining tiles: the epilogue appends every key
//      that reaches the threshold to the row's candidate list;
//   4. finalize: the same maxima threshold cuts each row's candidates to a
//      few more than K, which are sorted exactly (the radix select remains
//      for a row where more than kCollect keys reach it).  A row
//      whose list overflowed is recomputed exactly on CUDA cores (rare: only
//      adversarial weights defeat the pilot threshold).
// Steps 1-3 also run as one cooperative launch (gemm_tc.cu, fused mode) where
// the host's rule (use_fused) expects it to be faster: the pilot tiles come
// first, their epilogues write 32-row group maxima, the epilogue warps then
// take each row's threshold from those maxima, and the pilot tiles' own
// candidates come from the accumulators they kept.
// FP8 head (dflash2_unary_topk_fp8): the tokens' E4M3 codes and scales
// (quant.cu), then the same pipeline on kind::f8f6f4 MMAs with the logits
// scaled in the epilogue.
// fp32 pipeline: the same exact CUDA-core routine as the overflow path, one
// CTA per row, or per (row, vocab chunk) with the chunk lists merged exactly
// (merge.cu) when the caller passes the recommended workspace.
//
// Keys order (u descending, id ascending) as one uint64 (common.cuh), so the
// selection is a plain "K largest keys" problem with no ties.
#include "kernels.h"

#include <atomic>

#include <algorithm>
#include <type_traits>

namespace dflash2 {
namespace {

constexpr int kSelThreads = 256;
constexpr int kMaxTopK = 128;
constexpr int kMaxCandCap = 16384;
constexpr int kSmemKeys = 4096;     // candidate keys staged in shared memory
constexpr int kDirectBuf = 2048;    // keys buffered by the exact CUDA-core path
constexpr int kDirectRows = 64;     // vocab rows per buffered batch (8 warps x 8)

struct SelectShared {
    uint32_t hist[256];
    uint32_t bcast[4];
    uint32_t count;
    uint64_t top[kMaxTopK];
    uint64_t sort[kSelThreads];   // per-thread maxima, sorted
};

constexpr int kCollect = 512;  // keys at or above the maxima threshold sorted in shared memory

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
    const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, (uint32_t)v, m);
    const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, (uint32_t)(v >> 32), m);
    return ((uint64_t)hi << 32) | lo;
}

// Sorts the warp's 32 values (one per lane) descending by shuffles; lane i
// ends with the i-th largest.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint64_t other = shfl_xor_u64(v, stride);
            const bool desc = (lane & size) == 0 || size == 32;
            const bool lower = (lane & stride) == 0;
            v = (lower == desc) ? (v > other ? v : other) : (v < other ? v : other);
        }
    }
    return v;
}

// The k-th largest (1 <= k <= kSelThreads) of one float per thread, by the
// same bitonic scheme as block_kth_of_maxima (floats, no NaN).
__device__ float block_kth_of_maxima_f(float tmax, int k, float *s) {
    const int t = threadIdx.x;
    float v = tmax;
#pragma unroll 1
    for (int size = 2; size <= kSelThreads; size <<= 1) {
#pragma unroll 1
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            float other;
            if (stride >= 32) {
                s[t] = v;
                __syncthreads();
                other = s[t ^ stride];
                __syncthreads();
            } else {
                other = __shfl_xor_sync(0xFFFFFFFFu, v, stride);
            }
            const bool desc = (t & size) == 0;
            const bool lower = (t & stride) == 0;
            v = (lower == desc) ? fmaxf(v, other) : fminf(v, other);
        }
    }
    s[t] = v;
    __syncthreads();
    const float r = s[k - 1];
    __syncthreads();
    return r;
}

// The k-th largest (1 <= k <= kSelThreads) of the block's per-thread values
// tmax (one per thread), by a bitonic sort of kSelThreads elements: warp
// shuffles for strides below 32, shared memory for the others.  Every thread
// gets the result.  Used as a threshold: when each thread's value is the
// largest of the keys it holds, the k-th largest of these maxima is at most
// the k-th largest key of the block (k distinct keys reach it), and with many
// more threads than k it is rarely much lower.
__device__ uint64_t block_kth_of_maxima(uint64_t tmax, int k, SelectShared &sh) {
    const int t = threadIdx.x;
    uint64_t v = tmax;
#pragma unroll 1
    for (int size = 2; size <= kSelThreads; size <<= 1) {
#pragma unroll 1
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            uint64_t other;
            if (stride >= 32) {
                sh.sort[t] = v;
                __syncthreads();
                other = sh.sort[t ^ stride];
                __syncthreads();
            } else {
                other = shfl_xor_u64(v, stride);
            }
            const bool desc = (t & size) == 0;   // this block of `size` sorts descending
            const bool lower = (t & stride) == 0;
            v = (lower == desc) ? (v > other ? v : other) : (v < other ? v : other);
        }
    }
    sh.sort[t] = v;  // descending
    __syncthreads();
    const uint64_t r = sh.sort[k - 1];
    __syncthreads();
    return r;
}

// Sorts a[0, n) descending in place (n a power of two, at most 2 * kSelThreads
// per pass of the threads); all threads call it.
__device__ void block_sort_desc(uint64_t *a, int n) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int j = i ^ stride;
                if (j > i) {
                    const uint64_t x = a[i], y = a[j];
                    const bool desc = (i & size) == 0;
                    if (desc ? (x < y) : (x > y)) {
                        a[i] = y;
                        a[j] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// Exact k-th largest of keys[0, n) (1 <= k <= n), by 8-bit radix passes from
// the top byte.  All threads of the block call it; every thread gets the
// result.  keys may live in shared or global memory.
__device__ uint64_t block_kth_largest(const uint64_t *keys, int n, int k, SelectShared &sh) {
    uint64_t prefix = 0, mask = 0;
    uint32_t remaining = (uint32_t)k;
    const int lane = threadIdx.x & 31;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) sh.hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const uint64_t key = keys[i];
            if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            uint32_t c[8], tot = 0;
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                c[b] = sh.hist[lane * 8 + b];
                tot += c[b];
            }
            uint32_t suf = tot;  // keys in bins of this lane and all higher lanes
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, suf, o);
                if (lane + o < 32) suf += y;
            }
            const uint32_t above = suf - tot;
            if (above < remaining && remaining <= above + tot) {
                uint32_t acc = above;
                for (int b = 7; b >= 0; --b) {
                    if (acc + c[b] >= remaining) {
                        sh.bcast[0] = (uint32_t)(lane * 8 + b);
                        sh.bcast[1] = remaining - acc;
                        sh.bcast[2] = c[b];
                        break;
                    }
                    acc += c[b];
                }
            }
        }
        __syncthreads();
        const uint32_t digit = sh.bcast[0];
        remaining = sh.bcast[1];
        const uint32_t in_bin = sh.bcast[2];
        prefix |= (uint64_t)digit << shift;
        mask |= (uint64_t)0xFFu << shift;
        __syncthreads();
        if (in_bin == 1 && shift > 0) {
            // one key carries this prefix: it is the answer
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const uint64_t key = keys[i];
                if ((key & mask) == prefix) sh.bcast[3] = i;
            }
            __syncthreads();
            const uint64_t kth = keys[sh.bcast[3]];
            __syncthreads();
            return kth;
        }
    }
    return prefix;
}

// Collects the keys >= kth (nonzero) into sh.top (at most k of them), sorts
// them descending and returns how many there are.
__device__ int block_collect_sorted(const uint64_t *keys, int n, uint64_t kth, int k,
                                    SelectShared &sh) {
    if (threadIdx.x == 0) sh.count = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const uint64_t key = keys[i];
        if (key != 0 && key >= kth) {
            const uint32_t slot = atomicAdd(&sh.count, 1u);
            if (slot < (uint32_t)k) sh.top[slot] = key;
        }
    }
    __syncthreads();
    const int got = min((int)sh.count, k);
    int kpad = 1;
    while (kpad < k) kpad <<= 1;
    for (int i = got + threadIdx.x; i < kpad; i += blockDim.x) sh.top[i] = 0;
    __syncthreads();
    for (int size = 2; size <= kpad; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < kpad; i += blockDim.x) {
                const int j = i ^ stride;
                if (j > i) {
                    const uint64_t a = sh.top[i], b = sh.top[j];
                    const bool desc = (i & size) == 0;
                    if (desc ? (a < b) : (a > b)) {
                        sh.top[i] = b;
                        sh.top[j] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    return got;
}

__device__ void write_row(const SelectShared &sh, int got, int k, int64_t row, int64_t *ids,
                          float *vals, int32_t *err) {
    for (int i = threadIdx.x; i < k; i += blockDim.x) {
        if (i < got) {
            ids[row * k + i] = (int64_t)key_id(sh.top[i]);
            vals[row * k + i] = key_u(sh.top[i]);
        } else {
            ids[row * k + i] = 0;
            vals[row * k + i] = -INFINITY;
        }
    }
    if (got < k && threadIdx.x == 0 && err) atomicOr(err, DFLASH2_DEVERR_SHORT);
}

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}
template <> __device__ __forceinline__ float to_f<__nv_fp8_e4m3>(__nv_fp8_e4m3 v) {
    return static_cast<float>(v);
}

// Exact top-k of one row on CUDA cores: every vocab row's u is computed in
// fp32 (lane-strided FMA over hidden, then a warp tree sum), keys that reach
// the running threshold are buffered in shared memory, and a full buffer is
// cut back to its k best (whose k-th key becomes the new threshold).  Leaves
// the sorted result in sh.top and returns how many keys it holds.
// With w_scale (fp8 codes), the dot product is scaled by a_scale * w_scale[v],
// the expression the tensor-core epilogue uses.
template <typename T>
__device__ int direct_row_topk(const T *__restrict__ hrow, const T *__restrict__ w, int hidden,
                               int64_t draft_vocab, int64_t target_vocab, float mult, float cap,
                               int k, float *hs, uint64_t *buf, SelectShared &sh,
                               const float *__restrict__ w_scale = nullptr,
                               float a_scale = 1.0f) {
    for (int j = threadIdx.x; j < hidden; j += blockDim.x) hs[j] = to_f(hrow[j]);
    if (threadIdx.x == 0) sh.count = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int64_t vmax = draft_vocab < target_vocab ? draft_vocab : target_vocab;
    uint64_t theta = 0;
    for (int64_t v0 = 0; v0 < vmax; v0 += kDirectRows) {
        for (int r = warp; r < kDirectRows; r += nwarps) {
            const int64_t v = v0 + r;
            if (v >= vmax) break;
            const T *wr = w + v * hidden;
            float acc = 0.0f;
            for (int j = lane; j < hidden; j += 32) acc = fmaf(hs[j], to_f(wr[j]), acc);
            acc = warp_sum(acc);
            if (w_scale) acc *= a_scale * __ldg(w_scale + v);
            if (lane == 0) {
                const uint64_t key = make_key(unary_transform(acc, mult, cap), (uint32_t)v);
                if (key >= theta) {
                    const uint32_t slot = atomicAdd(&sh.count, 1u);
                    buf[slot] = key;  // slot < kDirectBuf: the buffer is cut below
                }
            }
        }
        __syncthreads();
        const int n = (int)sh.count;
        if (n > kDirectBuf - kDirectRows && n > k) {
            const uint64_t kth = block_kth_largest(buf, n, k, sh);
            const int got = block_collect_sorted(buf, n, kth, k, sh);
            for (int i = threadIdx.x; i < got; i += blockDim.x) buf[i] = sh.top[i];
            theta = kth;
            __syncthreads();
            if (threadIdx.x == 0) sh.count = (uint32_t)got;
            __syncthreads();
        }
    }
    const int n = (int)sh.count;
    const uint64_t kth = n > k ? block_kth_largest(buf, n, k, sh) : 1;
    return block_collect_sorted(buf, n, kth, k, sh);
}

// NVFP4 operands: packed E2M1 codes (two per byte, element 2i in the low
// nibble) with one E4M3 scale per 16 elements and an fp32 second-level scale
// (per row of h, one for the weights).
struct E2M1x2 {
    uint8_t bits;
};
struct NvScales {
    const uint8_t *sfh;        // [rows][hidden / 16]
    const uint8_t *sfw_tiles;  // the weights' scale tiles (blocks of 128 rows)
    const uint8_t *sfh_tiles;  // the tokens' scale tiles (blocks of the token tile)
    float w_global;
};
__device__ __forceinline__ float e2m1_value(uint32_t c) {
    const float m = (c & 1u) ? 1.5f : 1.0f;  // magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6
    const uint32_t e = (c >> 1) & 3u;
    const float v = e == 0 ? 0.5f * (float)(c & 1u) : m * (float)(1u << (e - 1));
    return (c & 8u) ? -v : v;
}
__device__ __forceinline__ float e4m3_value(uint8_t c) {
    __nv_fp8_e4m3 v;
    v.__x = c;
    return static_cast<float>(v);
}
__device__ __forceinline__ float nv_elem(const uint8_t *codes, const uint8_t *sf, int j) {
    const uint32_t b = codes[j >> 1];
    return e2m1_value((j & 1) ? b >> 4 : b & 15u) * e4m3_value(sf[j >> 4]);
}
// Scale of element j of weight row v, from scale tiles of 128-row blocks.
__device__ __forceinline__ uint8_t tiled_scale(const uint8_t *tiles, int64_t v, int j, int nw8) {
    const int64_t rb = v >> 7;
    const int rl = (int)(v & 127), b = j >> 4;
    return tiles[(rb * nw8 + (b >> 2)) * 512 + (rl & 31) * 16 + (rl >> 5) * 4 + (b & 3)];
}

// The exact top-k of one row for NVFP4 operands: as direct_row_topk, on the
// block-scaled values (code times block scale, exact in fp32) and the
// epilogue's second-level scale a_scale * w_global.
__device__ int direct_row_topk_nvfp4(const uint8_t *__restrict__ hrow,
                                     const uint8_t *__restrict__ sfh_row,
                                     const uint8_t *__restrict__ w,
                                     const uint8_t *__restrict__ sfw_tiles, int hidden,
                                     int64_t draft_vocab, int64_t target_vocab, float mult,
                                     float cap, int k, float *hs, uint64_t *buf, SelectShared &sh,
                                     float scale) {
    for (int j = threadIdx.x; j < hidden; j += blockDim.x) hs[j] = nv_elem(hrow, sfh_row, j);
    if (threadIdx.x == 0) sh.count = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int64_t vmax = draft_vocab < target_vocab ? draft_vocab : target_vocab;
    const int nw8 = (hidden / 64 + 7) / 8 * 8;
    uint64_t theta = 0;
    for (int64_t v0 = 0; v0 < vmax; v0 += kDirectRows) {
        for (int r = warp; r < kDirectRows; r += nwarps) {
            const int64_t v = v0 + r;
            if (v >= vmax) break;
            const uint8_t *wr = w + v * (hidden / 2);
            float acc = 0.0f;
            for (int j = lane; j < hidden; j += 32) {
                const uint32_t b = wr[j >> 1];
                const float wv = e2m1_value((j & 1) ? b >> 4 : b & 15u) *
                                 e4m3_value(tiled_scale(sfw_tiles, v, j, nw8));
                acc = fmaf(hs[j], wv, acc);
            }
            acc = warp_sum(acc);
            acc *= scale;
            if (lane == 0) {
                const uint64_t key = make_key(unary_transform(acc, mult, cap), (uint32_t)v);
                if (key >= theta) {
                    const uint32_t slot = atomicAdd(&sh.count, 1u);
                    buf[slot] = key;
                }
            }
        }
        __syncthreads();
        const int n = (int)sh.count;
        if (n > kDirectBuf - kDirectRows && n > k) {
            const uint64_t kth = block_kth_largest(buf, n, k, sh);
            const int got = block_collect_sorted(buf, n, kth, k, sh);
            for (int i = threadIdx.x; i < got; i += blockDim.x) buf[i] = sh.top[i];
            theta = kth;
            __syncthreads();
            if (threadIdx.x == 0) sh.count = (uint32_t)got;
            __syncthreads();
        }
    }
    const int n = (int)sh.count;
    const uint64_t kth = n > k ? block_kth_largest(buf, n, k, sh) : 1;
    return block_collect_sorted(buf, n, kth, k, sh);
}

// Shared-memory layout of the kernels that may take the exact path:
// [SelectShared][hidden floats][kDirectBuf keys] (and the staged candidates
// reuse the float + key area).
__host__ __device__ inline size_t direct_smem_bytes(int hidden) {
    return (((size_t)hidden * 4 + 15) & ~(size_t)15) + (size_t)kDirectBuf * 8;
}

template <typename T>
__global__ void __launch_bounds__(kSelThreads)
    direct_topk_kernel(const T *__restrict__ h, const T *__restrict__ w, int hidden,
                       int64_t draft_vocab, int64_t target_vocab, float mult, float cap, int k,
                       int64_t *ids, float *vals, int32_t *err) {
    grid_dep_wait();
    __shared__ SelectShared sh;
    extern __shared__ __align__(16) uint8_t dyn[];
    float *hs = reinterpret_cast<float *>(dyn);
    uint64_t *buf = reinterpret_cast<uint64_t *>(dyn + (((size_t)hidden * 4 + 15) & ~(size_t)15));
    const int64_t row = blockIdx.x;
    const int got = direct_row_topk<T>(h + row * hidden, w, hidden, draft_vocab, target_vocab, mult,
                                       cap, k, hs, buf, sh);
    write_row(sh, got, k, row, ids, vals, err);
}

// fp32 with a workspace: the vocab split into chunks of chunk_len rows, one
// CTA per (row, chunk) running the exact routine on its chunk; the lists
// ([chunks][rows][k], chunk-local ids, u = -inf where a chunk holds fewer than
// k entries) are merged by dflash2_topk_merge.
constexpr int kFp32ChunkMin = 256;   // vocab rows per chunk, at least
constexpr int kFp32MaxChunks = 32;

inline int fp32_chunks(int64_t rows, int64_t vmax, int k) {
    int64_t c = (304 + rows - 1) / rows;  // about two CTAs per SM of a 152-SM GPU
    const int64_t by_len = vmax / std::max<int64_t>(kFp32ChunkMin, k);
    if (c > by_len) c = by_len;
    if (c > kFp32MaxChunks) c = kFp32MaxChunks;
    if ((int64_t)c * k > 4096) c = 4096 / k;  // the merge's key budget
    return c < 1 ? 1 : (int)c;
}

__global__ void __launch_bounds__(kSelThreads)
    direct_chunk_kernel(const float *__restrict__ h, const float *__restrict__ w, int hidden,
                        int64_t vmax, int64_t chunk_len, float mult, float cap, int k,
                        int64_t *ids, float *vals) {
    grid_dep_wait();
    __shared__ SelectShared sh;
    extern __shared__ __align__(16) uint8_t dyn[];
    float *hs = reinterpret_cast<float *>(dyn);
    uint64_t *buf = reinterpret_cast<uint64_t *>(dyn + (((size_t)hidden * 4 + 15) & ~(size_t)15));
    const int64_t row = blockIdx.x, rows = gridDim.x;
    const int64_t c0 = (int64_t)blockIdx.y * chunk_len;
    const int64_t len = min(chunk_len, vmax - c0);
    const int got = direct_row_topk<float>(h + row * hidden, w + c0 * hidden, hidden, len, len,
                                           mult, cap, k, hs, buf, sh);
    const int64_t base = ((int64_t)blockIdx.y * rows + row) * k;
    for (int i = threadIdx.x; i < k; i += blockDim.x) {
        ids[base + i] = i < got ? (int64_t)key_id(sh.top[i]) : 0;
        vals[base + i] = i < got ? key_u(sh.top[i]) : -INFINITY;  // absent for the merge
    }
}

// Pilot select: threshold and seed candidates of each row from its pilot u.
//
// theta_pre: for mult > 0 and a positive threshold u_th, the transform obeys
// u <= mult * z (1 + 2^-21) after rounding: tanh(x) <= x for x >= 0, tanhf is
// within 2 ulp, and the divide and the two multiplies round once each (for
// mult * z < 0, u < 0 < u_th).  So any entry whose computed u reaches u_th has
// fl(mult * z) >= u_th (1 - 2^-21) > u_th (1 - 2^-18) = theta_pre, and the
// filter may skip the transform wherever fl(mult * z) < theta_pre.  With no
// threshold, mult <= 0 or u_th <= 0, theta_pre is -inf (every entry checked).
__global__ void __launch_bounds__(kSelThreads)
    pilot_select_kernel(const float *__restrict__ pilot_z, int n_pilot, int pilot_stride, int unit,
                        int k, float mult, float cap, uint64_t *theta, float *theta_pre,
                        uint32_t *cnt, uint64_t *cand, int cand_cap) {
    // The filter pass after this kernel reads only its inputs until its
    // epilogue waits for this grid, so it may start now (this kernel starts
    // only once the pilot pass, which waited for the inputs, has ended).
    grid_dep_launch();
    grid_dep_wait();
    __shared__ SelectShared sh;
    __shared__ float fsort[kSelThreads];
    const int64_t row = blockIdx.x;
    const int n = n_pilot * unit;  // unit == kSelThreads: entry i = tid + 256 j is row tid of unit j
    const float *pz = pilot_z + row * n;
    constexpr int kPer = kPilotTiles * kGemmTileW / kSelThreads;  // entries per thread, at most
    const int t = threadIdx.x;
    float z[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) z[j] = t + j * kSelThreads < n ? pz[t + j * kSelThreads] : -INFINITY;
    const auto vocab_id = [&](int j) { return (uint32_t)(j * pilot_stride * unit + t); };
    uint64_t th;
    float pre;
    if (mult > 0.0f) {
        // the transform is non-decreasing in z: theta from the raw logits, the
        // exact transform only where the pre-threshold lets a key reach theta.
        // z* = the k-th largest per-thread maximum; u* = its transformed value.
        // At least k entries have z >= z*, hence u >= u*, hence a key >= the
        // smallest key with value u*, which is theta: a lower bound of the
        // row's k-th best key.
        float zm = -INFINITY;
#pragma unroll
        for (int j = 0; j < kPer; ++j) zm = fmaxf(zm, z[j]);
        const float zs = block_kth_of_maxima_f(zm, k, fsort);
        if (zs == -INFINITY) {
            th = 0;  // fewer than k threads hold a valid entry: all are candidates
            pre = -INFINITY;
        } else {
            const float us = unary_transform(zs, mult, cap);
            th = make_key(us, 0xFFFFFFFFu);  // the smallest key of value u*
            pre = us > 0.0f ? us * (1.0f - 0x1p-18f) : -INFINITY;
        }
    } else {
        // no monotone shortcut: every entry's exact key, theta from their maxima
        uint64_t km = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j)
            if (z[j] != -INFINITY)
                km = max(km, make_key(unary_transform(z[j], mult, cap), vocab_id(j)));
        th = block_kth_of_maxima(km, k, sh);
        pre = -INFINITY;
    }
    if (t == 0) sh.count = 0;
    __syncthreads();
    // every pilot key at or above theta seeds the candidate list
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        if (z[j] != -INFINITY && mult * z[j] >= pre) {
            const uint64_t key = make_key(unary_transform(z[j], mult, cap), vocab_id(j));
            if (key >= th) {
                const uint32_t slot = atomicAdd(&sh.count, 1u);
                if (slot < (uint32_t)cand_cap) cand[row * cand_cap + slot] = key;
            }
        }
    }
    __syncthreads();
    if (t == 0) {
        theta[row] = th;
        theta_pre[row] = pre;
        cnt[row] = sh.count;  // more than cand_cap: finalize recomputes the row exactly
    }
}

// Final exact top-k of each row's candidate list (or the exact CUDA-core
// recomputation of the row when its list overflowed; T = the operands' type,
// with the fp8 scales when T is the E4M3 code).
template <typename T>
__global__ void __launch_bounds__(kSelThreads)
    finalize_kernel(const uint32_t *__restrict__ cnt, const uint64_t *__restrict__ cand,
                    int cand_cap, int k, int64_t *ids, float *vals, int32_t *err,
                    const T *__restrict__ h, const T *__restrict__ w, int hidden,
                    int64_t draft_vocab, int64_t target_vocab, float mult, float cap,
                    const float *__restrict__ a_scale, const float *__restrict__ w_scale,
                    NvScales nv) {
    grid_dep_wait();
    __shared__ SelectShared sh;
    extern __shared__ __align__(16) uint8_t dyn[];
    const int64_t row = blockIdx.x;
    const uint32_t n = cnt[row];
    if (n > (uint32_t)cand_cap) {
        float *hs = reinterpret_cast<float *>(dyn);
        uint64_t *buf =
            reinterpret_cast<uint64_t *>(dyn + (((size_t)hidden * 4 + 15) & ~(size_t)15));
        int got;
        if constexpr (std::is_same<T, E2M1x2>::value)
            got = direct_row_topk_nvfp4(
                reinterpret_cast<const uint8_t *>(h) + row * (hidden / 2),
                nv.sfh + row * (hidden / 16), reinterpret_cast<const uint8_t *>(w), nv.sfw_tiles,
                hidden, draft_vocab, target_vocab, mult, cap, k, hs, buf, sh,
                a_scale[row] * nv.w_global);
        else
            got = direct_row_topk<T>(h + row * hidden, w, hidden, draft_vocab, target_vocab, mult,
                                     cap, k, hs, buf, sh, w_scale, a_scale ? a_scale[row] : 1.0f);
        write_row(sh, got, k, row, ids, vals, err);
        if (threadIdx.x == 0 && err) atomicOr(err, DFLASH2_DEVINFO_TOPK_FALLBACK);
        return;
    }
    const uint64_t *src = cand + row * cand_cap;
    // the keys staged in shared memory once (when they fit) while the
    // per-thread maxima form the threshold; then an exact sort of the (few)
    // keys at or above it.  The radix select remains for the rare row where
    // more than kCollect keys reach the threshold.
    const bool staged = n <= (uint32_t)kSmemKeys;
    uint64_t *st = reinterpret_cast<uint64_t *>(dyn);
    const uint64_t *keys = staged ? st : src;
    uint64_t tmax = 0;
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) {
        const uint64_t key = src[i];
        if (staged) st[i] = key;
        tmax = key > tmax ? key : tmax;
    }
    const uint64_t th = block_kth_of_maxima(tmax, k, sh);  // its barriers also publish st
    uint64_t *col = reinterpret_cast<uint64_t *>(dyn) + (staged ? kSmemKeys : 0);  // kCollect keys
    if (threadIdx.x == 0) sh.count = 0;
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) {
        const uint64_t key = keys[i];
        if (key != 0 && key >= th) {
            const uint32_t slot = atomicAdd(&sh.count, 1u);
            if (slot < (uint32_t)kCollect) col[slot] = key;
        }
    }
    __syncthreads();
    const int c = (int)sh.count;
    if (c <= 32) {
        if (threadIdx.x < 32) {
            const uint64_t v = warp_sort_desc(threadIdx.x < c ? col[threadIdx.x] : 0, threadIdx.x);
            if ((int)threadIdx.x < k) sh.top[threadIdx.x] = v;
        }
        for (int i = 32 + threadIdx.x; i < k; i += blockDim.x) sh.top[i] = 0;
        __syncthreads();
        write_row(sh, c < k ? c : k, k, row, ids, vals, err);
        return;
    }
    if (c <= kCollect) {
        int np = 1;
        while (np < c) np <<= 1;
        for (int i = c + threadIdx.x; i < np; i += blockDim.x) col[i] = 0;
        __syncthreads();
        block_sort_desc(col, np);
        const int got = c < k ? c : k;
        for (int i = threadIdx.x; i < k; i += blockDim.x) sh.top[i] = i < got ? col[i] : 0;
        __syncthreads();
        write_row(sh, got, k, row, ids, vals, err);
        return;
    }
    const int kk = (int)n < k ? (int)n : k;
    const uint64_t kth = kk > 0 ? block_kth_largest(keys, (int)n, kk, sh) : ~0ull;
    const int got = block_collect_sorted(keys, (int)n, kth, k, sh);
    write_row(sh, got, k, row, ids, vals, err);
}

// ---- workspace layout (bf16) -------------------------------------------------
struct TopkLayout {
    int32_t n_wtiles, n_pilot, pilot_stride, cap;
    size_t theta_off, pre_off, cnt_off, pilot_off, pmax_off, sync_off, cand_off, fixed_bytes;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// The pilot and filter passes run on CTA pairs (2-CTA MMA over 256-row
// weight units): each CTA of a pair stages only half of the token tile, so a
// stage of 128 hidden elements is small enough for three stages in shared
// memory, where one CTA per 128-row unit fits two.
inline int unit_rows() { return 2 * kGemmTileW; }

inline TopkLayout topk_layout(int64_t rows, int64_t draft_vocab) {
    TopkLayout L{};
    const int unit = unit_rows();
    L.n_wtiles = (int32_t)((draft_vocab + unit - 1) / unit);
    pilot_layout(L.n_wtiles, &L.n_pilot, &L.pilot_stride, unit);
    L.theta_off = 0;
    L.pre_off = align256(L.theta_off + (size_t)rows * 8);
    L.cnt_off = align256(L.pre_off + (size_t)rows * 4);
    L.pilot_off = align256(L.cnt_off + (size_t)rows * 4);
    L.pmax_off = align256(L.pilot_off + (size_t)rows * L.n_pilot * unit * 4);
    L.sync_off = align256(L.pmax_off + (size_t)rows * L.n_pilot * (unit / 32) * 4);
    L.cand_off = L.sync_off + 256;  // the fused launch's two grid counters
    L.fixed_bytes = L.cand_off;
    return L;
}

inline int64_t recommended_cap(const TopkLayout &L, int k) {
    const int64_t rest = L.n_wtiles - L.n_pilot;
    int64_t cap = k + 4LL * k * ((rest + L.n_pilot - 1) / L.n_pilot) + 256;
    cap = (cap + 63) / 64 * 64;
    if (cap > kMaxCandCap) cap = kMaxCandCap;
    if (cap < k) cap = k;
    return cap;
}

// Token tile of the bf16 path: the rows in near-equal tiles of at most 256.
inline int token_tile(int64_t rows, int max_bn = 256) {
    const int64_t n_tiles = (rows + max_bn - 1) / max_bn;
    return (int)(((rows + n_tiles - 1) / n_tiles + 15) / 16 * 16);
}

// One cooperative launch (pilot tiles, the select on the epilogue warps,
// filter tiles) replaces the pilot pass, the select kernel and the filter
// pass when
//   - mult > 0 (its select relies on the monotone transform),
//   - the pilot has at least 4 K groups of 32 rows (8 per unit),
//   - each epilogue warp selects at most two rows and each CTA pair keeps at
//     most two pilot accumulators, so the thresholds are ready while the
//     first filter tiles are still in the tensor cores, and
//   - it adds at most one round of tiles per CTA pair over the filter pass
//     alone.  The pilot pass and the select it saves cost about 1.3 rounds at
//     the bf16 workloads (measured on GB300: 7 us faster with one extra
//     round, 11 us slower with two).
bool use_fused(const DeviceInfo &di, const TopkLayout &L, int64_t rows, int bn, float mult,
               int top_k, bool nv = false) {
    const int fused_warps = fused_epilogue_warps(di, nv);
    if (!(mult > 0.0f) || fused_warps <= 0 || rows > 2LL * fused_warps) return false;
    // its groups are 32-row slices of the pilot units; with fewer than 4 K of
    // them the threshold is loose and candidate lists overflow
    if ((int64_t)L.n_pilot * (unit_rows() / 32) < 4LL * top_k) return false;
    const int64_t tok_tiles = (rows + bn - 1) / bn;
    const int64_t all_tiles = (int64_t)L.n_wtiles * tok_tiles;
    const int64_t filter_tiles = (int64_t)(L.n_wtiles - L.n_pilot) * tok_tiles;
    const int64_t fused_pairs = std::min<int64_t>(all_tiles, fused_pair_count(di, nv));
    if ((int64_t)L.n_pilot * tok_tiles > 2 * fused_pairs) return false;
    const int64_t filter_pairs = std::min<int64_t>(filter_tiles, di.sm_count / 2);
    if (filter_pairs < 1) return true;  // the pilot covers the vocab
    return (all_tiles + fused_pairs - 1) / fused_pairs <=
           (filter_tiles + filter_pairs - 1) / filter_pairs + 1;
}

std::atomic<bool> g_topk_attr[64];  // per device; the attribute calls are idempotent

dflash2_status set_select_attrs(int device) {
    if (device < 0 || device >= 64) return DFLASH2_ERR_CUDA;
    if (g_topk_attr[device]) return DFLASH2_OK;
    const int bytes = 160 * 1024;
    if (cudaFuncSetAttribute(finalize_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(finalize_kernel<__nv_fp8_e4m3>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(finalize_kernel<E2M1x2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess ||
        cudaFuncSetAttribute(pilot_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess ||
        cudaFuncSetAttribute(direct_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess ||
        cudaFuncSetAttribute(direct_topk_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess ||
        cudaFuncSetAttribute(direct_topk_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
        cudaGetLastError();
        return DFLASH2_ERR_CUDA;
    }
    g_topk_attr[device] = true;
    return DFLASH2_OK;
}

constexpr int kMaxHidden = 32768;  // the exact path stages one h row as fp32 in shared memory

// The tensor-core top-K (T = __nv_bfloat16, or __nv_fp8_e4m3 codes with the
// per-row scales a_scale [rows] and w_scale [draft_vocab]): the pilot pass,
// select and filter pass (or their fused launch), then the final top-K.  The
// arguments are checked by the caller.
template <typename T>
dflash2_status run_tc_topk(const DeviceInfo &di, const void *h, const void *lm_head,
                           const float *a_scale, const float *w_scale, int64_t rows, int hidden,
                           int64_t draft_vocab, int64_t target_vocab, float mult, float cap,
                           int top_k, int64_t *cand_ids, float *cand_u, void *workspace,
                           size_t ws_bytes, int32_t *err_word, cudaStream_t st,
                           NvScales nvs = NvScales{}) {
    constexpr bool kNv = std::is_same<T, E2M1x2>::value;
    dflash2_status s = DFLASH2_OK;
    const size_t dsm = direct_smem_bytes(hidden);
    const TopkLayout L = topk_layout(rows, draft_vocab);
    if (!workspace || ws_bytes < L.fixed_bytes + (size_t)rows * top_k * 8)
        return DFLASH2_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return DFLASH2_ERR_MISALIGNED;
    int64_t cap_keys = (int64_t)((ws_bytes - L.fixed_bytes) / ((size_t)rows * 8));
    if (cap_keys > kMaxCandCap) cap_keys = kMaxCandCap;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint64_t *theta = reinterpret_cast<uint64_t *>(ws + L.theta_off);
    float *theta_pre = reinterpret_cast<float *>(ws + L.pre_off);
    uint32_t *cnt = reinterpret_cast<uint32_t *>(ws + L.cnt_off);
    float *pilot_u = reinterpret_cast<float *>(ws + L.pilot_off);
    uint64_t *cand = reinterpret_cast<uint64_t *>(ws + L.cand_off);

    const int bn = token_tile(rows, kNv ? 128 : 256);  // nvfp4: the scales' TMEM columns

    GemmParams p{};
    p.rows_w = (int32_t)draft_vocab;
    p.rows_h = (int32_t)rows;
    p.hidden = hidden;
    p.bn = bn;
    p.k_splits = 1;
    p.target_vocab = target_vocab;
    p.mult = mult;
    p.cap = cap;
    p.err = err_word;
    p.fp8 = std::is_same<T, __nv_fp8_e4m3>::value ? 1 : 0;
    p.a_scale = a_scale;
    p.w_scale = w_scale;
    p.nvfp4 = kNv ? 1 : 0;
    p.n_sf = hidden / 16;
    p.sfw = nvs.sfw_tiles;
    p.sfh = nvs.sfh_tiles;
    p.sf_nw8 = nvfp4_tile_cells(hidden);
    p.w_global = nvs.w_global;

    const bool pairs = true;
    const int unit = unit_rows();
    uint32_t *sync = reinterpret_cast<uint32_t *>(ws + L.sync_off);
    size_t fin_smem = ((size_t)kSmemKeys + kCollect) * 8;
    if (fin_smem < dsm) fin_smem = dsm;

    // the pilot pass, select and filter pass in one cooperative launch?
    if (use_fused(di, L, rows, bn, mult, top_k, kNv)) {
        if (cudaMemsetAsync(sync, 0, 2 * sizeof(uint32_t), st) != cudaSuccess) {
            cudaGetLastError();
            return DFLASH2_ERR_CUDA;
        }
        p.mode = kGemmFused;
        p.out = pilot_u;
        p.ldo = (int64_t)L.n_pilot * unit;
        p.theta = theta;
        p.theta_pre = theta_pre;
        p.cnt = cnt;
        p.cand = cand;
        p.cand_cap = (int32_t)cap_keys;
        p.top_k = top_k;
        p.sync = sync;
        p.pmax = reinterpret_cast<uint32_t *>(ws + L.pmax_off);
        p.ld_pmax = (int64_t)L.n_pilot * (unit / 32);
        s = launch_gemm_tc(di, lm_head, h, p, st, pairs);
        if (s != DFLASH2_OK) return s;
        launch_k(finalize_kernel<T>, (unsigned)rows, kSelThreads, fin_smem, st, cnt, cand,
                 (int)cap_keys, top_k, cand_ids, cand_u, err_word, static_cast<const T *>(h),
                 static_cast<const T *>(lm_head), hidden, draft_vocab, target_vocab, mult, cap,
                 a_scale, w_scale, nvs);
        return launch_status();
    }

    // The pilot covers at most 32 weight tiles: smaller token tiles spread
    // its work items over the SMs.
    p.mode = kGemmPilot;
    p.out = pilot_u;
    p.ldo = (int64_t)L.n_pilot * unit;
    if (!kNv) {  // nvfp4: the token scale tiles are cut at the filter's token tile
        int64_t want_tiles = (pairs ? di.sm_count / 2 : di.sm_count) / L.n_pilot;  // one wave
        if (want_tiles < 1) want_tiles = 1;
        int64_t per = (rows + want_tiles - 1) / want_tiles;
        per = (per + 15) / 16 * 16;
        p.bn = (int)(per < 16 ? 16 : (per > bn ? bn : per));
    }
    s = launch_gemm_tc(di, lm_head, h, p, st, pairs);
    if (s != DFLASH2_OK) return s;
    p.bn = bn;

    static_assert(2 * kGemmTileW == kSelThreads, "pilot select maps one unit row per thread");
    launch_k(pilot_select_kernel, (unsigned)rows, kSelThreads, 0, st, pilot_u, L.n_pilot,
        L.pilot_stride, unit, top_k, mult, cap, theta, theta_pre, cnt, cand,
        (int)cap_keys);
    s = launch_status();
    if (s != DFLASH2_OK) return s;

    p.mode = kGemmFilter;
    p.out = nullptr;
    p.theta = theta;
    p.theta_pre = theta_pre;
    p.cnt = cnt;
    p.cand = cand;
    p.cand_cap = (int32_t)cap_keys;
    s = launch_gemm_tc(di, lm_head, h, p, st, pairs);
    if (s != DFLASH2_OK) return s;

    // staged keys (a row with at most kSmemKeys candidates) followed by the
    // collect buffer
    launch_k(finalize_kernel<T>, (unsigned)rows, kSelThreads, fin_smem, st, cnt, cand,
             (int)cap_keys, top_k, cand_ids, cand_u, err_word, static_cast<const T *>(h),
             static_cast<const T *>(lm_head), hidden, draft_vocab, target_vocab, mult, cap,
             a_scale, w_scale, nvs);
    return launch_status();
}

}  // namespace
}  // namespace dflash2

using namespace dflash2;

extern "C" size_t dflash2_unary_topk_workspace_size(int64_t rows, int64_t draft_vocab, int32_t top_k,
                                                    int32_t dtype) {
    if (rows <= 0 || draft_vocab <= 0 || top_k <= 0) return 0;
    if (dtype == DFLASH2_F32) {
        // the chunked exact path's lists (none when one chunk covers the vocab)
        const int c = fp32_chunks(rows, draft_vocab, top_k);
        return c > 1 ? (size_t)c * rows * top_k * 12 : 0;
    }
    const TopkLayout L = topk_layout(rows, draft_vocab);
    return L.fixed_bytes + (size_t)rows * recommended_cap(L, top_k) * 8;
}

extern "C" size_t dflash2_unary_topk_workspace_min(int64_t rows, int64_t draft_vocab, int32_t top_k,
                                                   int32_t dtype) {
    if (rows <= 0 || draft_vocab <= 0 || top_k <= 0) return 0;
    if (dtype == DFLASH2_F32) return 0;
    const TopkLayout L = topk_layout(rows, draft_vocab);
    return L.fixed_bytes + (size_t)rows * top_k * 8;
}

extern "C" int32_t dflash2_unary_topk_launches(int64_t rows, int64_t draft_vocab, int32_t top_k,
                                               float mult, int32_t dtype) {
    if (dtype != DFLASH2_F32 && dtype != DFLASH2_BF16) return -1;
    if (rows < 0 || rows > INT32_MAX || draft_vocab <= 0 || draft_vocab > INT32_MAX ||
        top_k <= 0 || top_k > kMaxTopK || top_k > draft_vocab)
        return -1;
    if (rows == 0) return 0;
    if (dtype == DFLASH2_F32) return fp32_chunks(rows, draft_vocab, top_k) > 1 ? 2 : 1;
    DeviceInfo di;
    if (current_device(&di) != DFLASH2_OK) return -1;
    const TopkLayout L = topk_layout(rows, draft_vocab);
    if (use_fused(di, L, rows, token_tile(rows), mult, top_k)) return 2;  // fused GEMM, finalize
    return L.n_wtiles > L.n_pilot ? 4 : 3;  // pilot, select, (filter), finalize
}

namespace {
inline size_t fp8_ws_prefix(int64_t rows, int32_t hidden) {
    return align256((size_t)rows * hidden) + align256((size_t)rows * 4);
}
// The NVFP4 path's quantized activations at the workspace's start: codes
// [rows][hidden / 2], block scales [rows][hidden / 16], g [rows], and the
// scales again as tiles of the token tile.
inline size_t nvfp4_ws_prefix(int64_t rows, int32_t hidden) {
    return align256((size_t)rows * (hidden / 2)) + align256((size_t)rows * (hidden / 16)) +
           align256((size_t)rows * 4) +
           align256(nvfp4_tiles_bytes(rows, hidden, token_tile(rows, 128)));
}
}  // namespace

extern "C" size_t dflash2_unary_topk_fp8_workspace_size(int64_t rows, int32_t hidden,
                                                        int64_t draft_vocab, int32_t top_k) {
    if (rows <= 0 || hidden <= 0 || draft_vocab <= 0 || top_k <= 0) return 0;
    return fp8_ws_prefix(rows, hidden) +
           dflash2_unary_topk_workspace_size(rows, draft_vocab, top_k, DFLASH2_BF16);
}

extern "C" dflash2_status dflash2_unary_topk_fp8(const void *h, int32_t h_dtype,
                                                 const uint8_t *lm_head_q, const float *w_scale,
                                                 int64_t rows, int32_t hidden, int64_t draft_vocab,
                                                 int64_t target_vocab, float mult, float cap,
                                                 int32_t top_k, int64_t *cand_ids, float *cand_u,
                                                 void *workspace, size_t ws_bytes,
                                                 int32_t *err_word, void *stream) {
    if (h_dtype != DFLASH2_F32 && h_dtype != DFLASH2_BF16) return DFLASH2_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || rows > INT32_MAX || hidden <= 0 || hidden > kMaxHidden || draft_vocab <= 0 ||
        draft_vocab > INT32_MAX || target_vocab <= 0 || top_k <= 0 || top_k > kMaxTopK ||
        top_k > target_vocab || top_k > draft_vocab || !(cap >= 0.0f))
        return DFLASH2_ERR_INVALID_ARG;
    if (rows == 0) return DFLASH2_OK;
    if (!h || !lm_head_q || !w_scale || !cand_ids || !cand_u) return DFLASH2_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(cand_ids) % 8 != 0 ||
        reinterpret_cast<uintptr_t>(cand_u) % 4 != 0 ||
        reinterpret_cast<uintptr_t>(w_scale) % 4 != 0 ||
        reinterpret_cast<uintptr_t>(h) % (h_dtype == DFLASH2_BF16 ? 2 : 4) != 0)
        return DFLASH2_ERR_MISALIGNED;
    // TMA rows of codes: a 16-byte row stride and base
    if (hidden % 16 != 0 || !aligned16(lm_head_q)) return DFLASH2_ERR_MISALIGNED;
    const size_t prefix = fp8_ws_prefix(rows, hidden);
    if (!workspace || ws_bytes < prefix) return DFLASH2_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    dflash2_status s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    s = set_select_attrs(di.device);
    if (s != DFLASH2_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *qh = ws;
    float *dh = reinterpret_cast<float *>(ws + align256((size_t)rows * hidden));
    s = launch_quant_rows_e4m3(h, h_dtype, rows, hidden, qh, dh, st);
    if (s != DFLASH2_OK) return s;
    return run_tc_topk<__nv_fp8_e4m3>(di, qh, lm_head_q, dh, w_scale, rows, hidden, draft_vocab,
                                      target_vocab, mult, cap, top_k, cand_ids, cand_u,
                                      ws + prefix, ws_bytes - prefix, err_word, st);
}

extern "C" dflash2_status dflash2_unary_topk(const void *h, const void *lm_head, int64_t rows,
                                             int32_t hidden, int64_t draft_vocab,
                                             int64_t target_vocab, float mult, float cap,
                                             int32_t top_k, int32_t dtype, int64_t *cand_ids,
                                             float *cand_u, void *workspace, size_t ws_bytes,
                                             int32_t *err_word, void *stream) {
    if (dtype != DFLASH2_F32 && dtype != DFLASH2_BF16) return DFLASH2_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || rows > INT32_MAX || hidden <= 0 || hidden > kMaxHidden || draft_vocab <= 0 ||
        draft_vocab > INT32_MAX || target_vocab <= 0 || top_k <= 0 || top_k > kMaxTopK ||
        top_k > target_vocab || top_k > draft_vocab || !(cap >= 0.0f))
        return DFLASH2_ERR_INVALID_ARG;
    if (rows == 0) return DFLASH2_OK;
    if (!h || !lm_head || !cand_ids || !cand_u) return DFLASH2_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(cand_ids) % 8 != 0 || reinterpret_cast<uintptr_t>(cand_u) % 4 != 0)
        return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    dflash2_status s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    s = set_select_attrs(di.device);
    if (s != DFLASH2_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t dsm = direct_smem_bytes(hidden);

    if (dtype == DFLASH2_F32) {
        if ((reinterpret_cast<uintptr_t>(h) | reinterpret_cast<uintptr_t>(lm_head)) % 4 != 0)
            return DFLASH2_ERR_MISALIGNED;
        // chunks over the candidate vocab: the workspace size uses the draft
        // vocab (the host knows no target bound there), which only over-counts
        const int64_t vmax = std::min<int64_t>(draft_vocab, target_vocab);
        const int chunks = fp32_chunks(rows, vmax, top_k);
        const size_t need = (size_t)chunks * rows * top_k * 12;
        if (chunks > 1 && workspace && ws_bytes >= need &&
            reinterpret_cast<uintptr_t>(workspace) % 8 == 0) {
            const int64_t chunk_len = (vmax + chunks - 1) / chunks;
            const int n_chunks = (int)((vmax + chunk_len - 1) / chunk_len);
            int64_t *lid = static_cast<int64_t *>(workspace);
            float *lu = reinterpret_cast<float *>(lid + (size_t)n_chunks * rows * top_k);
            launch_k(direct_chunk_kernel, dim3((unsigned)rows, (unsigned)n_chunks), kSelThreads,
                     dsm, st, static_cast<const float *>(h), static_cast<const float *>(lm_head),
                     hidden, vmax, chunk_len, mult, cap, top_k, lid, lu);
            s = launch_status();
            if (s != DFLASH2_OK) return s;
            int64_t offs[kFp32MaxChunks];
            for (int c = 0; c < n_chunks; ++c) offs[c] = (int64_t)c * chunk_len;
            return dflash2_topk_merge(lid, lu, offs, n_chunks, rows, top_k, top_k, cand_ids,
                                      cand_u, err_word, stream);
        }
        launch_k(direct_topk_kernel<float>, (unsigned)rows, kSelThreads, dsm, st,
            static_cast<const float *>(h), static_cast<const float *>(lm_head), hidden, draft_vocab,

            target_vocab, mult, cap, top_k, cand_ids, cand_u, err_word);
        return launch_status();
    }

    if (hidden % 8 != 0 || !aligned16(h) || !aligned16(lm_head)) return DFLASH2_ERR_MISALIGNED;
    return run_tc_topk<__nv_bfloat16>(di, h, lm_head, nullptr, nullptr, rows, hidden, draft_vocab,
                                      target_vocab, mult, cap, top_k, cand_ids, cand_u,
                                      workspace, ws_bytes, err_word, st);
}

extern "C" size_t dflash2_unary_topk_nvfp4_workspace_size(int64_t rows, int32_t hidden,
                                                          int64_t draft_vocab, int32_t top_k) {
    if (rows <= 0 || hidden <= 0 || draft_vocab <= 0 || top_k <= 0) return 0;
    return nvfp4_ws_prefix(rows, hidden) +
           dflash2_unary_topk_workspace_size(rows, draft_vocab, top_k, DFLASH2_BF16);
}

extern "C" dflash2_status dflash2_unary_topk_nvfp4(
    const void *h, int32_t h_dtype, const uint8_t *lm_head_q, const uint8_t *w_scale_tiles,
    float w_global, int64_t rows, int32_t hidden, int64_t draft_vocab, int64_t target_vocab,
    float mult, float cap, int32_t top_k, int64_t *cand_ids, float *cand_u, void *workspace,
    size_t ws_bytes, int32_t *err_word, void *stream) {
    if (h_dtype != DFLASH2_F32 && h_dtype != DFLASH2_BF16) return DFLASH2_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || rows > INT32_MAX || hidden <= 0 || hidden > kMaxHidden || hidden % 64 != 0 ||
        draft_vocab <= 0 || draft_vocab > INT32_MAX || target_vocab <= 0 || top_k <= 0 ||
        top_k > kMaxTopK || top_k > target_vocab || top_k > draft_vocab || !(cap >= 0.0f) ||
        !(w_global > 0.0f) || !(w_global < INFINITY))
        return DFLASH2_ERR_INVALID_ARG;
    if (rows == 0) return DFLASH2_OK;
    if (!h || !lm_head_q || !w_scale_tiles || !cand_ids || !cand_u)
        return DFLASH2_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(cand_ids) % 8 != 0 ||
        reinterpret_cast<uintptr_t>(cand_u) % 4 != 0 || !aligned16(w_scale_tiles) ||
        reinterpret_cast<uintptr_t>(h) % (h_dtype == DFLASH2_BF16 ? 2 : 4) != 0)
        return DFLASH2_ERR_MISALIGNED;
    if (!aligned16(lm_head_q)) return DFLASH2_ERR_MISALIGNED;  // TMA rows of codes
    const size_t prefix = nvfp4_ws_prefix(rows, hidden);
    if (!workspace || ws_bytes < prefix) return DFLASH2_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    dflash2_status s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    s = set_select_attrs(di.device);
    if (s != DFLASH2_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *qh = ws;
    uint8_t *sh = ws + align256((size_t)rows * (hidden / 2));
    float *gh = reinterpret_cast<float *>(sh + align256((size_t)rows * (hidden / 16)));
    uint8_t *th = reinterpret_cast<uint8_t *>(gh) + align256((size_t)rows * 4);
    s = launch_quant_rows_nvfp4(h, h_dtype, rows, hidden, qh, sh, gh, st);
    if (s != DFLASH2_OK) return s;
    s = launch_nvfp4_tile_scales(sh, rows, hidden, token_tile(rows, 128), th, st);
    if (s != DFLASH2_OK) return s;
    NvScales nvs{sh, w_scale_tiles, th, w_global};
    return run_tc_topk<E2M1x2>(di, qh, lm_head_q, gh, nullptr, rows, hidden, draft_vocab,
                               target_vocab, mult, cap, top_k, cand_ids, cand_u, ws + prefix,
                               ws_bytes - prefix, err_word, st, nvs);
}
