// Selector lattice + walk (sglang DFlash2 PR: the PR body's edge formula,
// CandidateSelector.build_lattice / sample_path, _selector_walk_kernel,
// stage_sampling_params).
//
//   g[m, :] = h[m, :] . proj^T                           (tensor cores for bf16)
//   e[k]    = sum_j A[p, j] * g[b*S + s, j] * B[c_k, j] + cand_u[b, s, k]
//   greedy: index = smallest argmax e, q = one-hot;  sampled: q = softmax(e / T),
//   index = min(#{k : uniform >= cumsum(q)[k]}, K - 1);  token = c_index.
//
// One warp walks one request, as the Triton walk runs one single-warp program
// per request; a CTA holds several independent requests and no block-wide
// barrier is used.  The lattice is never materialised: only the K edges
// leaving the chosen predecessor are formed.  The rows a slot needs do not
// depend on the path, so they are fetched ahead with 1-D TMA bulk copies into
// a ring of shared-memory buffers: group s holds the B rows of slot s's
// candidates and, when shared memory allows, the A rows of its possible
// predecessors (the anchor at slot 0, else slot s-1's candidates).  The
// serial chain of a slot then touches shared memory and registers only.
#include "kernels.h"

#include <atomic>

namespace dflash2 {
namespace {

constexpr int kMaxK = 128;
constexpr int kMaxRank = 256;
constexpr int kMaxWarpsPerCta = 4;
constexpr int kMaxRing = 8;     // prefetch groups per warp
constexpr size_t kWalkSmemBytes = 224 * 1024;

struct WalkParams {
    const float *g;        // [k_splits][rows][rank] partial projections
    int32_t k_splits;
    int64_t split_stride;
    const void *A;
    const void *B;
    int64_t table_rows;
    const int64_t *anchors;
    const int64_t *cand;
    const float *cand_u;
    const float *temps;
    const uint8_t *greedy;
    const float *uniforms;
    int32_t batch, slots, rank, k;
    bool bulk_ids;
    // launched right after this library's projection of the same call: the
    // candidates, anchors and tables were complete before that projection
    // started, so the walk may read them before its grid dependency wait
    bool after_projection;
    int64_t *tokens;
    float *q;
    float *path_scores;
    int32_t *err;
};

// Per-warp shared-memory layout (byte offsets from the warp's base).
struct WalkLayout {
    int row_bytes;  // rank * sizeof(T): one table row
    int nbuf;       // prefetch ring size
    size_t bars, ids, cu, uni, gs, w, bbuf, abuf, scratch_bytes, total;
};

__host__ __device__ inline size_t pad16(size_t x) { return (x + 15) & ~(size_t)15; }

__host__ __device__ inline WalkLayout walk_layout(int slots, int k, int rank, int esz, bool prefetch_a,
                                                  int nbuf, int k_splits) {
    WalkLayout L;
    L.row_bytes = rank * esz;
    L.nbuf = nbuf;
    L.bars = 0;                                        // nbuf + 1 mbarriers
    L.ids = pad16((size_t)(kMaxRing + 1) * 8);
    L.cu = L.ids + pad16((size_t)slots * k * 8);
    L.uni = L.cu + pad16((size_t)slots * k * 4);
    L.gs = L.uni + pad16((size_t)slots * 4);
    L.w = L.gs + pad16((size_t)slots * rank * 4);
    L.bbuf = L.w + pad16((size_t)rank * 4);
    L.abuf = L.bbuf + (size_t)nbuf * k * L.row_bytes;
    size_t end = L.abuf + (prefetch_a ? (size_t)nbuf * k * L.row_bytes : 0);
    // the projection partials land in the ring buffers before the first group
    L.scratch_bytes = (size_t)k_splits * slots * rank * 4;
    if (L.bbuf + L.scratch_bytes > end) end = L.bbuf + L.scratch_bytes;
    L.total = pad16(end);
    return L;
}

template <typename T> __device__ __forceinline__ void unpack16(const uint4 &v, float (&f)[16 / sizeof(T)]);
template <> __device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4 &v, float (&f)[8]) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
template <> __device__ __forceinline__ void unpack16<float>(const uint4 &v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}
template <typename T> __device__ __forceinline__ float ld1(const T *p);
template <> __device__ __forceinline__ float ld1<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float ld1<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}

// 16-byte asynchronous copy global -> shared; invalid sources are zero-filled.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
    const uint32_t n = valid ? 16u : 0u;  // 0 source bytes: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)),
                 "l"(gmem), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 1-D TMA bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Bounded wait on a warp's own mbarrier.  After the limit the error bit is
// raised and *timed_out makes later waits return at once (the outputs are
// then invalid, but the kernel ends).
__device__ __forceinline__ void warp_bar_wait(uint64_t *bar, uint32_t parity, bool &timed_out,
                                              int32_t *err) {
    if (timed_out || mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            timed_out = true;
            if (err) atomicOr(err, DFLASH2_DEVERR_TIMEOUT);
            return;
        }
    }
}

__device__ __forceinline__ bool id_ok(int64_t c, int64_t rows) { return c >= 0 && c < rows; }

__device__ __forceinline__ void prefetch_l2_row(const void *row, int bytes) {
    for (int o = 0; o < bytes; o += 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const uint8_t *>(row) + o));
}

// Group s of the prefetch ring: one bulk copy per valid row (rows with an
// id outside the table are zero-filled with plain stores).  Lane 0 arms the
// group's mbarrier with the byte count before any copy is issued.
template <typename T, bool PA>
__device__ __forceinline__ void issue_group(const WalkParams &p, const WalkLayout &L, uint8_t *base,
                                            const int64_t *ids, int64_t anchor, int s, int lane) {
    const int K = p.k;
    const int buf = s % L.nbuf;
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + L.bars) + buf;
    uint8_t *bdst = base + L.bbuf + (size_t)buf * K * L.row_bytes;
    uint8_t *adst = base + L.abuf + (size_t)buf * K * L.row_bytes;
    const int64_t *bid = ids + (int64_t)s * K;
    const int64_t *aid = ids + (int64_t)(s - 1) * K;
    const int na = PA ? (s == 0 ? 1 : K) : 0;
    uint32_t valid = 0;
    for (int r = lane; r < K + na; r += 32) {
        const int64_t c = r < K ? bid[r] : (s == 0 ? anchor : aid[r - K]);
        valid += id_ok(c, p.table_rows) ? 1u : 0u;
    }
    for (int o = 16; o > 0; o >>= 1) valid += __shfl_xor_sync(0xFFFFFFFFu, valid, o);
    // order this buffer's earlier generic-proxy accesses before the copies
    fence_proxy_async_smem();
    if (lane == 0) mbar_arrive_expect_tx(bar, valid * (uint32_t)L.row_bytes);
    __syncwarp();
    const T *A = static_cast<const T *>(p.A);
    const T *B = static_cast<const T *>(p.B);
    for (int r = lane; r < K + na; r += 32) {
        const bool is_b = r < K;
        const int64_t c = is_b ? bid[r] : (s == 0 ? anchor : aid[r - K]);
        uint8_t *dst = is_b ? bdst + (size_t)r * L.row_bytes : adst + (size_t)(r - K) * L.row_bytes;
        if (id_ok(c, p.table_rows)) {
            bulk_copy(dst, (is_b ? B : A) + c * p.rank, (uint32_t)L.row_bytes, bar);
        } else {
            for (int o = 0; o < L.row_bytes; o += 16) *reinterpret_cast<uint4 *>(dst + o) = make_uint4(0, 0, 0, 0);
        }
    }
}

// The draw from one row of K edges held by one warp (lane owns candidates
// k = lane + 32 i; invalid entries are k >= K), with warp shuffles only.
// Greedy: the smallest index of the maximum, q one-hot.  Sampled: q =
// softmax(e / T) (T already clamped to >= 1e-5; divide, do not multiply by
// 1 / T), cdf = the inclusive prefix of q in candidate order (a blockwise
// warp scan), index = min(#{k : u >= cdf_k}, K - 1).  Returns the index (the
// same in every lane) and the lane's q values.
template <int E>
__device__ __forceinline__ int select_row(const float (&ev)[E], const bool (&valid)[E], bool greedy,
                                          float temp, float u, int K, int lane, float (&qv)[E]) {
    if (greedy) {
        float best = -INFINITY;
        int bi = INT32_MAX;
#pragma unroll
        for (int i = 0; i < E; ++i)
            if (valid[i] && (bi == INT32_MAX || ev[i] > best)) {
                best = ev[i];
                bi = lane + 32 * i;
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
            if (oi != INT32_MAX && (bi == INT32_MAX || ob > best || (ob == best && oi < bi))) {
                best = ob;
                bi = oi;
            }
        }
#pragma unroll
        for (int i = 0; i < E; ++i) qv[i] = (lane + 32 * i) == bi ? 1.0f : 0.0f;
        return bi;
    }
    float sc[E];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        sc[i] = valid[i] ? ev[i] / temp : -INFINITY;
        mx = fmaxf(mx, sc[i]);
    }
    mx = warp_max(mx);
    float local = 0.0f;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        qv[i] = valid[i] ? expf(sc[i] - mx) : 0.0f;
        local += qv[i];
    }
    const float total = warp_sum(local);
    float offset = 0.0f;  // mass of the previous 32-candidate blocks
    int count = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        qv[i] = qv[i] / total;
        float incl = qv[i];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        const float cdf = offset + incl;
        count += __popc(__ballot_sync(0xFFFFFFFFu, valid[i] && u >= cdf));
        if (i + 1 < E) offset = offset + __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    return count < K - 1 ? count : K - 1;
}

template <typename T, bool PA, int E>
__global__ void __launch_bounds__(kMaxWarpsPerCta * 32)
    walk_kernel(const WalkParams p, int warps_per_cta, WalkLayout L) {
    grid_dep_wait();
    extern __shared__ __align__(16) uint8_t dyn[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * warps_per_cta + warp;
    if (b >= p.batch) return;
    const int S = p.slots, K = p.k, R = p.rank;
    const int NB = L.nbuf;
    uint8_t *base = dyn + (size_t)warp * L.total;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + L.bars);
    int64_t *ids = reinterpret_cast<int64_t *>(base + L.ids);  // raw candidate ids
    float *cu = reinterpret_cast<float *>(base + L.cu);
    float *uni = reinterpret_cast<float *>(base + L.uni);
    float *gs = reinterpret_cast<float *>(base + L.gs);
    float *w = reinterpret_cast<float *>(base + L.w);
    const int64_t row0 = (int64_t)b * S;
    bool timed_out = false;

    if (lane == 0) {
        for (int i = 0; i <= NB; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // ---- prologue: ids, unary values and projection partials by bulk copy
    // (plain loads where the request's slice is not 16-byte aligned)
    uint64_t *pro = &bars[NB];
    float *scratch = reinterpret_cast<float *>(base + L.bbuf);
    const uint32_t part_bytes = (uint32_t)(S * R * 4);
    const bool bulk_ids = p.bulk_ids;  // the request's id and value slices are 16-byte aligned
    if (lane == 0)
        mbar_arrive_expect_tx(pro, (uint32_t)p.k_splits * part_bytes +
                                       (bulk_ids ? (uint32_t)(S * K * 12) : 0u));
    __syncwarp();
    if (lane < p.k_splits)
        bulk_copy(scratch + (size_t)lane * S * R, p.g + lane * p.split_stride + row0 * R, part_bytes,
                  pro);
    if (bulk_ids) {
        if (lane == 31) bulk_copy(ids, p.cand + row0 * K, (uint32_t)(S * K * 8), pro);
        if (lane == 30) bulk_copy(cu, p.cand_u + row0 * K, (uint32_t)(S * K * 4), pro);
    } else {
#pragma unroll 4
        for (int t = lane; t < S * K; t += 32) {
            ids[t] = p.cand[row0 * K + t];
            cu[t] = p.cand_u[row0 * K + t];
        }
    }
    for (int t = lane; t < S; t += 32) uni[t] = p.uniforms[row0 + t];
    const int64_t anchor = p.anchors[b];
    const bool greedy = p.greedy[b] != 0;
    float temp = p.temps[b];
    if (!(temp >= 1e-5f)) temp = 1e-5f;
    warp_bar_wait(pro, 0, timed_out, p.err);
    __syncwarp();
    // fixed-order sum of the partials
    for (int t = lane; t < S * R; t += 32) {
        float acc = scratch[t];
        for (int ks = 1; ks < p.k_splits; ++ks) acc += scratch[(size_t)ks * S * R + t];
        gs[t] = acc;
    }
    bool bad = !id_ok(anchor, p.table_rows);
    for (int t = lane; t < S * K; t += 32) bad |= !id_ok(ids[t], p.table_rows);
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && p.err) atomicOr(p.err, DFLASH2_DEVERR_ID_RANGE);
    __syncwarp();  // scratch (ring buffers) is free again

    for (int s0 = 0; s0 < NB - 1 && s0 < S; ++s0) issue_group<T, PA>(p, L, base, ids, anchor, s0, lane);

    constexpr int VN = 16 / sizeof(T);
    const T *A = static_cast<const T *>(p.A);
    int prev = 0;
    for (int s = 0; s < S; ++s) {
        const int64_t row = row0 + s;
        if (s + NB - 1 < S) issue_group<T, PA>(p, L, base, ids, anchor, s + NB - 1, lane);
        const int buf = s % NB;
        warp_bar_wait(&bars[buf], (uint32_t)(s / NB) & 1u, timed_out, p.err);
        __syncwarp();
        if (!PA && s + 1 < S) {
            // warm L2 with the A rows the next slot may need
            for (int t = lane; t < K; t += 32) {
                const int64_t c = ids[(int64_t)s * K + t];
                if (id_ok(c, p.table_rows)) prefetch_l2_row(A + c * R, L.row_bytes);
            }
        }
        // w = A[predecessor] (elementwise *) g
        const float *gsl = gs + (size_t)s * R;
        if (PA) {
            const T *arow = reinterpret_cast<const T *>(base + L.abuf + (size_t)buf * K * L.row_bytes +
                                                        (size_t)(s == 0 ? 0 : prev) * L.row_bytes);
            for (int j = lane; j < R; j += 32) w[j] = ld1<T>(arow + j) * gsl[j];
        } else {
            const int64_t pid = s == 0 ? anchor : ids[(int64_t)(s - 1) * K + prev];
            const bool ok = id_ok(pid, p.table_rows);
            for (int j = lane; j < R; j += 32) w[j] = (ok ? ld1<T>(A + pid * R + j) : 0.0f) * gsl[j];
        }
        __syncwarp();
        // edges: lane owns candidates k = lane + 32 i (two FMA chains each)
        const uint8_t *brows = base + L.bbuf + (size_t)buf * K * L.row_bytes;
        float ev[E];
        bool valid[E];
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const int kk = lane + 32 * i;
            valid[i] = kk < K;
            ev[i] = -INFINITY;
            if (valid[i]) {
                // rotate the starting vector by the lane so that lanes reading
                // different rows touch different banks
                const uint8_t *brow = brows + (size_t)kk * L.row_bytes;
                const int nvec = R / VN;
                float acc0 = 0.0f, acc1 = 0.0f;
                int v = lane % nvec;
                for (int n = 0; n < nvec; ++n, v = (v + 1 == nvec) ? 0 : v + 1) {
                    float bv[VN];
                    unpack16<T>(*reinterpret_cast<const uint4 *>(brow + v * 16), bv);
                    const float *wv = w + v * VN;
#pragma unroll
                    for (int e = 0; e < VN; e += 2) {
                        acc0 = fmaf(wv[e], bv[e], acc0);
                        acc1 = fmaf(wv[e + 1], bv[e + 1], acc1);
                    }
                }
                ev[i] = (acc0 + acc1) + cu[(int64_t)s * K + kk];
            }
        }
        // selection (warp shuffles only)
        float qv[E];
        const int index = select_row<E>(ev, valid, greedy, temp, uni[s], K, lane, qv);
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const int kk = lane + 32 * i;
            if (valid[i]) {
                p.q[row * K + kk] = qv[i];
                if (p.path_scores) p.path_scores[row * K + kk] = ev[i];
            }
        }
        if (lane == 0) p.tokens[row] = ids[(int64_t)s * K + index];
        prev = index;
        __syncwarp();  // w and this slot's buffer are rewritten next
    }
}

// ---------------------------------------------------------------------------
// Chain mode (bf16, top_k in (32, 128], rank a multiple of 8 up to 256): one
// CTA of four warps walks one request, so that every request of a large batch
// is resident at once (one CTA per request, a few per SM) and the serial chain
// of a slot is spread over 128 threads and touches shared memory only.
//   - Every candidate id of the request is staged once (int32; -1 marks an id
//     outside the table, whose rows are zero).
//   - Only the predecessor's A row is read: as soon as warp 0 has drawn slot
//     s, its lanes copy the drawn candidate's A row (16-byte cp.async per
//     lane, arrivals on one of two mbarriers) into one of two row slots,
//     which slot s + 1 waits for.  (Copying all K candidates' A rows a slot
//     and a half ahead, the first design, moved 64 times the bytes and left
//     each slot waiting about 3 us for them: 89 against 77 us for the walk
//     stage at batch 512 x 15 slots, K 64, rank 128.)
//   - The B rows of slot s (its candidates) are in a shared B buffer when its
//     edges are formed.  With at most 8 16-byte chunks per thread (top_k <= 64,
//     rank <= 128) each thread loads its own chunks of slot s + 2 into
//     registers while slot s is drawn and stores them into the single B buffer
//     after slot s + 1's edges; otherwise two B buffers are filled by warps
//     1-3 with cp.async, a slot and a half ahead.
//   - Edges: half-warp h owns candidates [h * CPH, (h + 1) * CPH); its lane
//     l16 owns the rank chunks l16 + 16 i of 8 elements, so the 16 lanes read
//     a B row's 256 contiguous bytes per chunk step (no bank conflicts).  Each
//     lane multiplies its chunk of w = A[predecessor] * g (fp32) into the
//     CPH rows, and a reduce-scatter over the 16 lanes leaves each candidate's
//     sum on one lane (two when CPH = 8), which adds the unary value.
//   - Warp 0 takes the slot's draw from the K edges (select_consecutive) and
//     writes q and the path's edges while warps 1-3 issue the copies.
// Measured on GB300 and not kept: one bulk (copy-engine) copy per row (64
// engine operations per group slowed the shuffles and shared-memory loads of
// every warp on the SM); L2 prefetches of the rows ahead (slower, line and
// bulk alike, also for the candidates' A rows ahead of the drawn-row copy);
// four-row copy-engine gathers of the A rows (no change); the
// edges on one warp with the other three only copying, the warps meeting at
// full/free mbarrier pairs instead of block barriers, the edges formed on
// CUDA cores (88 us against 66 at batch 512 x 15 slots, K 64, rank 128) or on
// the legacy tensor-core path (mma.sync on w split exactly into three bf16
// parts: 80-90 us).
// ---------------------------------------------------------------------------
constexpr int kChainThreads = 128;
constexpr int kChainCopyThreads = 96;  // warps 1-3 issue the cp.async copies

struct ChainLayout {
    int row_bytes;   // rank * 2
    int regb;        // B rows staged through registers into one shared buffer
    int slot_floats; // one entry of the slot-data ring: k_splits * rank partials, k unary values, the uniform
    size_t bars, sdat, ids, chosen, esm, ctl, abuf, bbuf, total;
};

__host__ __device__ inline ChainLayout chain_layout(int slots, int k, int rank, int k_splits, bool regb) {
    ChainLayout L;
    L.row_bytes = rank * 2;
    L.regb = regb ? 1 : 0;
    L.slot_floats = (int)((k_splits * rank + k + 1 + 3) / 4 * 4);
    L.bars = 0;                                              // chosen-A, B and slot-data mbarriers (2 each)
    L.sdat = 64;                                             // [2][slot_floats] slot-data ring
    L.ids = L.sdat + (size_t)2 * L.slot_floats * 4;          // [slots][k] ids (-1: outside the table)
    L.chosen = L.ids + pad16((size_t)slots * k * 4);         // [slots] drawn index
    L.esm = L.chosen + pad16((size_t)slots * 4);             // [k] the slot's edges
    L.ctl = L.esm + pad16((size_t)k * 4);                    // abort flag
    L.abuf = L.ctl + 16;                                     // [3] A rows: anchor, chosen (2 slots)
    L.bbuf = L.abuf + pad16((size_t)3 * L.row_bytes);        // [1 or 2][k] B rows
    L.total = L.bbuf + (size_t)(regb ? 1 : 2) * k * L.row_bytes;
    return L;
}

// The table rows tab[ids[c]] (c < K) into dst (row c at c * row_bytes) with
// 16-byte cp.async by the copy threads (t in [0, kChainCopyThreads)); rows
// whose id is -1 are zero-filled by the copies themselves.  Each copy thread
// then arrives on `bar`, whose phase completes once every copy thread's
// copies have landed.  nch = row_bytes / 16 chunks per row; lg = log2(nch)
// when it is a power of two, else -1.
__device__ __forceinline__ void chain_copy_rows(const int32_t *ids, int K, const __nv_bfloat16 *tab,
                                                int R, int nch, int lg, uint8_t *dst, uint64_t *bar,
                                                int t) {
    for (int c = t; c < K * nch; c += kChainCopyThreads) {
        const int row = lg >= 0 ? c >> lg : c / nch;
        const int j = c - row * nch;
        const int64_t id = ids[row];
        cp_async16(dst + (size_t)c * 16,
                   reinterpret_cast<const uint8_t *>(tab + (id >= 0 ? id : 0) * R) + 16 * j, id >= 0);
    }
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ float redux_max(float v) {
    float m;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(v));
    return m;
}

// The draw from one row of K edges held by one warp, lane owning the E
// consecutive candidates k = lane * E + i (invalid: k >= K).  Greedy: the
// smallest index of the maximum, q one-hot.  Sampled: q = softmax(e / T) (T
// already clamped to >= 1e-5; divide, do not multiply by 1 / T), cdf_k = the
// prefix of exp(e / T - max) in candidate order over their total (one warp
// scan of the lanes' sums), index = min(#{k : u >= cdf_k}, K - 1).  Returns
// the index (the same in every lane) and the lane's q values.
template <int E>
__device__ __forceinline__ int select_consecutive(const float (&ev)[E], int K, int lane, bool greedy,
                                                  float temp, float u, float (&qv)[E]) {
    if (greedy) {
        float best = -INFINITY;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const int k = lane * E + i;
            if (k < K && (bi < 0 || ev[i] > best)) {
                best = ev[i];
                bi = k;
            }
        }
        const float m = redux_max(best);
        // the lowest lane holding the maximum holds its smallest index
        const uint32_t has = __ballot_sync(0xFFFFFFFFu, bi >= 0 && best == m);
        const int index = __shfl_sync(0xFFFFFFFFu, bi, __ffs(has) - 1);
#pragma unroll
        for (int i = 0; i < E; ++i) qv[i] = (lane * E + i) == index ? 1.0f : 0.0f;
        return index;
    }
    float sc[E];
    float lm = -INFINITY;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        sc[i] = lane * E + i < K ? ev[i] / temp : -INFINITY;
        lm = fmaxf(lm, sc[i]);
    }
    const float m = redux_max(lm);
    float ex[E];
    float local = 0.0f;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        ex[i] = lane * E + i < K ? expf(sc[i] - m) : 0.0f;
        local += ex[i];
    }
    float incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    const float total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    float run = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
    if (lane == 0) run = 0.0f;
    int count = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        qv[i] = ex[i] / total;
        run += ex[i];
        count += __popc(__ballot_sync(0xFFFFFFFFu, lane * E + i < K && u >= run / total));
    }
    return count < K - 1 ? count : K - 1;
}

// One reduce-scatter step over a half-warp: of N partial sums, a lane keeps
// the lower half (its bit o clear) or the upper half (set), adds the
// partner's copy of the kept half, and moves it to positions [0, N / 2).
template <int N, int CPH>
__device__ __forceinline__ void rs_halve(float (&v)[CPH], int l16, int o) {
    const bool upper = (l16 & o) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float send = upper ? v[i] : v[i + N / 2];
        const float keep = upper ? v[i + N / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
    }
}

// Sum of each of CPH partials over the 16 lanes of a half-warp.  Afterwards
// lane l16 holds the total of candidate l16 (CPH = 16) or l16 >> 1 (CPH = 8;
// lanes l16 and l16 ^ 1 hold the same value).
template <int CPH>
__device__ __forceinline__ float reduce_scatter16(float (&v)[CPH], int l16) {
    static_assert(CPH == 8 || CPH == 16, "eight or sixteen candidates per half-warp");
    if constexpr (CPH == 16) {
        rs_halve<16>(v, l16, 8);
        rs_halve<8>(v, l16, 4);
        rs_halve<4>(v, l16, 2);
        rs_halve<2>(v, l16, 1);
    } else {
        rs_halve<8>(v, l16, 8);
        rs_halve<4>(v, l16, 4);
        rs_halve<2>(v, l16, 2);
        v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], 1);
    }
    return v[0];
}

// Bounded wait of the drain at the end of an aborted chain: the copies still
// in flight into this CTA's shared memory land (or the limit passes) before
// the CTA exits.
__device__ __forceinline__ void chain_drain_wait(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > kWaitLimitNs) return;
}

// This thread's 16-byte B chunks of one slot (rows hw * CPH + i, chunk
// l16 + 16 ch), from global memory into registers (zero past K, past the
// rank, or for an id outside the table).
// Slot-data entry of proposal row `row` into dst by the copy threads with
// cp.async: the projection partials (16-byte copies), the unary values and
// the uniform (4-byte copies); each copy thread then arrives on `bar`.
__device__ __forceinline__ void chain_copy_slot(const WalkParams &p, int64_t row, float *dst, uint64_t *bar,
                                                int t) {
    const int pr4 = p.rank / 4;  // 16-byte chunks of one partial row
    for (int c = t; c < p.k_splits * pr4; c += kChainCopyThreads) {
        const int ks = c / pr4;
        cp_async16(dst + 4 * c, p.g + ks * p.split_stride + row * p.rank + 4 * (c - ks * pr4), true);
    }
    float *du = dst + p.k_splits * p.rank;
    for (int c = t; c <= p.k; c += kChainCopyThreads) {
        const float *src = c < p.k ? p.cand_u + row * p.k + c : p.uniforms + row;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(du + c)), "l"(src) : "memory");
    }
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int CPH, int CH>
__device__ __forceinline__ void chain_load_b(const __nv_bfloat16 *B, const int32_t *ids, int K, int R,
                                             int nch, int hw, int l16, uint4 (&bq)[CPH * CH]) {
#pragma unroll
    for (int i = 0; i < CPH; ++i) {
        const int c = hw * CPH + i;
        const int64_t id = c < K ? ids[c] : -1;
#pragma unroll
        for (int ch = 0; ch < CH; ++ch) {
            const int j = l16 + 16 * ch;
            bq[i * CH + ch] = (id >= 0 && j < nch) ? __ldg(reinterpret_cast<const uint4 *>(B + id * R) + j)
                                                   : make_uint4(0, 0, 0, 0);
        }
    }
}

template <int CPH, int CH>
__device__ __forceinline__ void chain_store_b(uint8_t *bbuf, int row_bytes, int K, int nch, int hw, int l16,
                                              const uint4 (&bq)[CPH * CH]) {
#pragma unroll
    for (int i = 0; i < CPH; ++i) {
        const int c = hw * CPH + i;
#pragma unroll
        for (int ch = 0; ch < CH; ++ch) {
            const int j = l16 + 16 * ch;
            if (c < K && j < nch) *reinterpret_cast<uint4 *>(bbuf + (size_t)c * row_bytes + 16 * j) = bq[i * CH + ch];
        }
    }
}

template <int KM, int CH, bool REGB>
__global__ void __launch_bounds__(kChainThreads, 4)
    walk_chain_kernel(const WalkParams p, ChainLayout L) {
    if (!p.after_projection) grid_dep_wait();
    extern __shared__ __align__(16) uint8_t dyn[];
    constexpr int CPH = KM / 8;  // candidates per half-warp
    constexpr int E = KM / 32;   // candidates per lane of the selecting warp
    constexpr int NBQ = REGB ? CPH * CH : 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hw = tid >> 4, l16 = tid & 15;
    const int ct = tid - 32;  // copy thread index (warps 1-3)
    const int b = blockIdx.x;
    const int S = p.slots, K = p.k, R = p.rank;
    const int nch = R / 8;
    const size_t gbytes = (size_t)K * L.row_bytes;  // one buffer of K rows
    uint64_t *abar = reinterpret_cast<uint64_t *>(dyn + L.bars);  // [2]
    uint64_t *bbar = abar + 2;                                     // [2], two-buffer B only
    uint64_t *sbar = abar + 4;                                     // [2] slot-data ring
    float *sdat = reinterpret_cast<float *>(dyn + L.sdat);
    int32_t *ids = reinterpret_cast<int32_t *>(dyn + L.ids);
    int32_t *chosen = reinterpret_cast<int32_t *>(dyn + L.chosen);
    float *esm = reinterpret_cast<float *>(dyn + L.esm);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(dyn + L.ctl);
    uint8_t *abuf = dyn + L.abuf;
    uint8_t *bbuf = dyn + L.bbuf;
    const int64_t row0 = (int64_t)b * S;
    const __nv_bfloat16 *A = static_cast<const __nv_bfloat16 *>(p.A);
    const __nv_bfloat16 *B = static_cast<const __nv_bfloat16 *>(p.B);

    if (tid == 0) {
        // abar[0..1]: the chosen A row, copied by the nch lanes of warp 0;
        // bbar, sbar: the copy threads (warps 1-3)
        for (int i = 0; i < 2; ++i) mbar_init(&abar[i], (uint32_t)(R / 8));
        for (int i = 2; i < 6; ++i) mbar_init(&abar[i], kChainCopyThreads);
        *abort_flag = 0;
        fence_mbar_init();
    }
    const int lg = (nch & (nch - 1)) == 0 ? __ffs(nch) - 1 : -1;
    // every candidate id of the request, once
    bool bad = false;
    for (int t = tid; t < S * K; t += kChainThreads) {
        const int64_t id = p.cand[row0 * K + t];
        const bool ok = id_ok(id, p.table_rows);
        bad |= !ok;
        ids[t] = ok ? (int32_t)id : -1;
    }
    const int64_t anchor = p.anchors[b];
    const bool anchor_ok = id_ok(anchor, p.table_rows);
    bad |= tid == 0 && !anchor_ok;
    if (__syncthreads_or(bad) && tid == 0 && p.err) atomicOr(p.err, DFLASH2_DEVERR_ID_RANGE);
    // slot 0's predecessor: the anchor's A row (row 0 of the A rows)
    for (int j = tid; j < nch; j += kChainThreads)
        reinterpret_cast<uint4 *>(abuf)[j] =
            anchor_ok ? __ldg(reinterpret_cast<const uint4 *>(A + anchor * R) + j) : make_uint4(0, 0, 0, 0);
    // B rows of slots 0 and 1
    uint4 bq[NBQ];
    if constexpr (!REGB) {
        if (warp > 0) {
            chain_copy_rows(ids, K, B, R, nch, lg, bbuf, &bbar[0], ct);
            if (S > 1) chain_copy_rows(ids + K, K, B, R, nch, lg, bbuf + gbytes, &bbar[1], ct);
        }
    } else {
        chain_load_b<CPH, CH>(B, ids, K, R, nch, hw, l16, bq);
        chain_store_b<CPH, CH>(bbuf, L.row_bytes, K, nch, hw, l16, bq);
        if (S > 1) chain_load_b<CPH, CH>(B, ids + K, K, R, nch, hw, l16, bq);
    }
    // Up to here the kernel has read only the candidates, anchors and tables;
    // the slot data (the projection partials, written by the kernel before
    // this one) after the grid dependency.
    grid_dep_wait();
    if (warp > 0) {
        chain_copy_slot(p, row0, sdat, &sbar[0], ct);
        if (S > 1) chain_copy_slot(p, row0 + 1, sdat + L.slot_floats, &sbar[1], ct);
    }

    // the lane that adds the unary value and stores candidate cw's edge
    const int iw = CPH == 16 ? l16 : (l16 >> 1);
    const int cw = hw * CPH + iw;
    const bool writer = (CPH == 16 || (l16 & 1) == 0) && cw < K;
    const bool greedy = p.greedy[b] != 0;
    float temp = p.temps[b];
    if (!(temp >= 1e-5f)) temp = 1e-5f;
    __syncthreads();  // the anchor row and slot 0's B rows (register path) are visible

    int s = 0;
    for (; s < S; ++s) {
        const int64_t row = row0 + s;
        // the slot's projection (its partials summed in split order), unary
        // value and uniform, copied two slots ahead
        mbar_wait(&sbar[s & 1], (uint32_t)(s >> 1) & 1u, abort_flag, p.err);
        const float *sd = sdat + (size_t)(s & 1) * L.slot_floats;
        float g[8 * CH];
#pragma unroll
        for (int ch = 0; ch < CH; ++ch) {
            const int j = l16 + 16 * ch;
            float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
            if (j < nch) {
                lo = *reinterpret_cast<const float4 *>(sd + 8 * j);
                hi = *reinterpret_cast<const float4 *>(sd + 8 * j + 4);
                for (int ks = 1; ks < p.k_splits; ++ks) {
                    const float4 a = *reinterpret_cast<const float4 *>(sd + ks * R + 8 * j);
                    const float4 c = *reinterpret_cast<const float4 *>(sd + ks * R + 8 * j + 4);
                    lo.x += a.x; lo.y += a.y; lo.z += a.z; lo.w += a.w;
                    hi.x += c.x; hi.y += c.y; hi.z += c.z; hi.w += c.w;
                }
            }
            g[8 * ch + 0] = lo.x; g[8 * ch + 1] = lo.y; g[8 * ch + 2] = lo.z; g[8 * ch + 3] = lo.w;
            g[8 * ch + 4] = hi.x; g[8 * ch + 5] = hi.y; g[8 * ch + 6] = hi.z; g[8 * ch + 7] = hi.w;
        }
        const float cu = writer ? sd[p.k_splits * R + cw] : 0.0f;
        const float uni = sd[p.k_splits * R + K];
        // w = A[predecessor] * g on this lane's chunks: slot 0 reads the anchor
        // (A row 0), slot s the row drawn at slot s - 1 (A row 1 + (s - 1) % 2,
        // copied by warp 0 as soon as it drew it)
        if (s > 0) mbar_wait(&abar[(s - 1) & 1], (uint32_t)((s - 1) >> 1) & 1u, abort_flag, p.err);
        const uint8_t *arow = abuf + (size_t)(s > 0 ? 1 + ((s - 1) & 1) : 0) * L.row_bytes;
        float2 w[4 * CH];
#pragma unroll
        for (int ch = 0; ch < CH; ++ch) {
            const int j = l16 + 16 * ch;
            const uint4 av = j < nch ? *reinterpret_cast<const uint4 *>(arow + 16 * j) : make_uint4(0, 0, 0, 0);
            const __nv_bfloat162 *ap = reinterpret_cast<const __nv_bfloat162 *>(&av);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                w[4 * ch + e] = __fmul2_rn(__bfloat1622float2(ap[e]),
                                           make_float2(g[8 * ch + 2 * e], g[8 * ch + 2 * e + 1]));
        }
        // the slot's B rows
        const uint8_t *brows = bbuf;
        if constexpr (!REGB) {
            mbar_wait(&bbar[s & 1], (uint32_t)(s >> 1) & 1u, abort_flag, p.err);
            brows = bbuf + (size_t)(s & 1) * gbytes;
        }
        float part[CPH];
#pragma unroll
        for (int i = 0; i < CPH; ++i) {
            const int c = hw * CPH + i;
            float2 acc = make_float2(0.0f, 0.0f);
            if (c < K) {
#pragma unroll
                for (int ch = 0; ch < CH; ++ch) {
                    const int j = l16 + 16 * ch;
                    if (j < nch) {
                        const uint4 bv = *reinterpret_cast<const uint4 *>(brows + (size_t)c * L.row_bytes + 16 * j);
                        const __nv_bfloat162 *bp = reinterpret_cast<const __nv_bfloat162 *>(&bv);
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc = __ffma2_rn(w[4 * ch + e], __bfloat1622float2(bp[e]), acc);
                    }
                }
            }
            part[i] = acc.x + acc.y;
        }
        const float total = reduce_scatter16<CPH>(part, l16);
        if (writer) esm[cw] = total + cu;
        __syncthreads();
        if (*abort_flag) break;
        if (warp == 0) {
            float ev[E], qv[E];
#pragma unroll
            for (int i = 0; i < E; ++i) {
                const int k = lane * E + i;
                ev[i] = k < K ? esm[k] : -INFINITY;
            }
            const int index = select_consecutive<E>(ev, K, lane, greedy, temp, uni, qv);
            if (s + 1 < S && lane < nch) {
                // the drawn candidate's A row, the next slot's predecessor (a row
                // outside the table: zeros)
                const int32_t id = ids[(size_t)s * K + index];
                cp_async16(abuf + (size_t)(1 + (s & 1)) * L.row_bytes + 16 * lane,
                           reinterpret_cast<const uint8_t *>(A + (id >= 0 ? id : 0) * R) + 16 * lane,
                           id >= 0);
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                                 smem_u32(&abar[s & 1]))
                             : "memory");
            }
#pragma unroll
            for (int i = 0; i < E; ++i) {
                const int k = lane * E + i;
                if (k < K) {
                    p.q[row * K + k] = qv[i];
                    if (p.path_scores) p.path_scores[row * K + k] = ev[i];
                }
            }
            if (lane == 0) chosen[s] = index;
        } else {
            // slot s + 2's data and B rows into the entries slot s just read
            if (s + 2 < S)
                chain_copy_slot(p, row + 2, sdat + (size_t)(s & 1) * L.slot_floats, &sbar[s & 1], ct);
            if constexpr (!REGB) {
                if (s + 2 < S)
                    chain_copy_rows(ids + (size_t)(s + 2) * K, K, B, R, nch, lg, bbuf + (size_t)(s & 1) * gbytes,
                                    &bbar[s & 1], ct);
            }
        }
        if constexpr (REGB) {
            // slot s + 1's B chunks (loaded a slot ago) into the B buffer, then
            // slot s + 2's from global memory
            if (s + 1 < S) chain_store_b<CPH, CH>(bbuf, L.row_bytes, K, nch, hw, l16, bq);
            if (s + 2 < S) chain_load_b<CPH, CH>(B, ids + (size_t)(s + 2) * K, K, R, nch, hw, l16, bq);
        }
        __syncthreads();
    }
    // the tokens of the walked slots: the raw candidate ids
    for (int t = tid; t < s; t += kChainThreads)
        p.tokens[row0 + t] = p.cand[(row0 + t) * K + chosen[t]];
    // after an abort: let the copies still in flight land before exiting
    if (s < S && tid < nch) asm volatile("cp.async.wait_all;" ::: "memory");  // warp 0's row copies
    if (s < S && tid == 32) {
        for (int t = s - 1; t <= s + 1 && t < S; ++t) {
            if (!REGB && t >= 0) chain_drain_wait(&bbar[t & 1], (uint32_t)(t >> 1) & 1u);
            if (t >= 0) chain_drain_wait(&sbar[t & 1], (uint32_t)(t >> 1) & 1u);
        }
    }
}

// ---------------------------------------------------------------------------
// Lattice mode (top_k <= 32), two kernels.  Slot s's possible predecessors are
// exactly slot s-1's candidates (the anchor at slot 0), so every slot's K x K
// edges and the draw from every (slot, predecessor) row can be formed in
// parallel before the walk; the walk itself is then a chase through the
// per-row draws.
//   walk_rows_kernel, grid (batch, parts): a CTA forms the rows of a range of
//     slots of one request and writes their edges, softmax statistics and
//     draws to the workspace.  Parts spread a request over several SMs: one
//     SM per request was bound by its instruction issue.  A row is formed by
//     kLatGroup adjacent lanes (K / kLatGroup consecutive candidates each),
//     and its sums run in candidate order, as the sequential sums of the
//     walk's definition: the running value passes from lane to lane by
//     shuffles.
//   walk_chase_kernel, one CTA per request: follows the draws slot by slot
//     and writes the walked path's tokens, q and edges.
// ---------------------------------------------------------------------------
constexpr int kLatticeMaxK = 32;
constexpr int kRowThreads = 256;
constexpr int kLatGroup = 4;
constexpr int kChaseThreads = 256;

struct RowsLayout {
    int a_stride;   // bytes per staged A row (rank * esz + 16)
    int b_stride;   // bytes per staged B row (rank * esz + 16)
    int b_slot;     // bytes per slot of B rows (k * b_stride + 16)
    size_t ids, cu, uni, gs, brow, arow, total;
};

// Shared memory of a CTA covering spp slots: the ids of those slots and of the
// slot before them, their unary values, uniforms, projections, and the staged
// B (candidate) and A (predecessor) rows.
__host__ __device__ inline RowsLayout rows_layout(int spp, int k, int rank, int esz) {
    RowsLayout L;
    L.a_stride = rank * esz + 16;
    L.b_stride = rank * esz + 16;
    L.b_slot = k * L.b_stride + 16;
    L.ids = 0;
    L.cu = L.ids + pad16((size_t)(spp + 1) * k * 8);
    L.uni = L.cu + pad16((size_t)spp * k * 4);
    L.gs = L.uni + pad16((size_t)spp * 4);
    L.brow = L.gs + pad16((size_t)spp * rank * 4);
    L.arow = L.brow + (size_t)spp * L.b_slot;
    L.total = L.arow + pad16((size_t)spp * k * L.a_stride);
    return L;
}

// The lattice of every request in the workspace.
struct LatticeWs {
    float *lat;    // [batch][slots][K][K] edges, row (slot, predecessor)
    float2 *stat;  // [batch][slots][K] (max of e / T, sum of exp) of sampled rows
    int32_t *nxt;  // [batch][slots][K] the candidate drawn from each row
};

inline size_t align256w(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace offsets of the lattice buffers (after the projection partials).
inline void lattice_ws_layout(int64_t rows, int k, size_t base, size_t *lat, size_t *stat,
                              size_t *nxt, size_t *end) {
    *lat = align256w(base);
    *stat = align256w(*lat + (size_t)rows * k * k * 4);
    *nxt = align256w(*stat + (size_t)rows * k * 8);
    *end = align256w(*nxt + (size_t)rows * k * 4);
}

template <typename T, int KM>
__global__ void __launch_bounds__(kRowThreads)
    walk_rows_kernel(const WalkParams p, RowsLayout L, int spp, LatticeWs ws) {
    grid_dep_wait();
    extern __shared__ __align__(16) uint8_t dyn[];
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const int S = p.slots, K = p.k, R = p.rank;
    const int s0 = blockIdx.y * spp;
    if (s0 >= S) return;
    const int s1 = min(S, s0 + spp), ns = s1 - s0;
    const int sf = s0 > 0 ? s0 - 1 : 0;  // first slot whose ids are staged
    const int nid = s1 - sf;
    int64_t *ids = reinterpret_cast<int64_t *>(dyn + L.ids);  // [nid][K]: slot sf + i
    float *cu = reinterpret_cast<float *>(dyn + L.cu);        // [ns][K]: slot s0 + i
    float *uni = reinterpret_cast<float *>(dyn + L.uni);
    float *gs = reinterpret_cast<float *>(dyn + L.gs);
    uint8_t *brow = dyn + L.brow;
    uint8_t *arow = dyn + L.arow;
    const int64_t row0 = (int64_t)b * S;
    const T *A = static_cast<const T *>(p.A);
    const T *B = static_cast<const T *>(p.B);

    // ---- prologue
    bool bad = false;
    for (int t = tid; t < nid * K; t += kRowThreads) {
        const int64_t c = p.cand[(row0 + sf) * K + t];
        bad |= !id_ok(c, p.table_rows);
        ids[t] = c;
    }
    for (int t = tid; t < ns * K; t += kRowThreads) cu[t] = p.cand_u[(row0 + s0) * K + t];
    for (int t = tid; t < ns; t += kRowThreads) uni[t] = p.uniforms[row0 + s0 + t];
    {
        const float4 *g4 = reinterpret_cast<const float4 *>(p.g + (row0 + s0) * R);
        const int64_t stride4 = p.split_stride / 4;
        float4 *gs4 = reinterpret_cast<float4 *>(gs);
        for (int t = tid; t < ns * R / 4; t += kRowThreads) {
            float4 acc = g4[t];
            for (int ks = 1; ks < p.k_splits; ++ks) {
                const float4 v = g4[ks * stride4 + t];
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            gs4[t] = acc;
        }
    }
    const int64_t anchor = p.anchors[b];
    bad |= !id_ok(anchor, p.table_rows);
    if (__syncthreads_or(bad) && tid == 0 && p.err) atomicOr(p.err, DFLASH2_DEVERR_ID_RANGE);

    // ---- gather the rows of the range (16-byte copies, zero rows for bad ids):
    // B row (ls, kk) = candidate kk of slot s0 + ls; A row (ls, kp) = predecessor
    // kp of that slot (slot 0: the anchor, as row (0, 0))
    const int chunks = R * (int)sizeof(T) / 16;
    const int n_rows = ns * K;
    for (int t = tid; t < 2 * n_rows * chunks; t += kRowThreads) {
        const int r = t / chunks;
        const int ch = t - r * chunks;
        if (r < n_rows) {
            const int ls = r / K, kk = r - ls * K;
            const int64_t c = ids[(s0 + ls - sf) * K + kk];
            const bool ok = id_ok(c, p.table_rows);
            cp_async16(brow + (size_t)ls * L.b_slot + (size_t)kk * L.b_stride + ch * 16,
                       reinterpret_cast<const uint8_t *>(ok ? B + c * R : B) + ch * 16, ok);
        } else {
            const int ar = r - n_rows;
            const int ls = ar / K, kp = ar - ls * K;
            const int s = s0 + ls;
            const int64_t c = s == 0 ? (kp == 0 ? anchor : -1) : ids[(s - 1 - sf) * K + kp];
            const bool ok = id_ok(c, p.table_rows);
            cp_async16(arow + (size_t)ar * L.a_stride + ch * 16,
                       reinterpret_cast<const uint8_t *>(ok ? A + c * R : A) + ch * 16, ok);
        }
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    // ---- every lattice row of the range: K edges, then the row's draw.  The
    // kLatGroup lanes of a row hold candidates kk = g * KPT + q (q < KPT).
    const bool greedy = p.greedy[b] != 0;
    float temp = p.temps[b];
    if (!(temp >= 1e-5f)) temp = 1e-5f;
    constexpr int VN = 16 / sizeof(T);
    constexpr int KPT = KM / kLatGroup;
    const int g = tid & (kLatGroup - 1);
    const int gbase = (tid & 31) & ~(kLatGroup - 1);  // lane of the row's first member
    for (int base = 0; base < n_rows; base += kRowThreads / kLatGroup) {  // uniform trip count
        const int r = base + tid / kLatGroup;
        const int ls = r / K, kp = r - (r / K) * K;
        const int s = s0 + ls;
        // slot 0 has the anchor row only
        const bool active = r < n_rows && !(s == 0 && kp > 0);
        float acc[KPT];
#pragma unroll
        for (int q = 0; q < KPT; ++q) acc[q] = 0.0f;
        if (active) {
            const uint8_t *ar = arow + (size_t)r * L.a_stride;
            const uint8_t *bs = brow + (size_t)ls * L.b_slot;
            const float *gsl = gs + (size_t)ls * R;
            for (int v = 0; v < R / VN; ++v) {
                float av[VN], w[VN];
                unpack16<T>(*reinterpret_cast<const uint4 *>(ar + v * 16), av);
#pragma unroll
                for (int e = 0; e < VN; ++e) w[e] = av[e] * gsl[v * VN + e];
#pragma unroll
                for (int q = 0; q < KPT; ++q) {
                    const int kk = g * KPT + q;
                    if (kk < K) {
                        float bv[VN];
                        unpack16<T>(*reinterpret_cast<const uint4 *>(bs + (size_t)kk * L.b_stride + v * 16), bv);
#pragma unroll
                        for (int e = 0; e < VN; ++e) acc[q] = fmaf(w[e], bv[e], acc[q]);
                    }
                }
            }
        }
        const int64_t lrow_i = ((row0 + s) * K + kp);  // this row's index in the workspace
        float ev[KPT];
#pragma unroll
        for (int q = 0; q < KPT; ++q) {
            const int kk = g * KPT + q;
            ev[q] = (active && kk < K) ? acc[q] + cu[ls * K + kk] : -INFINITY;
            if (active && kk < K) ws.lat[lrow_i * K + kk] = ev[q];
        }
        int index = 0;
        if (greedy) {
            // first maximum in candidate order: per lane, then across the row's lanes
            float best = -INFINITY;
            int bi = K;
#pragma unroll
            for (int q = 0; q < KPT; ++q) {
                const int kk = g * KPT + q;
                if (kk < K && (bi == K || ev[q] > best)) {
                    best = ev[q];
                    bi = kk;
                }
            }
#pragma unroll
            for (int o = 1; o < kLatGroup; o <<= 1) {
                const float b2 = __shfl_xor_sync(0xFFFFFFFFu, best, o);
                const int i2 = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
                if (i2 < K && (bi == K || b2 > best || (b2 == best && i2 < bi))) {
                    best = b2;
                    bi = i2;
                }
            }
            index = bi;
        } else {
            float x[KPT];
            float mx = -INFINITY;
#pragma unroll
            for (int q = 0; q < KPT; ++q) {
                const int kk = g * KPT + q;
                x[q] = kk < K ? ev[q] / temp : -INFINITY;
                mx = fmaxf(mx, x[q]);
            }
#pragma unroll
            for (int o = 1; o < kLatGroup; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
#pragma unroll
            for (int q = 0; q < KPT; ++q) x[q] = g * KPT + q < K ? expf(x[q] - mx) : 0.0f;
            // total = the K terms summed in candidate order, lane after lane
            float run = 0.0f, prev = 0.0f;
#pragma unroll
            for (int h = 0; h < kLatGroup; ++h) {
                if (g == h) {
                    run = prev;
#pragma unroll
                    for (int q = 0; q < KPT; ++q)
                        if (g * KPT + q < K) run += x[q];
                }
                prev = __shfl_sync(0xFFFFFFFFu, run, gbase + h);
            }
            const float total = prev;
            const float u = uni[ls < ns ? ls : 0];
            // cdf_k = sequential prefix of x_k / total; count of u >= cdf_k
            float cdf = 0.0f;
            int count = 0;
            prev = 0.0f;
#pragma unroll
            for (int h = 0; h < kLatGroup; ++h) {
                if (g == h) {
                    cdf = prev;
#pragma unroll
                    for (int q = 0; q < KPT; ++q) {
                        if (g * KPT + q < K) {
                            cdf += x[q] / total;
                            count += (u >= cdf) ? 1 : 0;
                        }
                    }
                }
                prev = __shfl_sync(0xFFFFFFFFu, cdf, gbase + h);
            }
#pragma unroll
            for (int o = 1; o < kLatGroup; o <<= 1) count += __shfl_xor_sync(0xFFFFFFFFu, count, o);
            index = count < K - 1 ? count : K - 1;
            if (active && g == 0) ws.stat[lrow_i] = make_float2(mx, total);
        }
        if (active && g == 0) ws.nxt[lrow_i] = index;
    }
}

__global__ void __launch_bounds__(kChaseThreads)
    walk_chase_kernel(const WalkParams p, LatticeWs ws) {
    grid_dep_wait();
    extern __shared__ __align__(16) int32_t chase_smem[];
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const int S = p.slots, K = p.k;
    int32_t *nxt = chase_smem;       // [S][K]
    int32_t *path = chase_smem + S * K;
    const int64_t row0 = (int64_t)b * S;
    for (int t = tid; t < S * K; t += kChaseThreads) nxt[t] = ws.nxt[row0 * K + t];
    __syncthreads();
    // the walk: follow the drawn index slot by slot (slot 0 from the anchor row)
    if (tid == 0) {
        int prev = 0;
        for (int s = 0; s < S; ++s) {
            prev = nxt[s * K + prev];
            path[s] = prev;
        }
    }
    __syncthreads();
    const bool greedy = p.greedy[b] != 0;
    float temp = p.temps[b];
    if (!(temp >= 1e-5f)) temp = 1e-5f;
    for (int t = tid; t < S * K; t += kChaseThreads) {
        const int s = t / K, kk = t - s * K;
        const int kp = s == 0 ? 0 : path[s - 1];
        const int64_t lrow_i = (row0 + s) * K + kp;
        const float e = ws.lat[lrow_i * K + kk];
        float qv;
        if (greedy) {
            qv = kk == path[s] ? 1.0f : 0.0f;
        } else {
            const float2 st = ws.stat[lrow_i];
            qv = expf(e / temp - st.x) / st.y;
        }
        p.q[(row0 + s) * K + kk] = qv;
        if (p.path_scores) p.path_scores[(row0 + s) * K + kk] = e;
    }
    for (int s = tid; s < S; s += kChaseThreads) p.tokens[row0 + s] = p.cand[(row0 + s) * K + path[s]];
}

__global__ void __launch_bounds__(128)
    project_f32_kernel(const float *__restrict__ h, const float *__restrict__ proj, int hidden,
                       int rank, float *g) {
    grid_dep_wait();
    const int64_t m = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *hr = h + m * hidden;
    for (int j = warp; j < rank; j += 4) {
        const float *pr = proj + (int64_t)j * hidden;
        float acc = 0.0f;
        for (int i = lane; i < hidden; i += 32) acc = fmaf(hr[i], pr[i], acc);
        acc = warp_sum(acc);
        if (lane == 0) g[m * rank + j] = acc;
    }
}

// Tiling of the tensor-core projection (bf16); it depends on the shape only,
// so the workspace size does not depend on the device.
//   - Batches of at least 4096 rows run on CTA pairs with the tokens as the
//     weight side (256 rows a pair, 128 a CTA) and the projection matrix as
//     one token tile: each CTA stages 128 token rows and half of the matrix
//     per stage, so four stages keep 128 KB of h in flight per SM.  The
//     hidden dimension is split so that the pairs cover a 152-SM GB300
//     (76 pairs) about once.
//   - Smaller batches run one CTA per tile of 16 tokens, split over hidden
//     into enough items for the SMs.
// The walk sums the partials in a fixed order.
struct ProjTiling {
    bool pairs;
    int bn;
    int k_splits;
};

inline ProjTiling proj_tiling(int64_t rows, int hidden, int rank) {
    ProjTiling t{};
    const int num_kb = (hidden + kGemmStageK - 1) / kGemmStageK;
    int64_t ks;
    if (rows >= 4096) {
        t.pairs = true;
        t.bn = (rank + 15) / 16 * 16;
        ks = 76 / ((rows + 2 * kGemmTileW - 1) / (2 * kGemmTileW));
    } else {
        t.pairs = false;
        t.bn = 16;
        const int64_t tiles = (rows + t.bn - 1) / t.bn;
        ks = (148 + tiles - 1) / tiles;
    }
    if (ks > num_kb) ks = num_kb;
    if (ks > 8) ks = 8;
    if (ks < 1) ks = 1;
    t.k_splits = (int)ks;
    return t;
}

// Projection partials the workspace reserves (the tiling's split count before
// the GEMM launcher trims it; 1 for fp32).
inline int ksplits_ws(int64_t rows, int hidden, int rank, int32_t dtype) {
    return dtype == DFLASH2_BF16 ? proj_tiling(rows, hidden, rank).k_splits : 1;
}

std::atomic<bool> g_walk_attr[64];  // per device; the attribute calls are idempotent

}  // namespace
}  // namespace dflash2

using namespace dflash2;

extern "C" size_t dflash2_selector_walk_workspace_size(int32_t batch, int32_t slots, int32_t hidden,
                                                       int32_t rank, int32_t top_k, int32_t dtype) {
    if (batch <= 0 || slots <= 0 || hidden <= 0 || rank <= 0 || top_k <= 0) return 0;
    const int64_t rows = (int64_t)batch * slots;
    const size_t partials = (size_t)ksplits_ws(rows, hidden, rank, dtype) * rows * rank * sizeof(float);
    if (top_k > kLatticeMaxK) return partials;
    size_t o_lat, o_stat, o_nxt, o_end;
    lattice_ws_layout(rows, top_k, partials, &o_lat, &o_stat, &o_nxt, &o_end);
    return o_end;
}

namespace {

// Checks shared by the walk entry points, before any pointer is looked at.
dflash2_status check_walk_shape(int32_t batch, int32_t slots, int32_t hidden, int32_t rank,
                                int32_t top_k, int32_t dtype) {
    if (dtype != DFLASH2_F32 && dtype != DFLASH2_BF16) return DFLASH2_ERR_UNSUPPORTED_DTYPE;
    const int rank_mult = dtype == DFLASH2_BF16 ? 8 : 4;
    if (batch < 0 || slots < 0 || hidden <= 0 || rank <= 0 || rank > kMaxRank ||
        rank % rank_mult != 0 || top_k <= 0 || top_k > kMaxK)
        return DFLASH2_ERR_INVALID_ARG;
    return DFLASH2_OK;
}

// Projection partials the walk sums: the tiling's split count as the GEMM
// launcher trims it (every split gets at least one pipeline stage).
int kept_ksplits(int64_t rows, int hidden, int rank, int32_t dtype) {
    if (dtype != DFLASH2_BF16) return 1;
    const int ks = proj_tiling(rows, hidden, rank).k_splits;
    const int num_kb = (hidden + kGemmStageK - 1) / kGemmStageK;
    const int per = (num_kb + ks - 1) / ks;
    return (num_kb + per - 1) / per;
}

// Step a5: g = h . proj^T as k-split fp32 partials at the start of the workspace.
dflash2_status run_projection(const DeviceInfo &di, const void *h, const void *proj, int64_t rows,
                              int32_t hidden, int32_t rank, int32_t dtype, float *g,
                              int32_t *err_word, cudaStream_t st) {
    if (dtype == DFLASH2_BF16) {
        if (hidden % 8 != 0 || !aligned16(h) || !aligned16(proj)) return DFLASH2_ERR_MISALIGNED;
        const ProjTiling t = proj_tiling(rows, hidden, rank);
        GemmParams p{};
        p.hidden = hidden;
        p.bn = t.bn;
        p.k_splits = t.k_splits;
        p.out = g;
        p.ldo = rank;
        p.split_stride = rows * rank;
        p.err = err_word;
        if (t.pairs) {  // g[m, :] row by row: the tokens on the weight side
            p.rows_w = (int32_t)rows;
            p.rows_h = rank;
            p.mode = kGemmStoreRows;
            return launch_gemm_tc(di, h, proj, p, st, /*pair=*/true);
        }
        p.rows_w = rank;
        p.rows_h = (int32_t)rows;
        p.mode = kGemmStore;
        return launch_gemm_tc(di, proj, h, p, st);
    }
    if ((reinterpret_cast<uintptr_t>(h) | reinterpret_cast<uintptr_t>(proj)) % 4 != 0)
        return DFLASH2_ERR_MISALIGNED;
    launch_k(project_f32_kernel, (unsigned)rows, 128, 0, st, static_cast<const float *>(h),
             static_cast<const float *>(proj), hidden, rank, g);
    return launch_status();
}

dflash2_status set_walk_attributes(const DeviceInfo &di) {
    if (di.device < 0 || di.device >= 64 || g_walk_attr[di.device]) return DFLASH2_OK;
    const int bytes = (int)kWalkSmemBytes;
    cudaError_t e = cudaSuccess;
#define DFLASH2_WALK_ATTR(T_, PA_, E_)                                                          \
    if (e == cudaSuccess)                                                                      \
        e = cudaFuncSetAttribute(walk_kernel<T_, PA_, E_>,                                     \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)
    DFLASH2_WALK_ATTR(__nv_bfloat16, true, 1); DFLASH2_WALK_ATTR(__nv_bfloat16, true, 2);
    DFLASH2_WALK_ATTR(__nv_bfloat16, true, 4); DFLASH2_WALK_ATTR(__nv_bfloat16, false, 1);
    DFLASH2_WALK_ATTR(__nv_bfloat16, false, 2); DFLASH2_WALK_ATTR(__nv_bfloat16, false, 4);
    DFLASH2_WALK_ATTR(float, true, 1); DFLASH2_WALK_ATTR(float, true, 2);
    DFLASH2_WALK_ATTR(float, true, 4); DFLASH2_WALK_ATTR(float, false, 1);
    DFLASH2_WALK_ATTR(float, false, 2); DFLASH2_WALK_ATTR(float, false, 4);
#undef DFLASH2_WALK_ATTR
#define DFLASH2_LAT_ATTR(T_, KM_)                                                               \
    if (e == cudaSuccess)                                                                      \
        e = cudaFuncSetAttribute(walk_rows_kernel<T_, KM_>,                                    \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)
    DFLASH2_LAT_ATTR(__nv_bfloat16, 8); DFLASH2_LAT_ATTR(__nv_bfloat16, 16);
    DFLASH2_LAT_ATTR(__nv_bfloat16, 32); DFLASH2_LAT_ATTR(float, 8);
    DFLASH2_LAT_ATTR(float, 16); DFLASH2_LAT_ATTR(float, 32);
#undef DFLASH2_LAT_ATTR
#define DFLASH2_CHAIN_ATTR(KM_, CH_, RB_)                                                       \
    if (e == cudaSuccess)                                                                      \
        e = cudaFuncSetAttribute(walk_chain_kernel<KM_, CH_, RB_>,                             \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)
    DFLASH2_CHAIN_ATTR(64, 1, true); DFLASH2_CHAIN_ATTR(64, 2, false);
    DFLASH2_CHAIN_ATTR(128, 1, false); DFLASH2_CHAIN_ATTR(128, 2, false);
#undef DFLASH2_CHAIN_ATTR
    if (e != cudaSuccess) {
        cudaGetLastError();
        return DFLASH2_ERR_CUDA;
    }
    g_walk_attr[di.device] = true;
    return DFLASH2_OK;
}

// Steps a6-a7 from the projection partials at the start of the workspace.
dflash2_status run_walk(const DeviceInfo &di, WalkParams wp, int32_t hidden, int32_t dtype,
                        void *workspace, cudaStream_t st) {
    const int batch = wp.batch, slots = wp.slots, rank = wp.rank, top_k = wp.k;
    const int esz = dtype == DFLASH2_BF16 ? 2 : 4;
    const int64_t rows = (int64_t)batch * slots;
    const int ksplits = kept_ksplits(rows, hidden, rank, dtype);
    // Lattice mode (top_k <= 32): the request's slots in parts of spp slots,
    // enough parts that the batch gives each SM about two CTAs, when a part's
    // rows fit in shared memory; the lattice itself lives in the workspace.
    // about two CTAs per SM (measured on GB300 against one: even at batch 32,
    // 63 -> 56 us at batch 64 x 15 slots, 45 -> 41 us at batch 128 x 11 slots)
    int parts = (int)((2 * di.sm_count + batch - 1) / batch);
    if (parts > slots) parts = slots;
    if (parts < 1) parts = 1;
    const int spp = (slots + parts - 1) / parts;
    parts = (slots + spp - 1) / spp;
    const RowsLayout RL = rows_layout(spp, top_k, rank, esz);
    const bool lattice = top_k <= kLatticeMaxK && RL.total <= kWalkSmemBytes;
    // Chain mode (bf16 beyond the lattice): the deepest ring that still lets
    // every request's CTA be resident at once, else the shallowest (the most
    // CTAs per SM).
    // Chain mode (bf16 beyond the lattice): B rows staged through registers
    // when a thread's share is at most 8 chunks (top_k <= 64, rank <= 128),
    // else two shared B buffers.
    const bool regb = top_k <= 64 && rank <= 128;
    const ChainLayout CL = chain_layout(slots, top_k, rank, ksplits, regb);
    const bool chain = !lattice && dtype == DFLASH2_BF16 && rank % 8 == 0 && rank <= kMaxRank &&
                       wp.table_rows <= INT32_MAX && CL.total <= kWalkSmemBytes;
    // One warp per request.  Among the shared-memory layouts that fit, take
    // the fewest waves of CTAs, then A-row prefetch, then the deepest
    // prefetch ring (every slot in flight at most).
    bool prefetch_a = false;
    WalkLayout L{};
    int warps = 0;
    {
        const int max_ring = slots < 2 ? 2 : (slots < kMaxRing ? slots : kMaxRing);
        int64_t best_waves = INT64_MAX;
        int best_pa = -1;
        for (int pa = 1; pa >= 0; --pa) {
            for (int nb = max_ring; nb >= 2; --nb) {
                const WalkLayout c = walk_layout(slots, top_k, rank, esz, pa != 0, nb, ksplits);
                int wpc = (int)(kWalkSmemBytes / c.total);
                if (wpc < 1) continue;
                if (wpc > kMaxWarpsPerCta) wpc = kMaxWarpsPerCta;
                const int64_t ctas = (batch + wpc - 1) / wpc;
                int64_t per_sm = (int64_t)(227 * 1024) / (int64_t)(wpc * c.total + 1024);
                if (per_sm < 1) per_sm = 1;
                const int64_t waves = (ctas + di.sm_count * per_sm - 1) / (di.sm_count * per_sm);
                if (waves < best_waves) {  // ties keep the earlier (A prefetch, deeper ring)
                    best_waves = waves;
                    best_pa = pa;
                    L = c;
                    warps = wpc;
                }
            }
        }
        if (best_pa < 0 && !lattice && !chain) return DFLASH2_ERR_INVALID_ARG;  // one request's state exceeds shared memory
        // one mbarrier phase counts fewer than 2^20 transaction bytes
        if (!lattice && !chain &&
            (int64_t)ksplits * slots * rank * 4 + (int64_t)slots * top_k * 12 >= (1 << 20))
            return DFLASH2_ERR_INVALID_ARG;
        prefetch_a = best_pa != 0;
    }
    wp.g = static_cast<const float *>(workspace);
    wp.split_stride = rows * rank;
    wp.k_splits = ksplits;
    dflash2_status s = set_walk_attributes(di);
    if (s != DFLASH2_OK) return s;
    if (lattice) {
        LatticeWs lw;
        size_t o_lat, o_stat, o_nxt, o_end;
        lattice_ws_layout(rows, top_k, (size_t)ksplits_ws(rows, hidden, rank, dtype) * rows * rank * 4,
                          &o_lat, &o_stat, &o_nxt, &o_end);
        uint8_t *wsb = static_cast<uint8_t *>(workspace);
        lw.lat = reinterpret_cast<float *>(wsb + o_lat);
        lw.stat = reinterpret_cast<float2 *>(wsb + o_stat);
        lw.nxt = reinterpret_cast<int32_t *>(wsb + o_nxt);
        const int km = top_k <= 8 ? 8 : (top_k <= 16 ? 16 : 32);
        const dim3 rgrid((unsigned)batch, (unsigned)parts);
#define DFLASH2_LAT_LAUNCH(T_, KM_) \
    launch_k(walk_rows_kernel<T_, KM_>, rgrid, kRowThreads, RL.total, st, wp, RL, spp, lw)
        if (dtype == DFLASH2_BF16) {
            if (km == 8) DFLASH2_LAT_LAUNCH(__nv_bfloat16, 8);
            else if (km == 16) DFLASH2_LAT_LAUNCH(__nv_bfloat16, 16);
            else DFLASH2_LAT_LAUNCH(__nv_bfloat16, 32);
        } else {
            if (km == 8) DFLASH2_LAT_LAUNCH(float, 8);
            else if (km == 16) DFLASH2_LAT_LAUNCH(float, 16);
            else DFLASH2_LAT_LAUNCH(float, 32);
        }
#undef DFLASH2_LAT_LAUNCH
        s = launch_status();
        if (s != DFLASH2_OK) return s;
        launch_k(walk_chase_kernel, (unsigned)batch, kChaseThreads,
                 (size_t)(slots * top_k + slots) * sizeof(int32_t), st, wp, lw);
        return launch_status();
    }
    if (chain) {
        const unsigned grid = (unsigned)batch;
        if (regb)
            launch_k(walk_chain_kernel<64, 1, true>, grid, kChainThreads, CL.total, st, wp, CL);
        else if (top_k <= 64)
            launch_k(walk_chain_kernel<64, 2, false>, grid, kChainThreads, CL.total, st, wp, CL);
        else if (rank <= 128)
            launch_k(walk_chain_kernel<128, 1, false>, grid, kChainThreads, CL.total, st, wp, CL);
        else
            launch_k(walk_chain_kernel<128, 2, false>, grid, kChainThreads, CL.total, st, wp, CL);
        return launch_status();
    }
    wp.bulk_ids = ((int64_t)slots * top_k) % 4 == 0 && aligned16(wp.cand) && aligned16(wp.cand_u);
    const unsigned grid = (unsigned)((batch + warps - 1) / warps);
    const size_t smem = L.total * warps;
    const int threads = 32 * warps;
#define DFLASH2_WALK_LAUNCH(T_, PA_, E_) \
    launch_k(walk_kernel<T_, PA_, E_>, grid, threads, smem, st, wp, warps, L)
    const int E = top_k <= 32 ? 1 : (top_k <= 64 ? 2 : 4);
    if (dtype == DFLASH2_BF16) {
        if (prefetch_a) {
            if (E == 1) DFLASH2_WALK_LAUNCH(__nv_bfloat16, true, 1);
            else if (E == 2) DFLASH2_WALK_LAUNCH(__nv_bfloat16, true, 2);
            else DFLASH2_WALK_LAUNCH(__nv_bfloat16, true, 4);
        } else {
            if (E == 1) DFLASH2_WALK_LAUNCH(__nv_bfloat16, false, 1);
            else if (E == 2) DFLASH2_WALK_LAUNCH(__nv_bfloat16, false, 2);
            else DFLASH2_WALK_LAUNCH(__nv_bfloat16, false, 4);
        }
    } else {
        if (prefetch_a) {
            if (E == 1) DFLASH2_WALK_LAUNCH(float, true, 1);
            else if (E == 2) DFLASH2_WALK_LAUNCH(float, true, 2);
            else DFLASH2_WALK_LAUNCH(float, true, 4);
        } else {
            if (E == 1) DFLASH2_WALK_LAUNCH(float, false, 1);
            else if (E == 2) DFLASH2_WALK_LAUNCH(float, false, 2);
            else DFLASH2_WALK_LAUNCH(float, false, 4);
        }
    }
#undef DFLASH2_WALK_LAUNCH
    return launch_status();
}

// The walk's parameters from the entry-point arguments (g and the split
// count are filled by run_walk).
WalkParams walk_params(const void *A, const void *B, int64_t table_rows, const int64_t *anchor_ids,
                       const int64_t *cand_ids, const float *cand_u, const float *temperatures,
                       const uint8_t *greedy, const float *uniforms, int32_t batch, int32_t slots,
                       int32_t rank, int32_t top_k, int64_t *tokens, float *q, float *path_scores,
                       int32_t *err_word) {
    WalkParams wp{};
    wp.A = A;
    wp.B = B;
    wp.table_rows = table_rows;
    wp.anchors = anchor_ids;
    wp.cand = cand_ids;
    wp.cand_u = cand_u;
    wp.temps = temperatures;
    wp.greedy = greedy;
    wp.uniforms = uniforms;
    wp.batch = batch;
    wp.slots = slots;
    wp.rank = rank;
    wp.k = top_k;
    wp.tokens = tokens;
    wp.q = q;
    wp.path_scores = path_scores;
    wp.err = err_word;
    return wp;
}

}  // namespace

extern "C" dflash2_status dflash2_selector_walk(
    const void *h, const void *proj, const void *A, const void *B, int64_t table_rows,
    const int64_t *anchor_ids, const int64_t *cand_ids, const float *cand_u,
    const float *temperatures, const uint8_t *greedy, const float *uniforms, int32_t batch,
    int32_t slots, int32_t hidden, int32_t rank, int32_t top_k, int32_t dtype, int64_t *tokens,
    float *q, float *path_scores, void *workspace, size_t ws_bytes, int32_t *err_word,
    void *stream) {
    dflash2_status s = check_walk_shape(batch, slots, hidden, rank, top_k, dtype);
    if (s != DFLASH2_OK) return s;
    if (table_rows <= 0) return DFLASH2_ERR_INVALID_ARG;
    if (batch == 0 || slots == 0) return DFLASH2_OK;
    if (!h || !proj || !A || !B || !anchor_ids || !cand_ids || !cand_u || !temperatures || !greedy ||
        !uniforms || !tokens || !q)
        return DFLASH2_ERR_INVALID_ARG;
    const size_t need =
        dflash2_selector_walk_workspace_size(batch, slots, hidden, rank, top_k, dtype);
    if (!workspace || ws_bytes < need) return DFLASH2_ERR_WORKSPACE;
    if (!aligned16(A) || !aligned16(B) || reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    s = run_projection(di, h, proj, (int64_t)batch * slots, hidden, rank, dtype,
                       static_cast<float *>(workspace), err_word, st);
    if (s != DFLASH2_OK) return s;
    WalkParams wp = walk_params(A, B, table_rows, anchor_ids, cand_ids, cand_u, temperatures, greedy,
                                uniforms, batch, slots, rank, top_k, tokens, q, path_scores,
                                err_word);
    wp.after_projection = true;
    return run_walk(di, wp, hidden, dtype, workspace, st);
}

extern "C" dflash2_status dflash2_selector_project(const void *h, const void *proj, int32_t batch,
                                                   int32_t slots, int32_t hidden, int32_t rank,
                                                   int32_t top_k, int32_t dtype, void *workspace,
                                                   size_t ws_bytes, int32_t *err_word,
                                                   void *stream) {
    dflash2_status s = check_walk_shape(batch, slots, hidden, rank, top_k, dtype);
    if (s != DFLASH2_OK) return s;
    if (batch == 0 || slots == 0) return DFLASH2_OK;
    if (!h || !proj) return DFLASH2_ERR_INVALID_ARG;
    const size_t need =
        dflash2_selector_walk_workspace_size(batch, slots, hidden, rank, top_k, dtype);
    if (!workspace || ws_bytes < need) return DFLASH2_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    return run_projection(di, h, proj, (int64_t)batch * slots, hidden, rank, dtype,
                          static_cast<float *>(workspace), err_word,
                          static_cast<cudaStream_t>(stream));
}

extern "C" dflash2_status dflash2_selector_walk_projected(
    const void *A, const void *B, int64_t table_rows, const int64_t *anchor_ids,
    const int64_t *cand_ids, const float *cand_u, const float *temperatures, const uint8_t *greedy,
    const float *uniforms, int32_t batch, int32_t slots, int32_t hidden, int32_t rank,
    int32_t top_k, int32_t dtype, int64_t *tokens, float *q, float *path_scores, void *workspace,
    size_t ws_bytes, int32_t *err_word, void *stream) {
    dflash2_status s = check_walk_shape(batch, slots, hidden, rank, top_k, dtype);
    if (s != DFLASH2_OK) return s;
    if (table_rows <= 0) return DFLASH2_ERR_INVALID_ARG;
    if (batch == 0 || slots == 0) return DFLASH2_OK;
    if (!A || !B || !anchor_ids || !cand_ids || !cand_u || !temperatures || !greedy || !uniforms ||
        !tokens || !q)
        return DFLASH2_ERR_INVALID_ARG;
    const size_t need =
        dflash2_selector_walk_workspace_size(batch, slots, hidden, rank, top_k, dtype);
    if (!workspace || ws_bytes < need) return DFLASH2_ERR_WORKSPACE;
    if (!aligned16(A) || !aligned16(B) || reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    return run_walk(di,
                    walk_params(A, B, table_rows, anchor_ids, cand_ids, cand_u, temperatures,
                                greedy, uniforms, batch, slots, rank, top_k, tokens, q,
                                path_scores, err_word),
                    hidden, dtype, workspace, static_cast<cudaStream_t>(stream));
}
