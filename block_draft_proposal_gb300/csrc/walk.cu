// Selector lattice + walk (sglang DFlash2 PR: the PR body's edge formula,
// CandidateSelector.build_lattice / sample_path, _selector_walk_kernel,
// stage_sampling_params).
//
//   g[m, :] = h[m, :] . proj^T                           (tensor cores for bf16)
//   e[k]    = sum_j A[p, j] * g[b*S + s, j] * B[c_k, j] + cand_u[b, s, k]
//   greedy: index = smallest argmax e, q = one-hot;  sampled: q = softmax(e / T),
//   index = min(#{k : uniform >= cumsum(q)[k]}, K - 1);  token = c_index.
//
// One CTA per request walks its slots in order.  The lattice is never
// materialised: only the K edges leaving the chosen predecessor are formed.
// The B rows of a slot's K candidates do not depend on the path, so the rows
// of slot s+1 are fetched (cp.async) while slot s is being walked; only the
// predecessor's A row sits on the serial chain.  The K edges are reduced by
// one warp with shuffles (argmax, max, sum, prefix sum, count).
#include "kernels.h"

namespace dflash2 {
namespace {

constexpr int kWalkThreads = 128;
constexpr int kWalkWarps = kWalkThreads / 32;
constexpr int kMaxK = 128;
constexpr int kMaxRank = 256;
constexpr int kPerLane = kMaxK / 32;
constexpr int kWalkMaxSmem = 200 * 1024;  // two buffers of K candidate B rows

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
    int32_t slots, rank, k;
    int64_t *tokens;
    float *q;
    float *path_scores;
    int32_t *err;
};

template <typename T> __device__ __forceinline__ float2 ld2(const T *p);
template <> __device__ __forceinline__ float2 ld2<float>(const float *p) {
    return *reinterpret_cast<const float2 *>(p);
}
template <> __device__ __forceinline__ float2 ld2<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}
template <typename T> __device__ __forceinline__ float ld1(const T *p);
template <> __device__ __forceinline__ float ld1<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float ld1<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}

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

// Issue the copies of slot s's K candidate B rows into buffer `dst`.
template <typename T>
__device__ __forceinline__ void fetch_b_rows(const WalkParams &p, int64_t bs_row, T *dst) {
    const int chunks = p.rank * (int)sizeof(T) / 16;  // 16-byte pieces per row
    const T *B = static_cast<const T *>(p.B);
    for (int idx = threadIdx.x; idx < p.k * chunks; idx += kWalkThreads) {
        const int kk = idx / chunks;
        const int ch = idx - kk * chunks;
        const int64_t c = p.cand[bs_row * p.k + kk];
        const bool ok = c >= 0 && c < p.table_rows;
        const T *src = ok ? B + c * p.rank : B;
        cp_async16(reinterpret_cast<uint8_t *>(dst + (int64_t)kk * p.rank) + ch * 16,
                   reinterpret_cast<const uint8_t *>(src) + ch * 16, ok);
        if (!ok && ch == 0 && p.err) atomicOr(p.err, DFLASH2_DEVERR_ID_RANGE);
    }
    cp_async_commit();
}

template <typename T>
__global__ void __launch_bounds__(kWalkThreads) walk_kernel(const WalkParams p) {
    extern __shared__ __align__(16) uint8_t dyn[];
    T *bbuf[2];
    bbuf[0] = reinterpret_cast<T *>(dyn);
    bbuf[1] = bbuf[0] + (size_t)p.k * p.rank;
    __shared__ float w[kMaxRank];
    __shared__ float e[kMaxK];
    __shared__ int chosen;

    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.slots, K = p.k, R = p.rank;
    const bool is_greedy = p.greedy[b] != 0;
    float temp = p.temps[b];
    if (!(temp >= 1e-5f)) temp = 1e-5f;
    const T *A = static_cast<const T *>(p.A);

    if (S > 0) fetch_b_rows<T>(p, (int64_t)b * S, bbuf[0]);
    int prev = 0;
    for (int s = 0; s < S; ++s) {
        const int64_t bs_row = (int64_t)b * S + s;
        if (s + 1 < S) {
            fetch_b_rows<T>(p, bs_row + 1, bbuf[(s + 1) & 1]);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        // predecessor: the anchor at slot 0, else the previous slot's choice
        const int64_t pid = s == 0 ? p.anchors[b] : p.cand[(bs_row - 1) * K + prev];
        const bool p_ok = pid >= 0 && pid < p.table_rows;
        if (!p_ok && threadIdx.x == 0 && p.err) atomicOr(p.err, DFLASH2_DEVERR_ID_RANGE);
        for (int j = threadIdx.x; j < R; j += kWalkThreads) {
            float gj = 0.0f;
            for (int ks = 0; ks < p.k_splits; ++ks) gj += p.g[ks * p.split_stride + bs_row * R + j];
            const float a = p_ok ? ld1<T>(A + pid * R + j) : 0.0f;
            w[j] = a * gj;
        }
        __syncthreads();
        // edges: one warp per candidate, lanes over the rank in pairs
        const T *brow = bbuf[s & 1];
        for (int kk = warp; kk < K; kk += kWalkWarps) {
            const T *bk = brow + (int64_t)kk * R;
            float acc = 0.0f;
            for (int j = 2 * lane; j < R; j += 64) {
                const float2 bv = ld2<T>(bk + j);
                acc = fmaf(w[j], bv.x, acc);
                acc = fmaf(w[j + 1], bv.y, acc);
            }
            acc = warp_sum(acc);
            if (lane == 0) e[kk] = acc + p.cand_u[bs_row * K + kk];
        }
        __syncthreads();
        if (warp == 0) {
            const int E = (K + 31) >> 5;  // consecutive edges per lane
            float ev[kPerLane];
            bool valid[kPerLane];
#pragma unroll
            for (int i = 0; i < kPerLane; ++i) {
                const int kk = lane * E + i;
                valid[i] = i < E && kk < K;
                ev[i] = valid[i] ? e[kk] : -INFINITY;
            }
            float qv[kPerLane];
            int index;
            if (is_greedy) {
                float best = -INFINITY;
                int bi = INT32_MAX;
#pragma unroll
                for (int i = 0; i < kPerLane; ++i)
                    if (valid[i] && (bi == INT32_MAX || ev[i] > best)) {
                        best = ev[i];
                        bi = lane * E + i;
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
                index = bi;
#pragma unroll
                for (int i = 0; i < kPerLane; ++i) qv[i] = (lane * E + i) == index ? 1.0f : 0.0f;
            } else {
                float sc[kPerLane];
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < kPerLane; ++i) {
                    sc[i] = valid[i] ? ev[i] / temp : -INFINITY;
                    mx = fmaxf(mx, sc[i]);
                }
                mx = warp_max(mx);
                float local = 0.0f;
#pragma unroll
                for (int i = 0; i < kPerLane; ++i) {
                    qv[i] = valid[i] ? expf(sc[i] - mx) : 0.0f;
                    local += qv[i];
                }
                const float total = warp_sum(local);
                float run = 0.0f, cdf[kPerLane];
#pragma unroll
                for (int i = 0; i < kPerLane; ++i) {
                    qv[i] = qv[i] / total;
                    run += qv[i];
                    cdf[i] = run;
                }
                float incl = run;  // inclusive scan of the lane totals
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                    if (lane >= o) incl += y;
                }
                float excl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
                if (lane == 0) excl = 0.0f;
                const float uni = p.uniforms[bs_row];
                int count = 0;
#pragma unroll
                for (int i = 0; i < kPerLane; ++i)
                    if (valid[i] && uni >= excl + cdf[i]) ++count;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) count += __shfl_xor_sync(0xFFFFFFFFu, count, o);
                index = count < K - 1 ? count : K - 1;
            }
#pragma unroll
            for (int i = 0; i < kPerLane; ++i) {
                const int kk = lane * E + i;
                if (valid[i]) {
                    p.q[bs_row * K + kk] = qv[i];
                    if (p.path_scores) p.path_scores[bs_row * K + kk] = ev[i];
                }
            }
            if (lane == 0) {
                p.tokens[bs_row] = p.cand[bs_row * K + index];
                chosen = index;
            }
        }
        __syncthreads();
        prev = chosen;
    }
}

// fp32 projection on CUDA cores: one CTA per row, one warp per output column.
__global__ void __launch_bounds__(128)
    project_f32_kernel(const float *__restrict__ h, const float *__restrict__ proj, int hidden,
                       int rank, float *g) {
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

// Split of the hidden dimension for the tensor-core projection, so that
// small batches still spread over the SMs.  Depends on the shape only, so
// the workspace size does not depend on the device.
inline void proj_tiling(int64_t rows, int hidden, int *bn, int *k_splits) {
    *bn = rows >= 4096 ? 64 : 32;
    const int64_t tiles = (rows + *bn - 1) / *bn;
    const int num_kb = (hidden + kGemmTileK - 1) / kGemmTileK;
    int64_t ks = (148 + tiles - 1) / tiles;
    if (ks > num_kb) ks = num_kb;
    if (ks > 16) ks = 16;
    if (ks < 1) ks = 1;
    // the GEMM launcher trims k_splits so that every split has work; size
    // the workspace for the requested count
    *k_splits = (int)ks;
}

bool g_walk_attr[64];

}  // namespace
}  // namespace dflash2

using namespace dflash2;

extern "C" size_t dflash2_selector_walk_workspace_size(int32_t batch, int32_t slots, int32_t hidden,
                                                       int32_t rank, int32_t dtype) {
    if (batch <= 0 || slots <= 0 || hidden <= 0 || rank <= 0) return 0;
    const int64_t rows = (int64_t)batch * slots;
    int bn = 32, ks = 1;
    if (dtype == DFLASH2_BF16) proj_tiling(rows, hidden, &bn, &ks);
    return (size_t)ks * rows * rank * sizeof(float);
}

extern "C" dflash2_status dflash2_selector_walk(
    const void *h, const void *proj, const void *A, const void *B, int64_t table_rows,
    const int64_t *anchor_ids, const int64_t *cand_ids, const float *cand_u,
    const float *temperatures, const uint8_t *greedy, const float *uniforms, int32_t batch,
    int32_t slots, int32_t hidden, int32_t rank, int32_t top_k, int32_t dtype, int64_t *tokens,
    float *q, float *path_scores, void *workspace, size_t ws_bytes, int32_t *err_word,
    void *stream) {
    if (dtype != DFLASH2_F32 && dtype != DFLASH2_BF16) return DFLASH2_ERR_UNSUPPORTED_DTYPE;
    const int rank_mult = dtype == DFLASH2_BF16 ? 8 : 4;
    if (batch < 0 || slots < 0 || hidden <= 0 || rank <= 0 || rank > kMaxRank ||
        rank % rank_mult != 0 || top_k <= 0 || top_k > kMaxK || table_rows <= 0)
        return DFLASH2_ERR_INVALID_ARG;
    const size_t esz = dtype == DFLASH2_BF16 ? 2 : 4;
    const size_t smem = 2 * (size_t)top_k * rank * esz;
    if (smem > (size_t)kWalkMaxSmem) return DFLASH2_ERR_INVALID_ARG;
    if (batch == 0 || slots == 0) return DFLASH2_OK;
    if (!h || !proj || !A || !B || !anchor_ids || !cand_ids || !cand_u || !temperatures || !greedy ||
        !uniforms || !tokens || !q)
        return DFLASH2_ERR_INVALID_ARG;
    const size_t need = dflash2_selector_walk_workspace_size(batch, slots, hidden, rank, dtype);
    if (!workspace || ws_bytes < need) return DFLASH2_ERR_WORKSPACE;
    if (!aligned16(A) || !aligned16(B) || reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    dflash2_status s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t rows = (int64_t)batch * slots;
    float *g = static_cast<float *>(workspace);

    WalkParams wp{};
    wp.g = g;
    wp.split_stride = rows * rank;
    if (dtype == DFLASH2_BF16) {
        if (hidden % 8 != 0 || !aligned16(h) || !aligned16(proj)) return DFLASH2_ERR_MISALIGNED;
        int bn, ks;
        proj_tiling(rows, hidden, &bn, &ks);
        GemmParams p{};
        p.rows_w = rank;
        p.rows_h = (int32_t)rows;
        p.hidden = hidden;
        p.mode = kGemmStore;
        p.bn = bn;
        p.k_splits = ks;
        p.out = g;
        p.ldo = rank;
        p.split_stride = rows * rank;
        p.err = err_word;
        // the launcher may trim k_splits; recompute the count it will use
        const int num_kb = (hidden + kGemmTileK - 1) / kGemmTileK;
        const int per = (num_kb + ks - 1) / ks;
        wp.k_splits = (num_kb + per - 1) / per;
        s = launch_gemm_tc(di, proj, h, p, st);
        if (s != DFLASH2_OK) return s;
    } else {
        if ((reinterpret_cast<uintptr_t>(h) | reinterpret_cast<uintptr_t>(proj)) % 4 != 0)
            return DFLASH2_ERR_MISALIGNED;
        wp.k_splits = 1;
        project_f32_kernel<<<(unsigned)rows, 128, 0, st>>>(static_cast<const float *>(h),
                                                           static_cast<const float *>(proj), hidden,
                                                           rank, g);
        s = launch_status();
        if (s != DFLASH2_OK) return s;
    }
    wp.A = A;
    wp.B = B;
    wp.table_rows = table_rows;
    wp.anchors = anchor_ids;
    wp.cand = cand_ids;
    wp.cand_u = cand_u;
    wp.temps = temperatures;
    wp.greedy = greedy;
    wp.uniforms = uniforms;
    wp.slots = slots;
    wp.rank = rank;
    wp.k = top_k;
    wp.tokens = tokens;
    wp.q = q;
    wp.path_scores = path_scores;
    wp.err = err_word;
    if (di.device >= 0 && di.device < 64 && !g_walk_attr[di.device]) {
        if (cudaFuncSetAttribute(walk_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kWalkMaxSmem) != cudaSuccess ||
            cudaFuncSetAttribute(walk_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kWalkMaxSmem) != cudaSuccess) {
            cudaGetLastError();
            return DFLASH2_ERR_CUDA;
        }
        g_walk_attr[di.device] = true;
    }
    if (dtype == DFLASH2_BF16)
        walk_kernel<__nv_bfloat16><<<(unsigned)batch, kWalkThreads, smem, st>>>(wp);
    else
        walk_kernel<float><<<(unsigned)batch, kWalkThreads, smem, st>>>(wp);
    return launch_status();
}
