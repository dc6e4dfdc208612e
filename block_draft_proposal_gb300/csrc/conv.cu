// Block-causal grouped dynamic depthwise conv (sglang DFlash2 PR, _grouped_conv).
//
//   out[i, c] = sum_{t < taps, (i mod bs) >= t} (base[t, c] + delta[i, t, c / gs]) * x[i - t, c]
//
// HBM-bound: every x row is read once and every out row written once.  The
// fast path stages a tile of 16 token rows plus taps-1 halo rows (the rows
// that taps reach back to) of 32 16-byte vectors in shared memory with
// coalesced 16-byte loads, so the taps re-read shared memory instead of L2.
// One 16-byte vector is 8 bf16 (or 4 fp32) channels of one group, so the
// per-token coefficient delta is one scalar per (token, tap, vector).
#include "common.cuh"

namespace dflash2 {
namespace {

constexpr int kTileTokens = 16;
constexpr int kTileVecs = 32;
constexpr int kTokenLanes = 8;  // blockDim.y; blockDim.x = kTileVecs
constexpr int kMaxVecTaps = 64;

template <typename T> struct VecTraits;
template <> struct VecTraits<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void unpack(const uint4 &v, float (&f)[8]) {
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 t = __bfloat1622float2(p[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    __device__ static uint4 pack(const float (&f)[8]) {
        uint4 v;
        __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        return v;
    }
    __device__ static float scalar(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __nv_bfloat16 from(float v) { return __float2bfloat16_rn(v); }
};
template <> struct VecTraits<float> {
    static constexpr int N = 4;
    __device__ static void unpack(const uint4 &v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ static float scalar(float v) { return v; }
    __device__ static float from(float v) { return v; }
};

__device__ __forceinline__ int64_t in_block_pos(int64_t i, int bs, bool pow2) {
    return pow2 ? (i & (int64_t)(bs - 1)) : (i % bs);
}

// Tokens each thread covers (kTileTokens / kTokenLanes) and the largest tap
// count whose loads are issued together up front.
constexpr int kTokPerThread = kTileTokens / kTokenLanes;
constexpr int kRegTaps = 8;

// KT = 0: any tap count up to kMaxVecTaps, one tap's loads at a time.
// KT > 0: at most KT taps; the tile's base coefficients are loaded once into
// registers and every delta the thread needs is loaded before the first
// multiply-add, so a thread waits for memory about once instead of once per
// tap and token.  The arithmetic (order of taps, fp32 fma) is the same.
template <typename T, int KT>
__global__ void __launch_bounds__(kTileVecs *kTokenLanes)
    conv_vec_kernel(const T *__restrict__ x, const T *__restrict__ base,
                    const T *__restrict__ delta, int64_t dstride, T *__restrict__ out, int64_t n,
                    int hidden, int group_size, int taps, int bs, bool pow2) {
    grid_dep_wait();
    using V = VecTraits<T>;
    constexpr int VN = V::N;
    extern __shared__ uint4 tile[];  // [kTileTokens + taps - 1][kTileVecs]
    const int nvec = hidden / VN;
    // one-dimensional grid, token tiles fastest (at 8192 tokens x 7168 channels
    // 113 us against 128 us with vector tiles fastest, measured on GB300)
    const int n_ttiles = (int)((n + kTileTokens - 1) / kTileTokens);
    const int64_t i0 = (int64_t)(blockIdx.x % n_ttiles) * kTileTokens;
    const int v0 = (int)(blockIdx.x / n_ttiles) * kTileVecs;
    const int halo = taps - 1;
    const int rows = kTileTokens + halo;
    const int tid = threadIdx.y * kTileVecs + threadIdx.x;

    for (int idx = tid; idx < rows * kTileVecs; idx += kTileVecs * kTokenLanes) {
        const int r = idx / kTileVecs;
        const int vv = idx - r * kTileVecs;
        const int64_t gi = i0 - halo + r;
        const int gv = v0 + vv;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (gi >= 0 && gi < n && gv < nvec)
            val = __ldg(reinterpret_cast<const uint4 *>(x + gi * hidden) + gv);
        tile[idx] = val;
    }

    const int v = v0 + threadIdx.x;
    const bool active = v < nvec;
    const int groups = hidden / group_size;
    const int g = active ? (v * VN) / group_size : 0;
    const uint4 *base_v = reinterpret_cast<const uint4 *>(base) + v;

    if constexpr (KT > 0) {
        // loads first: the tile's base rows and every delta of this thread
        uint4 bq[KT];
        float d[kTokPerThread][KT];
#pragma unroll
        for (int t = 0; t < KT; ++t)
            bq[t] = active && t < taps ? __ldg(base_v + (int64_t)t * nvec) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < kTokPerThread; ++j) {
            const int64_t i = i0 + threadIdx.y + j * kTokenLanes;
            const int64_t pos = i < n ? in_block_pos(i, bs, pow2) : -1;
            const T *drow = delta + i * dstride + g;
#pragma unroll
            for (int t = 0; t < KT; ++t)
                d[j][t] = active && t <= pos && t < taps ? V::scalar(drow[(int64_t)t * groups]) : 0.0f;
        }
        __syncthreads();
        if (!active) return;
#pragma unroll
        for (int j = 0; j < kTokPerThread; ++j) {
            const int tt = threadIdx.y + j * kTokenLanes;
            const int64_t i = i0 + tt;
            if (i >= n) break;
            const int64_t pos = in_block_pos(i, bs, pow2);
            float acc[VN];
#pragma unroll
            for (int e = 0; e < VN; ++e) acc[e] = 0.0f;
#pragma unroll
            for (int t = 0; t < KT; ++t) {
                if (t < taps && t <= pos) {
                    float bf[VN], xf[VN];
                    V::unpack(bq[t], bf);
                    V::unpack(tile[(tt + halo - t) * kTileVecs + threadIdx.x], xf);
#pragma unroll
                    for (int e = 0; e < VN; ++e) acc[e] = fmaf(bf[e] + d[j][t], xf[e], acc[e]);
                }
            }
            reinterpret_cast<uint4 *>(out + i * hidden)[v] = V::pack(acc);
        }
    } else {
        __syncthreads();
        if (!active) return;
        for (int tt = threadIdx.y; tt < kTileTokens; tt += kTokenLanes) {
            const int64_t i = i0 + tt;
            if (i >= n) break;
            const int64_t pos = in_block_pos(i, bs, pow2);
            const int tmax = (int)min((int64_t)(taps - 1), pos);
            const T *drow = delta + i * dstride + g;
            float acc[VN];
#pragma unroll
            for (int e = 0; e < VN; ++e) acc[e] = 0.0f;
            for (int t = 0; t <= tmax; ++t) {
                const float dt = V::scalar(drow[(int64_t)t * groups]);
                float bf[VN], xf[VN];
                V::unpack(__ldg(base_v + (int64_t)t * nvec), bf);
                V::unpack(tile[(tt + halo - t) * kTileVecs + threadIdx.x], xf);
#pragma unroll
                for (int e = 0; e < VN; ++e) acc[e] = fmaf(bf[e] + dt, xf[e], acc[e]);
            }
            reinterpret_cast<uint4 *>(out + i * hidden)[v] = V::pack(acc);
        }
    }
}

// General layout: one thread per output element.
template <typename T>
__global__ void conv_scalar_kernel(const T *__restrict__ x, const T *__restrict__ base,
                                   const T *__restrict__ delta, int64_t dstride,
                                   T *__restrict__ out, int64_t n, int hidden, int group_size,
                                   int taps, int bs, bool pow2) {
    grid_dep_wait();
    using V = VecTraits<T>;
    const int groups = hidden / group_size;
    const int64_t total = n * hidden;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = idx / hidden;
        const int c = (int)(idx - i * hidden);
        const int64_t pos = in_block_pos(i, bs, pow2);
        const int tmax = (int)min((int64_t)(taps - 1), pos);
        float acc = 0.0f;
        for (int t = 0; t <= tmax; ++t) {
            const float coef = V::scalar(base[(int64_t)t * hidden + c]) +
                               V::scalar(delta[i * dstride + (int64_t)t * groups + c / group_size]);
            acc = fmaf(coef, V::scalar(x[(i - t) * hidden + c]), acc);
        }
        out[idx] = V::from(acc);
    }
}

template <typename T>
dflash2_status run_conv(const DeviceInfo &di, const void *x, const void *base, const void *delta,
                        int64_t dstride, void *out, int64_t n, int hidden, int gs, int taps, int bs,
                        cudaStream_t st) {
    constexpr int VN = VecTraits<T>::N;
    const int taps_eff = taps < bs ? taps : bs;  // taps >= bs never pass the position mask
    const bool pow2 = (bs & (bs - 1)) == 0;
    const bool vec_ok = (gs % VN) == 0 && aligned16(x) && aligned16(base) && aligned16(out) &&
                        taps_eff <= kMaxVecTaps;
    if (vec_ok) {
        const int nvec = hidden / VN;
        const int64_t ctas = (int64_t)((nvec + kTileVecs - 1) / kTileVecs) *
                             ((n + kTileTokens - 1) / kTileTokens);
        if (ctas > INT32_MAX) return DFLASH2_ERR_INVALID_ARG;
        const dim3 grid((unsigned)ctas);
        dim3 block(kTileVecs, kTokenLanes);
        const size_t smem = (size_t)(kTileTokens + taps_eff - 1) * kTileVecs * sizeof(uint4);
        const T *xp = static_cast<const T *>(x), *bp = static_cast<const T *>(base),
                *dp = static_cast<const T *>(delta);
        T *op = static_cast<T *>(out);
        if (taps_eff <= 4)
            launch_k(conv_vec_kernel<T, 4>, grid, block, smem, st, xp, bp, dp, dstride, op, n,
                     hidden, gs, taps_eff, bs, pow2);
        else if (taps_eff <= kRegTaps)
            launch_k(conv_vec_kernel<T, kRegTaps>, grid, block, smem, st, xp, bp, dp, dstride, op,
                     n, hidden, gs, taps_eff, bs, pow2);
        else
            launch_k(conv_vec_kernel<T, 0>, grid, block, smem, st, xp, bp, dp, dstride, op, n,
                     hidden, gs, taps_eff, bs, pow2);
    } else {
        const int64_t total = n * hidden;
        int64_t blocks = (total + 255) / 256;
        const int64_t cap = (int64_t)di.sm_count * 16;
        if (blocks > cap) blocks = cap;
        launch_k(conv_scalar_kernel<T>, (unsigned)blocks, 256, 0, st, static_cast<const T *>(x),
            static_cast<const T *>(base), static_cast<const T *>(delta),
            dstride, static_cast<T *>(out), n, hidden, gs, taps_eff, bs, pow2);
    }
    return launch_status();
}

}  // namespace
}  // namespace dflash2

extern "C" dflash2_status dflash2_grouped_conv(const void *x, const void *base, const void *delta,
                                               int64_t delta_row_stride, void *out,
                                               int64_t n_tokens, int32_t hidden,
                                               int32_t group_size, int32_t taps,
                                               int32_t block_size, int32_t dtype, void *stream) {
    using namespace dflash2;
    if (dtype != DFLASH2_F32 && dtype != DFLASH2_BF16) return DFLASH2_ERR_UNSUPPORTED_DTYPE;
    if (n_tokens < 0 || hidden <= 0 || group_size <= 0 || hidden % group_size != 0 || taps <= 0 ||
        block_size <= 0)
        return DFLASH2_ERR_INVALID_ARG;
    const int64_t groups = hidden / group_size;
    if (delta_row_stride < (int64_t)taps * groups) return DFLASH2_ERR_INVALID_ARG;
    if (n_tokens == 0) return DFLASH2_OK;
    if (!x || !base || !delta || !out) return DFLASH2_ERR_INVALID_ARG;
    const uintptr_t esz = dtype == DFLASH2_BF16 ? 2 : 4;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(base) |
         reinterpret_cast<uintptr_t>(delta) | reinterpret_cast<uintptr_t>(out)) %
            esz !=
        0)
        return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    dflash2_status s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == DFLASH2_BF16)
        return run_conv<__nv_bfloat16>(di, x, base, delta, delta_row_stride, out, n_tokens, hidden,
                                       group_size, taps, block_size, st);
    return run_conv<float>(di, x, base, delta, delta_row_stride, out, n_tokens, hidden, group_size,
                           taps, block_size, st);
}
