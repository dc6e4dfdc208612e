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
#include <atomic>

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
    __device__ static void unpack2(const uint4 &v, float2 (&f)[4]) {
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = __bfloat1622float2(p[i]);
    }
    __device__ static uint4 pack2(const float2 (&f)[4]) {
        uint4 v;
        __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = __float22bfloat162_rn(f[i]);
        return v;
    }
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
    __device__ static void unpack2(const uint4 &v, float2 (&f)[2]) {
        f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
        f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
    }
    __device__ static uint4 pack2(const float2 (&f)[2]) {
        return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x),
                          __float_as_uint(f[1].y));
    }
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

// ---------------------------------------------------------------------------
// Pipelined path.  Work items of kPipeTokens tokens x kPipeVecs vectors; a
// persistent grid of CTAs takes items in turn, and each CTA keeps
// kPipeStages items in flight: cp.async 16-byte copies stage an item's x rows
// and its delta slice [token][tap][groups of the item] in shared memory while
// the CTA computes an earlier item, so an SM's loads never wait behind its
// arithmetic or stores.  When the block size divides the tile, every tile
// starts a block and no tap reaches before it: no halo rows are loaded;
// otherwise taps - 1 halo rows come first.  The taps are summed in the same
// order as conv_vec_kernel (t = 0, 1, ...; fp32 fma), so both give the same
// bits.
// ---------------------------------------------------------------------------
constexpr int kPipeVecs = 64;
constexpr int kPipeTokens = 16;
constexpr int kPipeThreads = 256;
constexpr int kPipeStages = 4;
constexpr int kPipeTokPerThread = kPipeTokens * kPipeVecs / kPipeThreads;
constexpr int kPipeMaxTaps = 8;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
    const uint32_t n = valid ? 16u : 0u;  // 0 source bytes: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem),
                 "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Shared-memory bytes of one pipeline stage.
__host__ __device__ inline int pipe_stage_bytes(int halo, int taps, int gpv, int esz) {
    return (kPipeTokens + halo) * kPipeVecs * 16 + kPipeTokens * taps * gpv * esz;
}

// Largest number of 16-byte delta chunks per (token, tap) and item: 64 / gs
// with gs >= 8 for bf16 and >= 4 for fp32.
template <typename T> __host__ __device__ constexpr int pipe_max_dch() { return sizeof(T) == 2 ? 8 : 16; }

template <typename T, int KT>
__global__ void __launch_bounds__(kPipeThreads, 2)
    conv_pipe_kernel(const T *__restrict__ x, const T *__restrict__ base,
                     const T *__restrict__ delta, int64_t dstride, T *__restrict__ out, int64_t n,
                     int hidden, int group_size, int taps, int bs, bool pow2, int halo,
                     int n_ttiles, int n_strips) {
    grid_dep_wait();
    using V = VecTraits<T>;
    constexpr int VN = V::N;
    constexpr int VP = VN / 2;                 // float2 pairs of a vector
    constexpr int EPC = 16 / (int)sizeof(T);   // elements of a 16-byte chunk
    constexpr int kDC = kPipeTokens * KT * pipe_max_dch<T>() / kPipeThreads;  // delta chunks a thread copies, at most
    extern __shared__ __align__(16) uint8_t pipe_sm[];
    const int nvec = hidden / VN;
    const int groups = hidden / group_size;
    const int gpv = kPipeVecs * VN / group_size;  // groups of one item
    const int dch = gpv / EPC;                    // delta chunks per (token, tap)
    const int per_tok = taps * dch;
    const int xrows = kPipeTokens + halo;
    const int xbytes = xrows * kPipeVecs * 16;
    const int stage_bytes = pipe_stage_bytes(halo, taps, gpv, (int)sizeof(T));
    const int tid = threadIdx.x;

    // this thread's copies, the same for every item: x rows (tid >> 6) + 4 m
    // of vector tid & 63, and delta chunks tid + 256 m as (token, offset)
    int d_tt[kDC], d_q[kDC], d_off[kDC];
#pragma unroll
    for (int m = 0; m < kDC; ++m) {
        const int c = tid + kPipeThreads * m;
        const int tt = c / per_tok;
        const int rem = c - tt * per_tok;
        const int t = rem / dch;
        d_tt[m] = c < kPipeTokens * per_tok ? tt : kPipeTokens;  // kPipeTokens: no chunk
        d_q[m] = (rem - t * dch) * EPC;                          // group offset within the item
        d_off[m] = t * groups + d_q[m];
    }
    const int xv = tid & (kPipeVecs - 1);
    const int xr0 = tid / kPipeVecs;

    // Work split: CTA b keeps the 64-vector strip b % n_strips and takes
    // its token tiles b / n_strips, + tstep, ... (the grid is a multiple of
    // n_strips), so the strip's base coefficients are read once per CTA.
    const int strip = (int)blockIdx.x % n_strips;
    const int tstep = (int)gridDim.x / n_strips;
    const int tile0 = (int)blockIdx.x / n_strips;
    const int g0 = strip * gpv;

    auto issue = [&](int tile, int stage) {
        uint8_t *st = pipe_sm + (size_t)stage * stage_bytes;
        const int64_t i0 = (int64_t)tile * kPipeTokens;
        const int gv = strip * kPipeVecs + xv;
        for (int r = xr0; r < xrows; r += kPipeThreads / kPipeVecs) {
            const int64_t gi = i0 - halo + r;
            const bool ok = gi >= 0 && gi < n && gv < nvec;
            cp_async16(st + ((size_t)r * kPipeVecs + xv) * 16,
                       ok ? x + gi * hidden + (int64_t)gv * VN : x, ok);
        }
        const T *drow = delta + i0 * dstride + g0;
#pragma unroll
        for (int m = 0; m < kDC; ++m) {
            if (d_tt[m] < kPipeTokens) {
                const int c = tid + kPipeThreads * m;
                const int gg = g0 + d_q[m];
                const bool ok = i0 + d_tt[m] < n && gg < groups;
                cp_async16(st + xbytes + (size_t)c * 16,
                           ok ? drow + (int64_t)d_tt[m] * dstride + d_off[m] : delta, ok);
            }
        }
    };

    const int vv = tid % kPipeVecs;
    const int ty = tid / kPipeVecs;
    const int tt0 = ty * kPipeTokPerThread;
    const int gl = (vv * VN) / group_size;  // the vector's group within an item
    const int v = strip * kPipeVecs + vv;
    const bool active = v < nvec;
    int fetch = tile0;
#pragma unroll
    for (int st = 0; st < kPipeStages - 1; ++st) {
        if (fetch < n_ttiles) issue(fetch, st);
        cp_async_commit();
        fetch += tstep;
    }
    // the taps' base coefficients of this thread's vector: up to four taps
    // unpacked once for every item; more taps read at each use (L1 hits)
    constexpr bool kFlat = KT <= 4;
    constexpr int KF = kFlat ? KT : 1;
    const uint4 *base_v = reinterpret_cast<const uint4 *>(base) + v;
    float2 bf[KF][VP];
    if constexpr (kFlat) {
#pragma unroll
        for (int t = 0; t < KT; ++t)
            V::unpack2(active && t < taps ? __ldg(base_v + (int64_t)t * nvec)
                                          : make_uint4(0, 0, 0, 0),
                       bf[t]);
    }
    for (int k = 0, tile = tile0; tile < n_ttiles; ++k, tile += tstep) {
        cp_async_wait<kPipeStages - 2>();
        __syncthreads();  // item k is staged; every thread is done with item k - 1
        if (fetch < n_ttiles) issue(fetch, (k + kPipeStages - 1) % kPipeStages);
        cp_async_commit();
        fetch += tstep;

        if (!active) continue;
        const uint8_t *st = pipe_sm + (size_t)(k % kPipeStages) * stage_bytes;
        const uint4 *xs = reinterpret_cast<const uint4 *>(st) + vv;
        const T *ds = reinterpret_cast<const T *>(st + xbytes) + gl;
        const int64_t i0 = (int64_t)tile * kPipeTokens;
        // block position of the thread's first token
        int pos = pow2 ? (int)((i0 + tt0) & (int64_t)(bs - 1)) : (int)((i0 + tt0) % bs);
        // a window of the last KT x rows of this vector: xw[t] is row tt - t
        // of the token tt in hand (rows before the tile's staged range are
        // never used: the block-position mask excludes them).  Up to four taps
        // the window is unpacked once per row; more taps read x from shared
        // memory at each use.
        float2 xw[KF][VP];
        if constexpr (kFlat) {
#pragma unroll
            for (int t = 1; t < KT; ++t) {
                const int r = tt0 - t + halo;
                V::unpack2((t < taps && r >= 0) ? xs[r * kPipeVecs] : make_uint4(0, 0, 0, 0),
                           xw[t]);
            }
        }
        T *orow = out + (i0 + tt0) * hidden + (int64_t)v * VN;
        // Every tap of every token inside its block (full), or the thread's
        // first token starting a block that its tokens do not leave (start):
        // then the masks are known per (token, tap) without the position and
        // the tokens' sums interleave freely.  The same for a whole warp: its
        // 32 threads share tt0.  The arithmetic is the general loop's.
        const bool full = pos >= KT - 1 && pos + kPipeTokPerThread <= bs;
        const bool start = pos == 0 && kPipeTokPerThread <= bs;
        if (kFlat && taps == KT && (full || start) && i0 + tt0 + kPipeTokPerThread <= n) {
#pragma unroll
            for (int j = 0; j < kPipeTokPerThread; ++j) {
                const int tt = tt0 + j;
                if (j > 0) {
#pragma unroll
                    for (int t = KF - 1; t > 0; --t)
#pragma unroll
                        for (int e = 0; e < VP; ++e) xw[t][e] = xw[t - 1][e];
                }
                V::unpack2(xs[(tt + halo) * kPipeVecs], xw[0]);
                float2 acc[VP];
#pragma unroll
                for (int e = 0; e < VP; ++e) acc[e] = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int t = 0; t < KF; ++t) {
                    if (t <= j || full) {
                        const float dt = V::scalar(ds[(tt * KT + t) * gpv]);
                        const float2 d2 = make_float2(dt, dt);
#pragma unroll
                        for (int e = 0; e < VP; ++e)
                            acc[e] = __ffma2_rn(__fadd2_rn(bf[t][e], d2), xw[t][e], acc[e]);
                    }
                }
                *reinterpret_cast<uint4 *>(orow) = V::pack2(acc);
                orow += hidden;
            }
            continue;
        }
#pragma unroll
        for (int j = 0; j < kPipeTokPerThread; ++j) {
            const int tt = tt0 + j;
            if (i0 + tt >= n) break;
            if (j > 0) {
                if (++pos == bs) pos = 0;
                if constexpr (kFlat) {
#pragma unroll
                    for (int t = KT - 1; t > 0; --t)
#pragma unroll
                        for (int e = 0; e < VP; ++e) xw[t][e] = xw[t - 1][e];
                }
            }
            if constexpr (kFlat) V::unpack2(xs[(tt + halo) * kPipeVecs], xw[0]);
            float2 acc[VP];
#pragma unroll
            for (int e = 0; e < VP; ++e) acc[e] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int t = 0; t < KT; ++t) {
                if (t < taps && t <= pos) {
                    const float dt = V::scalar(ds[(tt * taps + t) * gpv]);
                    const float2 d2 = make_float2(dt, dt);
                    float2 bt[VP], xt[VP];
                    if constexpr (kFlat) {
#pragma unroll
                        for (int e = 0; e < VP; ++e) {
                            bt[e] = bf[t][e];
                            xt[e] = xw[t][e];
                        }
                    } else {
                        V::unpack2(__ldg(base_v + (int64_t)t * nvec), bt);
                        V::unpack2(xs[(tt + halo - t) * kPipeVecs], xt);
                    }
                    // acc = (base + delta) * x + acc, each lane rounded as fmaf(bf + dt, x, acc)
#pragma unroll
                    for (int e = 0; e < VP; ++e) acc[e] = __ffma2_rn(__fadd2_rn(bt[e], d2), xt[e], acc[e]);
                }
            }
            *reinterpret_cast<uint4 *>(orow) = V::pack2(acc);
            orow += hidden;
        }
    }
    cp_async_wait<0>();
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

std::atomic<bool> g_pipe_attr[2][64];  // per element type and device; idempotent calls

// Opt the pipelined kernels into more than 48 KB of dynamic shared memory.
template <typename T> dflash2_status set_pipe_attrs(const DeviceInfo &di) {
    const int ti = sizeof(T) == 2 ? 0 : 1;
    if (di.device < 0 || di.device >= 64) return DFLASH2_ERR_CUDA;
    if (g_pipe_attr[ti][di.device]) return DFLASH2_OK;
    const int bytes = 227 * 1024;
    if (cudaFuncSetAttribute(conv_pipe_kernel<T, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess ||
        cudaFuncSetAttribute(conv_pipe_kernel<T, kPipeMaxTaps>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
        cudaGetLastError();
        return DFLASH2_ERR_CUDA;
    }
    g_pipe_attr[ti][di.device] = true;
    return DFLASH2_OK;
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
    // the pipelined path: whole 16-byte chunks of delta per (token, tap) and
    // item, 16-byte aligned rows, and at most kPipeMaxTaps live taps
    const int groups = hidden / gs;
    const int gpv_num = kPipeVecs * VN;
    const int esz = (int)sizeof(T);
    const bool pipe_ok = vec_ok && taps_eff <= kPipeMaxTaps && gpv_num % gs == 0 &&
                         ((gpv_num / gs) * esz) % 16 == 0 && (groups * esz) % 16 == 0 &&
                         (dstride * esz) % 16 == 0 && aligned16(delta);
    if (pipe_ok) {
        const int gpv = gpv_num / gs;
        const int halo = (kPipeTokens % bs == 0) ? 0 : taps_eff - 1;
        const int nvec = hidden / VN;
        const int64_t n_ttiles = (n + kPipeTokens - 1) / kPipeTokens;
        const int n_strips = (nvec + kPipeVecs - 1) / kPipeVecs;
        const int64_t n_items = n_ttiles * n_strips;
        if (n_items > INT32_MAX / 2) return DFLASH2_ERR_INVALID_ARG;
        const size_t smem = (size_t)kPipeStages * pipe_stage_bytes(halo, taps_eff, gpv, esz);
        if (smem > 227 * 1024) return DFLASH2_ERR_INVALID_ARG;  // taps <= 8 keeps it below 160 KB
        int per_sm = (int)((227 * 1024) / (smem + 1024));
        if (per_sm > 2) per_sm = 2;
        // a whole number of CTAs per strip (each CTA keeps one strip), at most
        // the CTAs resident at once and at most one per item
        int64_t per_strip = (int64_t)di.sm_count * per_sm / n_strips;
        if (per_strip < 1) per_strip = 1;
        if (per_strip > n_ttiles) per_strip = n_ttiles;
        const int64_t grid = per_strip * n_strips;
        const T *xp = static_cast<const T *>(x), *bp = static_cast<const T *>(base),
                *dp = static_cast<const T *>(delta);
        T *op = static_cast<T *>(out);
        dflash2_status s = set_pipe_attrs<T>(di);
        if (s != DFLASH2_OK) return s;
        if (taps_eff <= 4)
            launch_k(conv_pipe_kernel<T, 4>, (unsigned)grid, kPipeThreads, smem, st, xp, bp, dp,
                     dstride, op, n, hidden, gs, taps_eff, bs, pow2, halo, (int)n_ttiles, n_strips);
        else
            launch_k(conv_pipe_kernel<T, kPipeMaxTaps>, (unsigned)grid, kPipeThreads, smem, st, xp,
                     bp, dp, dstride, op, n, hidden, gs, taps_eff, bs, pow2, halo, (int)n_ttiles,
                     n_strips);
        return launch_status();
    }
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
