// Per-row E4M3 quantization of activations (W8A8 with dynamic per-token
// scales), the first step of the FP8-head unary path:
//
//   amax = max_j |x[m, j]|,  inv = 448 / amax,  d[m] = amax / 448   (fp32)
//   q[m, j] = E4M3(x[m, j] * inv)    round to nearest even, saturating at 448
//
// A row of zeros gets code 0 everywhere and d = 1.  The divides and the
// multiply are IEEE fp32 operations (no contraction), so the codes are fixed
// by the inputs.  One CTA per row.
#include <cuda_fp4.h>

#include "kernels.h"

namespace dflash2 {
namespace {

constexpr int kQuantThreads = 256;

template <typename T> __device__ __forceinline__ float qf(T v);
template <> __device__ __forceinline__ float qf<float>(float v) { return v; }
template <> __device__ __forceinline__ float qf<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

template <typename T>
__global__ void __launch_bounds__(kQuantThreads)
    quant_rows_kernel(const T *__restrict__ x, int cols, uint8_t *__restrict__ q,
                      float *__restrict__ d) {
    grid_dep_wait();
    __shared__ float red[kQuantThreads / 32];
    const int64_t row = blockIdx.x;
    const T *xr = x + row * cols;
    uint8_t *qr = q + row * cols;
    float amax = 0.0f;
    for (int j = threadIdx.x; j < cols; j += kQuantThreads) amax = fmaxf(amax, fabsf(qf(xr[j])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    if (amax == 0.0f) {
        for (int j = threadIdx.x; j < cols; j += kQuantThreads) qr[j] = 0;
        if (threadIdx.x == 0) d[row] = 1.0f;
        return;
    }
    const float inv = __fdiv_rn(448.0f, amax);
    for (int j = threadIdx.x; j < cols; j += kQuantThreads)
        qr[j] = (uint8_t)__nv_cvt_float_to_fp8(__fmul_rn(qf(xr[j]), inv), __NV_SATFINITE,
                                               __NV_E4M3);
    if (threadIdx.x == 0) d[row] = __fdiv_rn(amax, 448.0f);
}

// Per-row NVFP4 quantization (the activations of the NVFP4-head unary path):
//
//   amax = max_j |x[m, j]|,  enc = 2688 / amax,  g[m] = amax / 2688   (fp32;
//   2688 = 6 * 448; a row of zeros: enc = g = 1)
//   block b of 16 elements: a_b = max |x| over it,
//   s_b = E4M3((a_b / 6) * enc)  (round to nearest even, saturating),
//   codes q_j = E2M1(x_j * (enc / dec(s_b)))  (round to nearest even,
//   saturating at 6), all zero when s_b is zero.
//
// Each operation is one IEEE fp32 operation (no contraction), so the codes
// and scales are fixed by the inputs.  One CTA per row; thread t takes blocks
// t, t + 256, ...
template <typename T>
__global__ void __launch_bounds__(kQuantThreads)
    quant_rows_nvfp4_kernel(const T *__restrict__ x, int cols, uint8_t *__restrict__ codes,
                            uint8_t *__restrict__ scales, float *__restrict__ g) {
    grid_dep_wait();
    __shared__ float red[kQuantThreads / 32];
    const int64_t row = blockIdx.x;
    const T *xr = x + row * cols;
    float amax = 0.0f;
    for (int j = threadIdx.x; j < cols; j += kQuantThreads) amax = fmaxf(amax, fabsf(qf(xr[j])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    const float enc = amax == 0.0f ? 1.0f : __fdiv_rn(2688.0f, amax);
    const int nb = cols / 16;
    for (int b = threadIdx.x; b < nb; b += kQuantThreads) {
        float v[16];
        float ab = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            v[e] = qf(xr[16 * b + e]);
            ab = fmaxf(ab, fabsf(v[e]));
        }
        const float t = __fmul_rn(__fdiv_rn(ab, 6.0f), enc);
        const __nv_fp8_storage_t sc = __nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
        __nv_fp8_e4m3 sv;
        sv.__x = sc;
        const float ds = static_cast<float>(sv);
        uint32_t lo = 0, hi = 0;  // the 16 codes, 8 per word, element 2i in the low nibble
        if (ds != 0.0f) {
            const float r = __fdiv_rn(enc, ds);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const uint32_t c =
                    (uint32_t)__nv_cvt_float_to_fp4(__fmul_rn(v[e], r), __NV_E2M1, cudaRoundNearest) &
                    15u;
                if (e < 8)
                    lo |= c << (4 * e);
                else
                    hi |= c << (4 * (e - 8));
            }
        }
        reinterpret_cast<uint2 *>(codes + row * (cols / 2))[b] = make_uint2(lo, hi);
        scales[row * nb + b] = (uint8_t)sc;
    }
    if (threadIdx.x == 0) g[row] = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
}

// Scale tiles from row-major scales [rows][hidden / 16]: one thread per
// 32-bit cell of the tiles, zeros included, so the tiles need no clearing.
__global__ void __launch_bounds__(256)
    nvfp4_tile_kernel(const uint8_t *__restrict__ scales, int64_t rows, int n_sf,
                      int block_rows, int nw8, int64_t cells, uint32_t *__restrict__ tiles) {
    grid_dep_wait();
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < cells;
         c += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = c >> 7;  // 128 cells of 4 bytes per 512-byte tile
        const int in = (int)(c & 127), l = in >> 2, j = in & 3;
        const int64_t rb = tile / nw8;
        const int w = (int)(tile - rb * nw8);
        const int rl = l + 32 * j;
        const int64_t row = rb * block_rows + rl;
        uint32_t v = 0;
        if (rl < block_rows && row < rows && 4 * w < n_sf)
            v = __ldg(reinterpret_cast<const uint32_t *>(scales + row * n_sf) + w);
        tiles[c] = v;
    }
}

}  // namespace

dflash2_status launch_nvfp4_tile_scales(const uint8_t *scales, int64_t rows, int32_t hidden,
                                        int32_t block_rows, uint8_t *tiles, cudaStream_t st) {
    const int nw8 = nvfp4_tile_cells(hidden);
    const int64_t cells = (int64_t)nvfp4_tiles_bytes(rows, hidden, block_rows) / 4;
    int64_t blocks = (cells + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    launch_k(nvfp4_tile_kernel, (unsigned)blocks, 256, 0, st, scales, rows, hidden / 16,
             block_rows, nw8, cells, reinterpret_cast<uint32_t *>(tiles));
    return launch_status();
}

dflash2_status launch_quant_rows_nvfp4(const void *x, int32_t dtype, int64_t rows, int32_t cols,
                                       uint8_t *codes, uint8_t *scales, float *g,
                                       cudaStream_t st) {
    if (dtype == DFLASH2_BF16)
        launch_k(quant_rows_nvfp4_kernel<__nv_bfloat16>, (unsigned)rows, kQuantThreads, 0, st,
                 static_cast<const __nv_bfloat16 *>(x), cols, codes, scales, g);
    else
        launch_k(quant_rows_nvfp4_kernel<float>, (unsigned)rows, kQuantThreads, 0, st,
                 static_cast<const float *>(x), cols, codes, scales, g);
    return launch_status();
}

dflash2_status launch_quant_rows_e4m3(const void *x, int32_t dtype, int64_t rows, int32_t cols,
                                      uint8_t *q, float *d, cudaStream_t st) {
    if (dtype == DFLASH2_BF16)
        launch_k(quant_rows_kernel<__nv_bfloat16>, (unsigned)rows, kQuantThreads, 0, st,
                 static_cast<const __nv_bfloat16 *>(x), cols, q, d);
    else
        launch_k(quant_rows_kernel<float>, (unsigned)rows, kQuantThreads, 0, st,
                 static_cast<const float *>(x), cols, q, d);
    return launch_status();
}

}  // namespace dflash2

extern "C" dflash2_status dflash2_quantize_rows_e4m3(const void *x, int64_t rows, int32_t cols,
                                                     int32_t dtype, uint8_t *q, float *scale,
                                                     void *stream) {
    using namespace dflash2;
    if (dtype != DFLASH2_F32 && dtype != DFLASH2_BF16) return DFLASH2_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || rows > INT32_MAX || cols <= 0) return DFLASH2_ERR_INVALID_ARG;
    if (rows == 0) return DFLASH2_OK;
    if (!x || !q || !scale) return DFLASH2_ERR_INVALID_ARG;
    const uintptr_t esz = dtype == DFLASH2_BF16 ? 2 : 4;
    if (reinterpret_cast<uintptr_t>(x) % esz != 0 || reinterpret_cast<uintptr_t>(scale) % 4 != 0)
        return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    dflash2_status s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    return launch_quant_rows_e4m3(x, dtype, rows, cols, q, scale, static_cast<cudaStream_t>(stream));
}

extern "C" dflash2_status dflash2_quantize_rows_nvfp4(const void *x, int64_t rows, int32_t cols,
                                                      int32_t dtype, uint8_t *codes,
                                                      uint8_t *scales, float *g, void *stream) {
    using namespace dflash2;
    if (dtype != DFLASH2_F32 && dtype != DFLASH2_BF16) return DFLASH2_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || rows > INT32_MAX || cols <= 0 || cols % 16 != 0) return DFLASH2_ERR_INVALID_ARG;
    if (rows == 0) return DFLASH2_OK;
    if (!x || !codes || !scales || !g) return DFLASH2_ERR_INVALID_ARG;
    const uintptr_t esz = dtype == DFLASH2_BF16 ? 2 : 4;
    if (reinterpret_cast<uintptr_t>(x) % esz != 0 || reinterpret_cast<uintptr_t>(codes) % 8 != 0 ||
        reinterpret_cast<uintptr_t>(g) % 4 != 0)
        return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    dflash2_status s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    return launch_quant_rows_nvfp4(x, dtype, rows, cols, codes, scales, g,
                                   static_cast<cudaStream_t>(stream));
}

extern "C" size_t dflash2_nvfp4_scale_tiles_size(int64_t rows, int32_t hidden) {
    if (rows <= 0 || hidden <= 0 || hidden % 64 != 0) return 0;
    return dflash2::nvfp4_tiles_bytes(rows, hidden, 128);
}

extern "C" dflash2_status dflash2_nvfp4_tile_scales(const uint8_t *scales, int64_t rows,
                                                    int32_t hidden, uint8_t *tiles, void *stream) {
    using namespace dflash2;
    if (rows < 0 || rows > INT32_MAX || hidden <= 0 || hidden % 64 != 0)
        return DFLASH2_ERR_INVALID_ARG;
    if (rows == 0) return DFLASH2_OK;
    if (!scales || !tiles) return DFLASH2_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(scales) % 4 != 0 || !aligned16(tiles))
        return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    dflash2_status s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    return launch_nvfp4_tile_scales(scales, rows, hidden, 128, tiles,
                                    static_cast<cudaStream_t>(stream));
}
