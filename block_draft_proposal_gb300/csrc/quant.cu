// Per-row E4M3 quantization of activations (W8A8 with dynamic per-token
// scales), the first step of the FP8-head unary path:
//
//   amax = max_j |x[m, j]|,  inv = 448 / amax,  d[m] = amax / 448   (fp32)
//   q[m, j] = E4M3(x[m, j] * inv)    round to nearest even, saturating at 448
//
// A row of zeros gets code 0 everywhere and d = 1.  The divides and the
// multiply are IEEE fp32 operations (no contraction), so the codes are fixed
// by the inputs.  One CTA per row.
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

}  // namespace

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
