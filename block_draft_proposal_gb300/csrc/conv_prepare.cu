// DFlashGroupedConv prepare / finish (sglang DFlash2 PR).
//
// One bias-free linear map of the input, kernel_projection =
// Linear(hidden, 2 * taps * groups), gives each token the dynamic
// coefficients of both convolutions, laid out [2, taps, groups]:
//
//   coef[i, r] = sum_j x[i, j] * w_kp[r, j],   r = (side * taps + t) * groups + g
//
// stored in the layer's dtype.  prepare() convolves the input with side 0 (and
// base_kernel[0]) and hands side 1 back for finish(), which convolves the
// sublayer's output with side 1 (and base_kernel[1]).  The projection runs on
// the tcgen05 GEMM (bf16, CTA pairs, bf16-rounding epilogue) or on CUDA cores
// (fp32); the convolutions read their side of coef in place through the
// conv's delta row stride.
#include "kernels.h"

namespace dflash2 {
namespace {

// fp32 projection on CUDA cores: one CTA per token, one warp per output at a
// time, lane-strided FMA over hidden then a warp tree sum.
__global__ void __launch_bounds__(256)
    kproj_f32_kernel(const float *__restrict__ x, const float *__restrict__ w, int hidden,
                     int out_features, float *coef) {
    grid_dep_wait();
    const int64_t i = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *xr = x + i * hidden;
    for (int r = warp; r < out_features; r += 8) {
        const float *wr = w + (int64_t)r * hidden;
        float acc = 0.0f;
        for (int j = lane; j < hidden; j += 32) acc = fmaf(xr[j], wr[j], acc);
        acc = warp_sum(acc);
        if (lane == 0) coef[i * out_features + r] = acc;
    }
}

// Token tile of the bf16 projection on CTA pairs: the candidate with the
// fewest estimated issue-bound cycles (waves x stages x per-stage cycles,
// where a stage of 8 MMAs costs the issuing thread about 750 cycles and the
// tensor pipe 4 * bn), larger tiles first on ties.
int kproj_tile(int64_t n_tokens, int out_features, int hidden, int sm_count) {
    const int64_t units = (out_features + 2 * kGemmTileW - 1) / (2 * kGemmTileW);
    const int64_t stages = (hidden + kGemmStageK - 1) / kGemmStageK;
    const int64_t pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
    int best_bn = 16;
    double best = -1.0;
    for (int bn : {256, 192, 128, 96, 64, 32, 16}) {
        if (bn > 16 && (int64_t)bn - 16 >= n_tokens) continue;  // a smaller tile covers it
        const int64_t items = units * ((n_tokens + bn - 1) / bn);
        const int64_t waves = (items + pairs - 1) / pairs;
        const double cost = (double)waves * (double)stages * (4.0 * bn > 750.0 ? 4.0 * bn : 750.0);
        if (best < 0.0 || cost < best) {
            best = cost;
            best_bn = bn;
        }
    }
    return best_bn;
}

}  // namespace
}  // namespace dflash2

using namespace dflash2;

extern "C" dflash2_status dflash2_conv_prepare(const void *x, const void *w_kp, const void *base2,
                                               int64_t n_tokens, int32_t hidden,
                                               int32_t group_size, int32_t taps,
                                               int32_t block_size, int32_t dtype, void *out,
                                               void *coef, int32_t *err_word, void *stream) {
    if (dtype != DFLASH2_F32 && dtype != DFLASH2_BF16) return DFLASH2_ERR_UNSUPPORTED_DTYPE;
    if (n_tokens < 0 || n_tokens > INT32_MAX || hidden <= 0 || group_size <= 0 ||
        hidden % group_size != 0 || taps < 1 || block_size < 1)
        return DFLASH2_ERR_INVALID_ARG;
    const int64_t groups = hidden / group_size;
    const int64_t out_features = 2 * (int64_t)taps * groups;
    if (out_features > INT32_MAX) return DFLASH2_ERR_INVALID_ARG;
    if (n_tokens == 0) return DFLASH2_OK;
    if (!x || !w_kp || !base2 || !out || !coef) return DFLASH2_ERR_INVALID_ARG;
    DeviceInfo di;
    dflash2_status s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == DFLASH2_F32) {
        if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_kp) |
             reinterpret_cast<uintptr_t>(coef)) % 4 != 0)
            return DFLASH2_ERR_MISALIGNED;
        launch_k(kproj_f32_kernel, (unsigned)n_tokens, 256, 0, st, static_cast<const float *>(x),
            static_cast<const float *>(w_kp), hidden,
            (int)out_features, static_cast<float *>(coef));
        s = launch_status();
    } else {
        // TMA: 16-byte aligned bases and row strides (hidden % 8 == 0)
        if (hidden % 8 != 0 || !aligned16(x) || !aligned16(w_kp) ||
            reinterpret_cast<uintptr_t>(coef) % 2 != 0)
            return DFLASH2_ERR_MISALIGNED;
        GemmParams p{};
        p.rows_w = (int32_t)out_features;
        p.rows_h = (int32_t)n_tokens;
        p.hidden = hidden;
        p.mode = kGemmStoreBf16;
        p.bn = kproj_tile(n_tokens, (int)out_features, hidden, di.sm_count);
        p.k_splits = 1;
        p.out_bf16 = static_cast<__nv_bfloat16 *>(coef);
        p.ldo = out_features;
        p.err = err_word;
        s = launch_gemm_tc(di, w_kp, x, p, st, /*pair=*/true);
    }
    if (s != DFLASH2_OK) return s;
    return dflash2_grouped_conv(x, base2, coef, out_features, out, n_tokens, hidden, group_size,
                                taps, block_size, dtype, stream);
}

extern "C" dflash2_status dflash2_conv_finish(const void *y, const void *base2, const void *coef,
                                              int64_t n_tokens, int32_t hidden, int32_t group_size,
                                              int32_t taps, int32_t block_size, int32_t dtype,
                                              void *out, void *stream) {
    if (dtype != DFLASH2_F32 && dtype != DFLASH2_BF16) return DFLASH2_ERR_UNSUPPORTED_DTYPE;
    if (n_tokens < 0 || hidden <= 0 || group_size <= 0 || hidden % group_size != 0 || taps < 1 ||
        block_size < 1)
        return DFLASH2_ERR_INVALID_ARG;
    if (n_tokens == 0) return DFLASH2_OK;
    if (!y || !base2 || !coef || !out) return DFLASH2_ERR_INVALID_ARG;
    const int64_t groups = hidden / group_size;
    const size_t esz = dtype == DFLASH2_BF16 ? 2 : 4;
    const uint8_t *base1 = static_cast<const uint8_t *>(base2) + (size_t)taps * hidden * esz;
    const uint8_t *coef1 = static_cast<const uint8_t *>(coef) + (size_t)taps * groups * esz;
    return dflash2_grouped_conv(y, base1, coef1, 2 * (int64_t)taps * groups, out, n_tokens, hidden,
                                group_size, taps, block_size, dtype, stream);
}
