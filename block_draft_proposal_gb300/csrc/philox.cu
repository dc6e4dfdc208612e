// Counter-based uniforms for the selector walk.
//
// The sglang DFlash2 sampler (_SelectorDraftSampler) draws the walk's
// uniforms inside the captured CUDA graph from a Philox generator whose state
// advances at every replay.  The generator here is Philox4x64 with 10 rounds
// (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2,
// 3", SC 2011).  Uniform i is word i % 4 of the block at counter
// (base + i / 4, 0, 0, 0) under key (seed, 0), mapped to [0, 1) as
// (word >> 40) * 2^-24, which fp32 holds exactly.
#include "common.cuh"

namespace dflash2 {
namespace {

// Round multipliers and Weyl key increments of Philox4x64 (the published
// constants of the generator).
constexpr uint64_t kPhiloxM0 = 0xD2E7470EE14C6C93ull;
constexpr uint64_t kPhiloxM1 = 0xCA5A826395121157ull;
constexpr uint64_t kPhiloxW0 = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kPhiloxW1 = 0xBB67AE8584CAA73Bull;
constexpr int64_t kMaxCounterUniforms = int64_t(1) << 24;  // one CTA serves the counter form

__device__ __forceinline__ void philox4x64_10(uint64_t c0, uint64_t k0, uint64_t k1,
                                              uint64_t (&w)[4]) {
    uint64_t c1 = 0, c2 = 0, c3 = 0;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t hi0 = __umul64hi(kPhiloxM0, c0), lo0 = kPhiloxM0 * c0;
        const uint64_t hi1 = __umul64hi(kPhiloxM1, c2), lo1 = kPhiloxM1 * c2;
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
    w[0] = c0;
    w[1] = c1;
    w[2] = c2;
    w[3] = c3;
}

__device__ __forceinline__ float unit_float(uint64_t w) {
    return (float)(uint32_t)(w >> 40) * 0x1p-24f;
}

// Writes the (up to) four uniforms of block j.
__device__ __forceinline__ void write_block(float *out, int64_t n, int64_t j, uint64_t base,
                                            uint64_t seed, bool vec) {
    uint64_t w[4];
    philox4x64_10(base + (uint64_t)j, seed, 0, w);
    const int64_t i0 = 4 * j;
    if (vec && i0 + 3 < n) {
        *reinterpret_cast<float4 *>(out + i0) =
            make_float4(unit_float(w[0]), unit_float(w[1]), unit_float(w[2]), unit_float(w[3]));
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (i0 + q < n) out[i0 + q] = unit_float(w[q]);
    }
}

__global__ void philox_kernel(uint64_t seed, uint64_t base, int64_t n, float *out) {
    grid_dep_wait();
    const bool vec = (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    const int64_t nb = (n + 3) / 4;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < nb;
         j += (int64_t)gridDim.x * blockDim.x)
        write_block(out, n, j, base, seed, vec);
}

// Counter form: one CTA; thread 0 reads the counter, and after the block
// broadcast, advances it by the blocks this call used.  Only thread 0 touches
// the counter, so its read precedes its write.
__global__ void philox_counter_kernel(uint64_t seed, uint64_t offset, uint64_t *counter, int64_t n,
                                      float *out) {
    grid_dep_wait();
    __shared__ uint64_t base_s;
    const int64_t nb = (n + 3) / 4;
    if (threadIdx.x == 0) {
        const uint64_t c = *counter;
        base_s = c + offset;
        *counter = c + (uint64_t)nb;
    }
    __syncthreads();
    const uint64_t base = base_s;
    const bool vec = (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    for (int64_t j = threadIdx.x; j < nb; j += blockDim.x) write_block(out, n, j, base, seed, vec);
}

}  // namespace
}  // namespace dflash2

extern "C" dflash2_status dflash2_philox_uniforms(uint64_t seed, uint64_t offset, uint64_t *counter,
                                                  int64_t n, float *out, void *stream) {
    using namespace dflash2;
    if (n < 0) return DFLASH2_ERR_INVALID_ARG;
    if (n == 0) return DFLASH2_OK;
    if (!out) return DFLASH2_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(out) % 4 != 0 || reinterpret_cast<uintptr_t>(counter) % 8 != 0)
        return DFLASH2_ERR_MISALIGNED;
    if (counter && n > kMaxCounterUniforms) return DFLASH2_ERR_INVALID_ARG;
    DeviceInfo di;
    dflash2_status s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (counter) {
        launch_k(philox_counter_kernel, 1, 256, 0, st, seed, offset, counter, n, out);
    } else {
        int64_t blocks = ((n + 3) / 4 + 255) / 256;
        const int64_t cap = (int64_t)di.sm_count * 4;
        if (blocks > cap) blocks = cap;
        launch_k(philox_kernel, (unsigned)blocks, 256, 0, st, seed, offset, n, out);
    }
    return launch_status();
}
