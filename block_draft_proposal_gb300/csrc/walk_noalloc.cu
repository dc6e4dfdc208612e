// dflash2_selector_walk_noalloc: the selector walk without a caller-provided
// workspace.
//
// Some callers cannot hand the library a device buffer at call time:
//   - serving loops whose device memory is owned by another allocator, for
//     example a framework's caching allocator that reserved the pool up front
//     and must not be bypassed or fragmented;
//   - latency-critical paths that must never call into the CUDA allocator,
//     because cudaMalloc / cudaFree can synchronise the device and stall
//     every stream.
// For them this entry point keeps its scratch in a fixed array in the
// library's own device memory instead.  The array is defined at file scope,
// so every GPU that loads the library holds it until the process exits.
#include <mutex>

#include "common.cuh"

namespace dflash2 {
namespace {

// Upper bound of the scratch this entry point can use.  The walk's scratch
// holds the hidden-split partial projections (k_splits x rows x rank fp32)
// and, for top_k <= 32, the lattice (rows x top_k x (top_k + 3) x 4 bytes);
// 4 MiB covers, for example, 480 rows at rank 64 and top_k 16 (1.2 MiB) or
// 1408 rows at rank 64 and top_k 16 (2.3 MiB), but not 960 rows at top_k 32
// (4.3 MiB of lattice) nor 7680 rows at rank 128.
constexpr size_t kNoAllocScratchBytes = 4u << 20;
// The walk's shape limits (include/dflash2.h, dflash2_selector_walk).
constexpr int kNoAllocMaxRank = 256;
constexpr int kNoAllocMaxK = 128;

static __device__ __align__(256) unsigned char g_walk_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];  // device address of g_walk_scratch, per device

// Looks up (once per device, with that device current) the device address of
// the scratch array.  In host code the array's name is only a host-side
// stand-in, never a device address, so it is not passed to kernels directly.
// The address is kept for the life of the process: it stays valid as long as
// the device's primary context is not reset (cudaDeviceReset) meanwhile.
dflash2_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return DFLASH2_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_walk_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return DFLASH2_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return DFLASH2_OK;
}

}  // namespace
}  // namespace dflash2

extern "C" dflash2_status dflash2_selector_walk_noalloc(
    const void *h, const void *proj, const void *A, const void *B, int64_t table_rows,
    const int64_t *anchor_ids, const int64_t *cand_ids, const float *cand_u,
    const float *temperatures, const uint8_t *greedy, const float *uniforms, int32_t batch,
    int32_t slots, int32_t hidden, int32_t rank, int32_t top_k, int32_t dtype, int64_t *tokens,
    float *q, float *path_scores, int32_t *err_word, void *stream) {
    using namespace dflash2;
    // The same shape checks as the workspace entry point, first, so that an
    // invalid shape gets the same status from both; an empty batch queues
    // nothing and needs no scratch.
    if (dtype != DFLASH2_F32 && dtype != DFLASH2_BF16) return DFLASH2_ERR_UNSUPPORTED_DTYPE;
    const int rank_mult = dtype == DFLASH2_BF16 ? 8 : 4;
    if (batch < 0 || slots < 0 || hidden <= 0 || rank <= 0 || rank > kNoAllocMaxRank ||
        rank % rank_mult != 0 || top_k <= 0 || top_k > kNoAllocMaxK || table_rows <= 0)
        return DFLASH2_ERR_INVALID_ARG;
    if (batch == 0 || slots == 0) return DFLASH2_OK;
    // Then the scratch the shapes need: refuse what does not fit before
    // touching the device.
    const size_t need =
        dflash2_selector_walk_workspace_size(batch, slots, hidden, rank, top_k, dtype);
    if (need > kNoAllocScratchBytes) return DFLASH2_ERR_WORKSPACE;
    void *scratch = nullptr;
    const dflash2_status s = scratch_address(&scratch);
    if (s != DFLASH2_OK) return s;
    // The walk writes every partial it later reads, so the scratch needs no
    // clearing between calls.
    return dflash2_selector_walk(h, proj, A, B, table_rows, anchor_ids, cand_ids, cand_u,
                                 temperatures, greedy, uniforms, batch, slots, hidden, rank, top_k,
                                 dtype, tokens, q, path_scores, scratch, kNoAllocScratchBytes,
                                 err_word, stream);
}
