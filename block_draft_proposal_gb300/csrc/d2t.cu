// Draft-to-target id remap (vLLM Qwen3DSparkForCausalLM.map_draft_to_target):
// target = draft + d2t[draft] (d2t holds offsets); no table = identity.
#include "common.cuh"

namespace dflash2 {
namespace {

__global__ void d2t_kernel(const int64_t *__restrict__ ids, const int64_t *__restrict__ d2t,
                           int64_t n, int64_t draft_vocab, int64_t target_vocab,
                           int64_t *target_ids, int32_t *err) {
    grid_dep_wait();
    bool bad_any = false;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t d = ids[i];
        int64_t t = 0;
        bool bad = d < 0 || d >= draft_vocab;
        if (!bad) {
            t = d2t ? d + __ldg(d2t + d) : d;
            bad = t < 0 || t >= target_vocab;
        }
        target_ids[i] = bad ? 0 : t;
        bad_any |= bad;
    }
    if (bad_any && err) atomicOr(err, DFLASH2_DEVERR_ID_RANGE);
}

}  // namespace
}  // namespace dflash2

extern "C" dflash2_status dflash2_d2t_remap(const int64_t *draft_ids, const int64_t *d2t, int64_t n,
                                            int64_t draft_vocab, int64_t target_vocab,
                                            int64_t *target_ids, int32_t *err_word,
                                            void *stream) {
    using namespace dflash2;
    if (n < 0 || draft_vocab <= 0 || target_vocab <= 0) return DFLASH2_ERR_INVALID_ARG;
    // A table exists exactly for a pruned draft vocab (draft < target).
    if ((draft_vocab < target_vocab) != (d2t != nullptr)) return DFLASH2_ERR_INVALID_ARG;
    if (n == 0) return DFLASH2_OK;
    if (!draft_ids || !target_ids) return DFLASH2_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(draft_ids) | reinterpret_cast<uintptr_t>(target_ids) |
         reinterpret_cast<uintptr_t>(d2t)) % 8 != 0)
        return DFLASH2_ERR_MISALIGNED;
    DeviceInfo di;
    dflash2_status s = current_device(&di);
    if (s != DFLASH2_OK) return s;
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = (int64_t)di.sm_count * 8;
    if (blocks > cap) blocks = cap;
    launch_k(d2t_kernel, (unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream), draft_ids,
        d2t, n, draft_vocab, target_vocab, target_ids, err_word);
    return launch_status();
}
