// Test probe, not part of the library: one pipeline wait that nothing ever
// completes, to check that the library's bounded wait gives up after its
// limit, sets the DFLASH2_DEVERR_TIMEOUT bit and returns, leaving the context
// usable.  Built and run by tests/test_gpu_wait_timeout.py.
#include "../block_draft_proposal_gb300/csrc/common.cuh"

using namespace dflash2;

__global__ void wait_probe_kernel(int32_t *err, unsigned long long *elapsed_ns, int *result) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_timer_ns();
        // phase 0 of a fresh barrier with one expected arrival: nobody arrives
        const bool done = mbar_wait(&bar, 0, &abort_flag, err);
        *elapsed_ns = global_timer_ns() - t0;
        *result = done ? 1 : (abort_flag ? 2 : 3);  // 2: gave up and raised the abort flag
    }
}

extern "C" int wait_probe(int32_t *err, unsigned long long *elapsed_ns, int *result) {
    wait_probe_kernel<<<1, 32>>>(err, elapsed_ns, result);
    return (int)cudaDeviceSynchronize();
}
