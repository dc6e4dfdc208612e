// Exact merge of vocab-sharded top-K lists.
//
// With the lm_head split by vocab rows over shards (one per GPU), each shard
// runs the unary GEMM and a top-K over its own rows; an all-gather of the
// [rows, K] (u, id) lists and this merge give every rank the unsharded
// result.  The logits of a vocab row do not depend on which shard computes
// them (the same tile loop over hidden), so the merge reproduces the
// unsharded top-K exactly: the K largest keys make_key(u, global id) of the
// union, ordered by u descending, equal u by the smaller id.
//
// One CTA per row: the shards' keys go to shared memory (an absent entry, u =
// -inf or NaN, becomes key 0, below every real key), a bitonic sort orders
// them descending, and the first k_out are written.  No input order is
// assumed.
#include "common.cuh"

namespace dflash2 {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kMergeMaxKeys = 4096;  // shards * k_in, padded to a power of two
constexpr int kMergeMaxShards = 64;
constexpr int kMergeMaxK = 128;  // the largest top-K dflash2_unary_topk produces

struct MergeOffsets {
    int64_t off[kMergeMaxShards];
};

__global__ void __launch_bounds__(kMergeThreads)
    merge_kernel(const int64_t *__restrict__ ids, const float *__restrict__ u, MergeOffsets offs,
                 int shards, int64_t rows, int k_in, int k_out, int n_pad, int64_t *out_ids,
                 float *out_u, int32_t *err) {
    grid_dep_wait();
    extern __shared__ uint64_t keys[];
    const int64_t row = blockIdx.x;
    const int n = shards * k_in;
    bool bad = false;
    for (int i = threadIdx.x; i < n_pad; i += kMergeThreads) {
        uint64_t key = 0;
        if (i < n) {
            const int s = i / k_in, j = i - s * k_in;
            const int64_t at = ((int64_t)s * rows + row) * k_in + j;
            const float v = u[at];
            if (v != -INFINITY && v == v) {
                const int64_t gid = ids[at] + offs.off[s];
                if (gid < 0 || gid > (int64_t)0xFFFFFFFEu) {
                    bad = true;  // an id no vocab can hold: dropped
                } else {
                    key = make_key(v, (uint32_t)gid);
                }
            }
        }
        keys[i] = key;
    }
    if (bad && err) atomicOr(err, DFLASH2_DEVERR_ID_RANGE);
    __syncthreads();
    for (int k2 = 2; k2 <= n_pad; k2 <<= 1) {
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n_pad; i += kMergeThreads) {
                const int x = i ^ j;
                if (x > i) {
                    const uint64_t a = keys[i], b = keys[x];
                    if ((a < b) == ((i & k2) == 0)) {  // descending blocks where (i & k2) == 0
                        keys[i] = b;
                        keys[x] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    bool short_row = false;
    for (int i = threadIdx.x; i < k_out; i += kMergeThreads) {
        const uint64_t key = i < n_pad ? keys[i] : 0;
        if (key != 0) {
            out_ids[row * k_out + i] = (int64_t)key_id(key);
            out_u[row * k_out + i] = key_u(key);
        } else {
            out_ids[row * k_out + i] = 0;
            out_u[row * k_out + i] = -INFINITY;
            short_row = true;
        }
    }
    if (short_row && err) atomicOr(err, DFLASH2_DEVERR_SHORT);
}

}  // namespace
}  // namespace dflash2

extern "C" dflash2_status dflash2_topk_merge(const int64_t *ids, const float *u,
                                             const int64_t *id_offsets, int32_t shards,
                                             int64_t rows, int32_t k_in, int32_t k_out,
                                             int64_t *out_ids, float *out_u, int32_t *err_word,
                                             void *stream) {
    using namespace dflash2;
    if (shards < 1 || shards > kMergeMaxShards || rows < 0 || rows > INT32_MAX || k_in < 1 ||
        k_out < 1 || k_out > kMergeMaxK || (int64_t)shards * k_in > kMergeMaxKeys)
        return DFLASH2_ERR_INVALID_ARG;
    if (rows == 0) return DFLASH2_OK;
    if (!ids || !u || !id_offsets || !out_ids || !out_u) return DFLASH2_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ids) | reinterpret_cast<uintptr_t>(out_ids)) % 8 != 0 ||
        (reinterpret_cast<uintptr_t>(u) | reinterpret_cast<uintptr_t>(out_u)) % 4 != 0)
        return DFLASH2_ERR_MISALIGNED;
    MergeOffsets offs{};
    for (int s = 0; s < shards; ++s) {
        if (id_offsets[s] < 0 || id_offsets[s] > INT32_MAX) return DFLASH2_ERR_INVALID_ARG;
        offs.off[s] = id_offsets[s];
    }
    DeviceInfo di;
    dflash2_status st = current_device(&di);
    if (st != DFLASH2_OK) return st;
    int n_pad = 1;
    while (n_pad < shards * k_in || n_pad < k_out) n_pad <<= 1;
    launch_k(merge_kernel, (unsigned)rows, kMergeThreads, (size_t)n_pad * sizeof(uint64_t),
             static_cast<cudaStream_t>(stream), ids, u, offs, shards, rows, (int)k_in,
             (int)k_out, n_pad, out_ids, out_u, err_word);
    return launch_status();
}
