// Internal helpers shared by the CUDA translation units of libdflash2.
//
// Device side: ordered (u, id) keys, warp reductions, and thin inline-PTX
// wrappers for mbarrier, TMA (cp.async.bulk.tensor) and the 5th-generation
// tensor-core instructions (tcgen05: TMEM alloc, MMA, commit, load).
// Host side: device capability check, SM count, tensor-map encoding.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "../../include/dflash2.h"

namespace dflash2 {

// ---------------------------------------------------------------------------
// Launches with programmatic stream serialization: a kernel of this library
// may be scheduled while the kernel before it on the stream drains (its launch
// latency and on-chip prologue overlap the previous kernel's tail).  Every
// kernel therefore calls grid_dep_wait() before it touches global memory that
// an earlier kernel may write, which returns once the previous grid has
// completed and its writes are visible; so the stream order of the data stays
// exactly as without it.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel on the stream be scheduled before this one ends: it may
// start once every CTA of this grid has executed this or exited.  It makes
// nothing visible to that kernel (whose grid_dep_wait() still waits for this
// grid to complete), so before its own grid_dep_wait() the next kernel may
// read only data that was complete before this kernel started.
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// Host helpers (host_common.cu)
// ---------------------------------------------------------------------------
struct DeviceInfo {
    int device;
    int sm_count;
    int max_smem_optin;
    bool supported;  // compute capability 10.3
};

// Fills `info` for the current device (cached per device).  Returns a status.
dflash2_status current_device(DeviceInfo *info);

// Encodes a 2-D bf16 tensor map over a row-major [rows, cols] matrix with a
// {64 columns, box_rows rows} box, 128-byte swizzle, zero fill out of bounds.
dflash2_status encode_tmap_bf16(CUtensorMap *map, const void *base, uint64_t rows,
                                uint64_t cols, uint32_t box_rows);
// The same for 1-byte (elem_bytes = 1, uint8 codes) or bf16 (2) elements: the
// box is one 128-byte swizzle row wide (128 / elem_bytes columns).
dflash2_status encode_tmap_bytes_2d(CUtensorMap *map, const void *base, uint64_t rows,
                                    uint64_t cols, uint32_t box_cols, uint32_t box_rows);
dflash2_status encode_tmap_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                              uint32_t box_rows, uint32_t elem_bytes);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

inline dflash2_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Ordered keys: one uint64 per (u, vocab id), larger key = better candidate.
// High word: the fp32 bits of u mapped to an unsigned order (negative values
// flipped, positive values with the sign bit set); low word: ~id, so an equal
// u prefers the smaller id.  -0 is folded onto +0 first so that the two zeros
// tie like equal floats do.  Key 0 never encodes a real entry (every finite
// or infinite u maps to a high word >= 0x007FFFFF), so 0 means "none".
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ uint32_t order_bits(float u) {
    if (u == 0.0f) u = 0.0f;
#ifdef __CUDA_ARCH__
    uint32_t b = __float_as_uint(u);
#else
    uint32_t b;
    memcpy(&b, &u, 4);
#endif
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__host__ __device__ __forceinline__ float order_to_float(uint32_t o) {
    uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
#ifdef __CUDA_ARCH__
    return __uint_as_float(b);
#else
    float f;
    memcpy(&f, &b, 4);
    return f;
#endif
}
__host__ __device__ __forceinline__ uint64_t make_key(float u, uint32_t id) {
    return ((uint64_t)order_bits(u) << 32) | (uint64_t)(0xFFFFFFFFu - id);
}
__host__ __device__ __forceinline__ uint32_t key_id(uint64_t k) {
    return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFu);
}
__host__ __device__ __forceinline__ float key_u(uint64_t k) { return order_to_float((uint32_t)(k >> 32)); }

// Softcap / multiplier transform of a raw logit (fp32).
__device__ __forceinline__ float unary_transform(float z, float mult, float cap) {
    return cap > 0.0f ? cap * tanhf((mult * z) / cap) : mult * z;
}

// ---------------------------------------------------------------------------
// Warp helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
    uint32_t lo = __shfl_sync(0xFFFFFFFFu, (uint32_t)v, src);
    uint32_t hi = __shfl_sync(0xFFFFFFFFu, (uint32_t)(v >> 32), src);
    return ((uint64_t)hi << 32) | lo;
}

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers (bounded waits), TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Every pipeline wait is bounded: after kWaitLimitNs without progress the
// waiter raises the CTA's abort flag and the device error bit and returns
// false; waiters that see the abort flag return false as well.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                if (err) atomicOr(err, DFLASH2_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Grid-wide counters of a cooperative launch (every CTA resident at once).
// A warp publishes what its lanes wrote with counter_arrive (all lanes call
// it); a waiter polls with acquire loads, bounded like mbar_wait, and reads
// the published data through L2 (__ldcg) afterwards.
__device__ __forceinline__ void counter_arrive(uint32_t *ctr, int lane) {
    __syncwarp();
    if (lane == 0) {
        __threadfence();
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
    }
    __syncwarp();
}
__device__ __forceinline__ bool counter_wait(const uint32_t *ctr, uint32_t target,
                                             volatile int *abort_flag, int32_t *err, int lane) {
    int ok = 1;
    if (lane == 0) {
        const uint64_t t0 = global_timer_ns();
        for (;;) {
            uint32_t v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
            if (v >= target) break;
            if (*abort_flag) {
                ok = 0;
                break;
            }
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                if (err) atomicOr(err, DFLASH2_DEVERR_TIMEOUT);
                ok = 0;
                break;
            }
            __nanosleep(128);
        }
        __threadfence();
    }
    return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// 2-D tiled TMA load into this CTA's shared memory; completion is signalled
// on `bar` as transaction bytes.  c0 is the column (inner) coordinate.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (Blackwell 5th-generation tensor cores, TMEM accumulators)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Loads 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane
// per thread) and waits for them, in one asm statement so that no use of the
// registers can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// One fp32 TMEM column of this warp's 32 lanes (one value per thread), waited.
__device__ __forceinline__ float tmem_ld1_wait(uint32_t taddr) {
    uint32_t r;
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r)
        : "r"(taddr)
        : "memory");
    return __uint_as_float(r);
}

// ---- CTA pairs (clusters of 2) for the 2-CTA tensor-core MMA ----------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
// Arrive on an mbarrier given by its shared::cluster address (possibly remote).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
// 2-D TMA load into this CTA's shared memory whose completion is counted on
// an mbarrier of the pair's leader CTA (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void *smem_dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster_addr, int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D[tmem] (+)= A * B^T over the CTA pair: M = 256 rows split across the two
// CTAs' shared memory (same offsets), N columns split likewise; issued by the
// leader CTA only.
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The same for 8-bit operands (kind::f8f6f4: K = 32 elements = 32 bytes per MMA,
// so the shared-memory descriptors advance exactly as for bf16).
__device__ __forceinline__ void tc_mma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The same for E2M1 operands with block scales (kind::mxf4nvf4, one E4M3
// scale per 16 elements: K = 64 elements = 32 bytes per MMA).  The scales are
// read from TMEM at sfa / sfb, laid out as measured on GB300 with tcgen05.st:
// row i of a CTA's 128 weight rows in its lane i, column sfa + i / 32; token n
// in column sfb + n / 32 of every lane quarter (lane 32q + n % 32), in each
// CTA of the pair (both CTAs hold every token's scales); byte b of a 32-bit
// cell scales elements 16b .. 16b + 15 of the MMA's 64.
__device__ __forceinline__ void tc_mma_nvfp4_pair(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc, uint32_t sfa,
                                                  uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
        "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}
// Stores of 32-bit cells into TMEM: lane i of the warp writes lane
// (its quarter's base + i), columns taddr .. taddr + N - 1.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v)
                 : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2,
                                         uint32_t v3) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
                 "r"(v0), "r"(v1), "r"(v2), "r"(v3)
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrive once on the mbarrier at this shared offset in every CTA of `mask`
// when the pair's tcgen05 operations issued so far complete.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(mask)
        : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor for a K-major bf16 tile written by TMA with
// 128-byte swizzle: rows of 128 bytes (64 elements), 8-row groups 1024 bytes
// apart.  Advancing K by 16 elements inside the 128-byte row adds 32 bytes
// to the start address (the swizzle is a function of the address bits, so the
// tile base must be 1024-byte aligned).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);  // start address, 16-byte units
    d |= (uint64_t)1 << 16;                        // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;              // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                        // descriptor version for sm_100 family
    d |= (uint64_t)2 << 61;                        // layout: 128-byte swizzle
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 x bf16 -> fp32,
// both operands K-major, tile M x N.
// Instruction descriptor of kind::f8f6f4 with E4M3 A and B (format code 0 for
// both), fp32 accumulator, K-major operands.
__host__ __device__ constexpr uint32_t idesc_e4m3(int m, int n) {
    return (1u << 4)                      // accumulator format fp32
           | (0u << 7)                    // A format E4M3
           | (0u << 10)                   // B format E4M3
           | ((uint32_t)(n >> 3) << 17)   // N / 8
           | ((uint32_t)(m >> 4) << 24);  // M / 16
}
// Instruction descriptor of kind::mxf4nvf4 (block-scaled): E2M1 A and B
// (format code 1), UE4M3 scales (bit 23 clear), scale-factor ids 0 (a 4X
// scale vector fills the 32-bit cell), K-major operands, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_nvfp4(int m, int n) {
    return (1u << 7)                      // A format E2M1
           | (1u << 10)                   // B format E2M1
           | ((uint32_t)(n >> 3) << 17)   // N / 8
           | ((uint32_t)(m >> 4) << 24);  // M / 16
}
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4)                      // accumulator format fp32
           | (1u << 7)                    // A format bf16
           | (1u << 10)                   // B format bf16
           | ((uint32_t)(n >> 3) << 17)   // N / 8
           | ((uint32_t)(m >> 4) << 24);  // M / 16
}

}  // namespace dflash2
