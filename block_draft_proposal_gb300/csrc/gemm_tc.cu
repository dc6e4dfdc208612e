// Persistent warp-specialised GEMM on the 5th-generation tensor cores, bf16
// (kind::f16) or, on CTA pairs, E4M3 codes with per-row scales (kind::f8f6f4).
//
//   C[m, v] = sum_j h[m, j] * w[v, j]      (w: lm_head or selector projection)
//   fp8:   C[m, v] = a_scale[m] * w_scale[v] * sum_j h[m, j] * w[v, j]
//
// Swap-AB: the weight rows are the MMA's M side (128-row tiles) and the
// tokens its N side (bn-column tiles, bn <= 256), so the fp32 accumulator of
// one tile is 128 TMEM lanes x bn columns and each epilogue thread owns one
// weight row (one vocab id) across the tile's tokens.
//
// Roles (192 threads, one CTA per SM, persistent over work items):
//   warp 0  lane 0: TMA producer (cp.async.bulk.tensor, 128-byte swizzle)
//   warp 1  lane 0: MMA issuer (tcgen05.mma kind::f16, accumulator in TMEM)
//   warps 2-5     : epilogue (tcgen05.ld; 4 warps cover the 128 TMEM lanes)
// Shared-memory stages are handed over with mbarriers (full: TMA bytes
// landed; empty: the MMAs reading the stage completed).  Two TMEM
// accumulators alternate so the epilogue of one tile overlaps the MMAs of
// the next.  Every wait is bounded (common.cuh).
//
// A stage holds 128 hidden elements of both operands, as two 64-element
// boxes (one 128-byte swizzle row each), so one wait and one commit cover 8
// MMAs.  The issuing thread is the limit at these tile sizes: an MMA costs
// it tens of cycles to issue, and each wait / fence / commit round a few
// hundred, against 120 tensor cycles per MMA at N = 240.  Its loop therefore
// keeps precomputed descriptors and an incremental stage / phase counter.
//
// An E4M3 box holds 128 codes in the same 128-byte row, so a stage of the
// same bytes covers 256 hidden elements and the same descriptor steps (32
// bytes per MMA, K = 32 codes) serve both kinds.
//
// Work items are ordered with the token tile fastest, so the CTAs that run
// at the same time share weight tiles in L2 and the weight matrix streams
// from HBM about once per group of token tiles (the token rows go in groups
// of at most 64 MB).  Modes: store (split-K fp32 partials), store-rows,
// store-bf16, the top-K's pilot and filter passes, and their fused
// cooperative launch (the CTA-pair variant below).  The store modes let the
// next kernel on the stream launch at their entry.
#include "kernels.h"

#include <atomic>

namespace dflash2 {
namespace {

constexpr uint32_t kWTileBytes = kGemmTileW * kGemmTileK * 2;  // one weight box: 16 KiB
constexpr uint32_t kWStageBytes = 2 * kWTileBytes;              // weight rows of one stage
constexpr size_t kGemmSmemBytes = 220 * 1024;                   // dynamic shared memory cap
constexpr double kTokGroupBytes = 64.0 * 1024 * 1024;          // token rows kept in L2 per group

__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// The 8 MMAs (K = 16 each) of one stage.  wd / hd are the descriptors of the
// stage's first weight / token box; +2 advances 32 bytes (16 elements) inside
// the 128-byte swizzled row, +wsub / +hsub moves to the second box (all in the
// descriptor's 16-byte address units).
template <bool PAIR>
__device__ __forceinline__ void mma_stage(uint32_t d, uint64_t wd, uint64_t hd, uint32_t wsub,
                                          uint32_t hsub, uint32_t idesc, uint32_t acc0) {
    if (PAIR) {
        tc_mma_bf16_pair(d, wd, hd, idesc, acc0);
        tc_mma_bf16_pair(d, wd + 2, hd + 2, idesc, 1u);
        tc_mma_bf16_pair(d, wd + 4, hd + 4, idesc, 1u);
        tc_mma_bf16_pair(d, wd + 6, hd + 6, idesc, 1u);
        tc_mma_bf16_pair(d, wd + wsub, hd + hsub, idesc, 1u);
        tc_mma_bf16_pair(d, wd + wsub + 2, hd + hsub + 2, idesc, 1u);
        tc_mma_bf16_pair(d, wd + wsub + 4, hd + hsub + 4, idesc, 1u);
        tc_mma_bf16_pair(d, wd + wsub + 6, hd + hsub + 6, idesc, 1u);
    } else {
        tc_mma_bf16(d, wd, hd, idesc, acc0);
        tc_mma_bf16(d, wd + 2, hd + 2, idesc, 1u);
        tc_mma_bf16(d, wd + 4, hd + 4, idesc, 1u);
        tc_mma_bf16(d, wd + 6, hd + 6, idesc, 1u);
        tc_mma_bf16(d, wd + wsub, hd + hsub, idesc, 1u);
        tc_mma_bf16(d, wd + wsub + 2, hd + hsub + 2, idesc, 1u);
        tc_mma_bf16(d, wd + wsub + 4, hd + hsub + 4, idesc, 1u);
        tc_mma_bf16(d, wd + wsub + 6, hd + hsub + 6, idesc, 1u);
    }
}

// The 8 MMAs of one stage for 8-bit operands on a CTA pair (K = 32 elements,
// still 32 bytes per MMA: the same descriptor steps, twice the hidden span).
__device__ __forceinline__ void mma_stage_f8_pair(uint32_t d, uint64_t wd, uint64_t hd,
                                                  uint32_t wsub, uint32_t hsub, uint32_t idesc,
                                                  uint32_t acc0) {
    tc_mma_f8_pair(d, wd, hd, idesc, acc0);
    tc_mma_f8_pair(d, wd + 2, hd + 2, idesc, 1u);
    tc_mma_f8_pair(d, wd + 4, hd + 4, idesc, 1u);
    tc_mma_f8_pair(d, wd + 6, hd + 6, idesc, 1u);
    tc_mma_f8_pair(d, wd + wsub, hd + hsub, idesc, 1u);
    tc_mma_f8_pair(d, wd + wsub + 2, hd + hsub + 2, idesc, 1u);
    tc_mma_f8_pair(d, wd + wsub + 4, hd + hsub + 4, idesc, 1u);
    tc_mma_f8_pair(d, wd + wsub + 6, hd + hsub + 6, idesc, 1u);
}

// The 8 MMAs of one stage for E2M1 operands on a CTA pair (K = 64 elements =
// 32 bytes per MMA), MMA i (= 4 * box + step) reading its scales from TMEM
// columns sf + 4i (weight rows) and sf + 32 + 4i (tokens).
__device__ __forceinline__ void mma_stage_nvfp4_pair(uint32_t d, uint64_t wd, uint64_t hd,
                                                     uint32_t wsub, uint32_t hsub, uint32_t idesc,
                                                     uint32_t acc0, uint32_t sf) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t off = (i >= 4 ? 1u : 0u), step = 2u * (uint32_t)(i & 3);
        tc_mma_nvfp4_pair(d, wd + off * wsub + step, hd + off * hsub + step, idesc,
                          sf + 4u * (uint32_t)i, sf + 32u + 4u * (uint32_t)i, i == 0 ? acc0 : 1u);
    }
}

// Waits (bounded) until the last `stages` loads this producer issued have
// landed, so no copy is still writing shared memory when the CTA leaves.
__device__ __forceinline__ void drain_loads(uint64_t *full_bar, uint32_t issued, uint32_t stages) {
    for (uint32_t n = issued > stages ? issued - stages : 0; n < issued; ++n)
        mbar_wait_drain(&full_bar[n % stages], (n / stages) & 1u);
}

// Which weight tile the j-th tile of this launch's pass is.
__device__ __forceinline__ int pass_tile(const GemmParams &p, int j) {
    if (p.mode == kGemmPilot) return j * p.pilot_stride;
    if (p.mode == kGemmFused) {  // the pilot tiles first, then the filter's order
        if (j < p.n_pilot) return j * p.pilot_stride;
        j -= p.n_pilot;
    }
    if (p.mode == kGemmFilter || p.mode == kGemmFused) {
        const int per = p.pilot_stride - 1;  // non-pilot tiles between two pilot tiles
        const int in_blocks = p.n_pilot * per;
        if (per > 0 && j < in_blocks) return (j / per) * p.pilot_stride + 1 + (j % per);
        return p.n_pilot * p.pilot_stride + (j - in_blocks);
    }
    return j;
}

struct Item {
    int wt, nt, ks, j;
    bool pilot;   // a pilot tile: raw logits to out
    bool filter;  // a filter tile: candidates against the row thresholds
};
__device__ __forceinline__ Item decode(const GemmParams &p, int w) {
    Item it;
    it.ks = w % p.k_splits;
    const int rest = w / p.k_splits;
    if (p.tok_group <= 0 || p.tok_group >= p.n_tok_tiles) {
        it.nt = rest % p.n_tok_tiles;
        it.j = rest / p.n_tok_tiles;
    } else {
        // groups of tok_group token tiles, each over every weight unit of the
        // pass, token tiles fastest within a group
        const int per = p.tok_group * p.pass_tiles;
        const int q = rest / per;
        const int r = rest - q * per;
        const int t0 = q * p.tok_group;
        const int gq = min(p.tok_group, p.n_tok_tiles - t0);
        it.nt = t0 + r % gq;
        it.j = r / gq;
    }
    it.wt = pass_tile(p, it.j);
    it.pilot = p.mode == kGemmPilot || (p.mode == kGemmFused && it.j < p.n_pilot);
    it.filter = p.mode == kGemmFilter || (p.mode == kGemmFused && it.j >= p.n_pilot);
    return it;
}

// Epilogue of 32 accumulator columns (tokens m0 .. m0+31) of one weight row v.
__device__ __forceinline__ void epilogue_chunk(const GemmParams &p, const float (&z)[32], int64_t v,
                                               int row_in_tile, int m0, int ncols, const Item &it,
                                               int lane) {
    if (p.mode == kGemmStore) {
        if (v < p.rows_w) {
            float *o = p.out + (int64_t)it.ks * p.split_stride + v;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int m = m0 + i;
                if (i < ncols && m < p.rows_h) o[(int64_t)m * p.ldo] = z[i];
            }
        }
    } else if (p.mode == kGemmStoreRows) {
        if (v < p.rows_w) {
            float *o = p.out + (int64_t)it.ks * p.split_stride + v * p.ldo + m0;
            if (ncols == 32 && m0 + 32 <= p.rows_h) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4 *>(o + i) = make_float4(z[i], z[i + 1], z[i + 2], z[i + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < ncols && m0 + i < p.rows_h) o[i] = z[i];
            }
        }
    } else if (p.mode == kGemmStoreBf16) {
        if (v < p.rows_w) {
            __nv_bfloat16 *o = p.out_bf16 + v;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int m = m0 + i;
                if (i < ncols && m < p.rows_h) o[(int64_t)m * p.ldo] = __float2bfloat16_rn(z[i]);
            }
        }
    } else if (it.pilot) {
        // raw logits; the pilot select applies the transform (-inf = padded / out of range)
        const bool valid = v < p.rows_w && v < p.target_vocab;
        float *o = p.out + (int64_t)it.j * p.unit + row_in_tile;  // row_in_tile: offset in the unit
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int m = m0 + i;
            if (i < ncols && m < p.rows_h) o[(int64_t)m * p.ldo] = valid ? z[i] : -INFINITY;
        }
    }
}

// Bf16 store of one 32 x 32 chunk on CTA pairs: the warp's weight rows v0 ..
// v0 + 31 (lane i holds row v0 + i) and tokens m0 .. m0 + ncols - 1.  The
// chunk goes through the warp's shared tile [32 tokens][32 rows] (rows of 64
// bytes), so that each lane then writes 8 consecutive outputs of one token
// row with one 16-byte store (vec: 16-byte aligned rows), instead of 32
// two-byte stores per lane.
__device__ __forceinline__ void store_bf16_chunk(const GemmParams &p, const float (&z)[32], int64_t v0,
                                                 int m0, int ncols, bool vec, __nv_bfloat16 *tile,
                                                 int lane) {
#pragma unroll
    for (int i = 0; i < 32; ++i) tile[i * 32 + lane] = __float2bfloat16_rn(z[i]);
    __syncwarp();
    const int64_t vq = v0 + 8 * (lane & 3);  // this lane's 8 consecutive rows
    const bool full = vec && vq + 8 <= p.rows_w;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = 8 * j + (lane >> 2);  // the token of this store within the chunk
        const int m = m0 + r;
        if (r < ncols && m < p.rows_h) {
            const uint4 val = *reinterpret_cast<const uint4 *>(tile + r * 32 + 8 * (lane & 3));
            __nv_bfloat16 *o = p.out_bf16 + (int64_t)m * p.ldo + vq;
            if (full) {
                *reinterpret_cast<uint4 *>(o) = val;
            } else {
                const __nv_bfloat16 *e = reinterpret_cast<const __nv_bfloat16 *>(&val);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (vq + q < p.rows_w) o[q] = e[q];
            }
        }
    }
    __syncwarp();  // the tile is rewritten by the next chunk
}

// Fused pilot tile: the warp's 32 vocab rows form group g; lane i stores the
// order bits of the group's largest logit for token m0 + i (NaN and invalid
// rows count as -inf).
__device__ __forceinline__ void group_max_chunk(const GemmParams &p, const float (&z)[32],
                                                bool valid, int m0, int ncols, int g, int lane) {
    uint32_t mine = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float zi = valid && z[i] == z[i] ? z[i] : -INFINITY;
        const uint32_t r = __reduce_max_sync(0xFFFFFFFFu, order_bits(zi));
        if (lane == i) mine = r;
    }
    const int m = m0 + lane;
    if (lane < ncols && m < p.rows_h) p.pmax[(int64_t)m * p.ld_pmax + g] = mine;
}

// fp8: C = acc * (a_scale[m] * w_scale[v]) for a chunk of 32 tokens m0 ..
// m0 + 31 (lane i loads a_scale[m0 + i], zero past the last token; wsv is the
// thread's w_scale[v]).  Returns the lane's a_scale, with which a single
// column re-read later is scaled by the same expression.
__device__ __forceinline__ float fp8_scale_chunk(const GemmParams &p, float (&z)[32], int m0,
                                                 float wsv, int lane) {
    const int m = m0 + lane;
    const float a = m < p.rows_h ? __ldg(p.a_scale + m) : 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] *= __shfl_sync(0xFFFFFFFFu, a, i) * wsv;
    return a;
}

// Per-epilogue-warp shared scratch of the filter mode: the thresholds of the
// current tile's tokens and a buffer of survivors waiting for their global
// slots.
constexpr int kEpiBuf = 128;
template <int COLS>
struct EpiScratchT {
    float pre[COLS];
    uint64_t th[COLS];
    uint64_t key[kEpiBuf];
    int32_t row[kEpiBuf];
};
using EpiScratch = EpiScratchT<256>;      // one CTA: a warp covers every column of a tile
constexpr int kPairEpiWarps = 8;          // CTA pairs: two warps per TMEM lane quarter,
constexpr int kPairEpiCols = 128;         // each on half of the tile's columns
using EpiScratchPair = EpiScratchT<kPairEpiCols>;
constexpr int kPairThreads = 64 + 32 * kPairEpiWarps;  // producer, MMA issuer, epilogue
constexpr uint32_t kBf16TileBytes = 32 * 32 * 2;       // an epilogue warp's bf16 transpose tile
// nvfp4: TMEM holds the two accumulators (<= 128 columns each) and then 64
// scale columns per stage: 32 for the weight rows (4 per MMA) and 32 for
// the tokens.  A stage's scales come with its operands: the producer's TMA
// copies 8 scale tiles of each side (4 KB) into the stage's shared scale
// slot, and the MMA warp moves them into TMEM with tcgen05.cp ahead of the
// stage's MMAs, in issue order with them.  (Scale-loader warps that wrote
// TMEM themselves made every stage wait for a software round trip: 0.52 ms
// against 0.37 for bf16 at the Qwen3-8B size.)
constexpr uint32_t kSfBase = 256;
constexpr uint32_t kSfCols = 64;
constexpr int kNvStages = 3;                    // operand stages and TMEM scale slots
constexpr uint32_t kNvSfStageBytes = 2 * 4096;  // 8 tiles of weight-row and of token scales
static_assert(kSfBase + kNvStages * kSfCols <= 512, "TMEM columns");

// One 512-byte scale tile (32 rows x 16 bytes, no swizzle: core matrices of
// 8 rows x 16 bytes, 128 bytes apart) from shared memory into TMEM columns
// taddr .. taddr + 3 of every lane quarter, on both CTAs of the pair (each
// from its own shared memory at the same offset).  Measured on GB300 to give
// the layout the block-scaled MMA reads.
__device__ __forceinline__ void tc_cp_sf_pair(uint32_t taddr, uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128 >> 4) << 16;  // leading byte offset
    d |= (uint64_t)(128 >> 4) << 32;  // stride byte offset: 8 rows x 16 bytes
    d |= (uint64_t)1 << 46;           // descriptor version for the sm_100 family
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d)
                 : "memory");
}

// Moves the buffered survivors to their rows' candidate lists: one global
// atomic per survivor, issued by all lanes together.
template <typename S>
__device__ __noinline__ void flush_survivors(const GemmParams &p, S &es, int n, int lane) {
    __syncwarp();
#pragma unroll 4
    for (int e = lane; e < n; e += 32) {
        const int row = es.row[e];
        const uint32_t slot = atomicAdd(p.cnt + row, 1u);
        if (slot < (uint32_t)p.cand_cap) p.cand[(int64_t)row * p.cand_cap + slot] = es.key[e];
    }
    __syncwarp();
}

// Filter epilogue of 32 columns (tokens m0 .. m0+31; c0 indexes them in the
// warp's scratch, tcol in TMEM).
// fl(mult * z), the first rounding step of the transform, is compared with
// the token's pre-threshold; only where some lane passes is the exact key
// formed and compared with the threshold key (pilot_select_kernel shows the
// pre-threshold never drops a key that reaches it).  The rare columns with a
// hit are visited in a compact loop that re-reads the one column from TMEM,
// which keeps the code small.  Keys that pass are buffered in shared memory;
// nbuf counts them (warp-uniform).
template <typename S>
__device__ __forceinline__ void filter_chunk(const GemmParams &p, const float (&z)[32], int64_t v,
                                             int m0, int c0, uint32_t tcol, S &es,
                                             int &nbuf, int lane, float asc = 1.0f,
                                             float wsv = 1.0f) {
    const bool valid_v = v < p.rows_w && v < p.target_vocab;
    float pre[32];  // the 32 tokens' pre-thresholds: broadcast 16-byte shared loads
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 v4 = reinterpret_cast<const float4 *>(es.pre + c0)[q];
        pre[4 * q] = v4.x;
        pre[4 * q + 1] = v4.y;
        pre[4 * q + 2] = v4.z;
        pre[4 * q + 3] = v4.w;
    }
    uint32_t hits = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) hits |= (p.mult * z[i] >= pre[i]) ? (1u << i) : 0u;
    if (!valid_v) hits = 0;
    uint32_t cols = __reduce_or_sync(0xFFFFFFFFu, hits);
    if (cols == 0) return;
    const uint64_t th_lane = es.th[c0 + lane];
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll 1
    while (cols) {  // warp-uniform
        const int i = __ffs(cols) - 1;
        cols &= cols - 1;
        float zi = tmem_ld1_wait(tcol + (uint32_t)i);
        if (p.fp8 || p.nvfp4) zi *= __shfl_sync(0xFFFFFFFFu, asc, i) * wsv;  // as fp8_scale_chunk
        const uint64_t th = shfl_u64(th_lane, i);
        bool pass = false;
        uint64_t key = 0;
        if ((hits >> i) & 1u) {
            key = make_key(unary_transform(zi, p.mult, p.cap), (uint32_t)v);
            pass = key >= th;
        }
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, pass);
        if (b) {
            if (nbuf + 32 > kEpiBuf) {
                flush_survivors(p, es, nbuf, lane);
                nbuf = 0;
            }
            if (pass) {
                const int pos = nbuf + __popc(b & lt);
                es.key[pos] = key;
                es.row[pos] = m0 + i;
            }
            nbuf += __popc(b);
        }
    }
}

// ---- fused mode: the row thresholds on the epilogue warps -------------------
// One row's pilot select on one warp.  The groups are the 32-row slices of
// the pilot units (lane l holds unit l's 8 group maxima, written by the pilot
// tiles' epilogues).  z* = the k-th largest group maximum, found by a bitwise
// search over their order bits in registers: at least k entries have
// z >= z*, hence u >= u* = the transform of z*, hence a key at or above the
// smallest key of value u*, which is theta (a lower bound of the row's k-th
// best key; the pre-threshold follows from u* as in pilot_select_kernel in
// topk.cu).  The pilot tiles' own candidates are then taken from their
// accumulators like any filter tile's, so the select writes only theta, the
// pre-threshold and a zero count.  It keeps off shared memory and nearly off
// the load path, which are busy feeding the tensor cores while it runs.
// Used only with mult > 0 (a non-decreasing transform).
__device__ __noinline__ void fused_select_row(const GemmParams &p, int64_t row, int lane) {
    const int k = p.top_k;
    const uint32_t kNegInf = order_bits(-INFINITY);
    uint32_t ob[8];
    if (lane < p.n_pilot) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.pmax + row * p.ld_pmax + 8 * lane);
        const uint4 a = __ldcg(src), b = __ldcg(src + 1);
        ob[0] = a.x; ob[1] = a.y; ob[2] = a.z; ob[3] = a.w;
        ob[4] = b.x; ob[5] = b.y; ob[6] = b.z; ob[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) ob[i] = kNegInf;
    }
    // the largest T with at least k maxima >= T is the k-th largest maximum
    uint32_t T = 0;
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t c = T | (1u << bit);
        uint32_t n = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) n += ob[i] >= c ? 1u : 0u;
        if (__reduce_add_sync(0xFFFFFFFFu, n) >= (uint32_t)k) T = c;
    }
    const float zs = order_to_float(T);
    uint64_t th;
    float pre;
    if (zs == -INFINITY) {
        th = 0;  // fewer than k groups hold a valid entry: all are candidates
        pre = -INFINITY;
    } else {
        const float us = unary_transform(zs, p.mult, p.cap);
        th = make_key(us, 0xFFFFFFFFu);  // the smallest key of value u*
        pre = us > 0.0f ? us * (1.0f - 0x1p-18f) : -INFINITY;
    }
    if (lane == 0) {
        const_cast<uint64_t *>(p.theta)[row] = th;
        const_cast<float *>(p.theta_pre)[row] = pre;
        p.cnt[row] = 0;
    }
}

// Every epilogue warp of the launch (kPairEpiWarps per CTA) waits for the pilot tiles'
// group maxima, selects rows gw, gw + nw, ... and publishes; false when a
// bounded wait gave up.
__device__ bool fused_select(const GemmParams &p, volatile int *abort_flag, int lane) {
    const int nw = (int)gridDim.x * kPairEpiWarps;
    const int gw = (int)blockIdx.x * kPairEpiWarps + ((int)(threadIdx.x >> 5) - 2);
    // every epilogue warp of both CTAs arrives once per pilot tile
    const uint32_t pilot_warps =
        (uint32_t)p.n_pilot * (uint32_t)p.n_tok_tiles * (2u * kPairEpiWarps);
    if (!counter_wait(p.sync, pilot_warps, abort_flag, p.err, lane)) return false;
    for (int64_t row = gw; row < p.rows_h; row += nw) fused_select_row(p, row, lane);
    counter_arrive(p.sync + 1, lane);
    return true;
}

__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
                   const GemmParams p) {
    extern __shared__ uint8_t dsmem[];
    __shared__ uint64_t full_bar[kGemmMaxStages];
    __shared__ uint64_t empty_bar[kGemmMaxStages];
    __shared__ uint64_t acc_full[2];
    __shared__ uint64_t acc_empty[2];
    __shared__ uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t h_sub = (uint32_t)p.bn * kGemmTileK * 2;  // one token box
    const uint32_t h_stage = 2 * h_sub;
    uint8_t *w_smem = smem;
    uint8_t *h_smem = smem + (size_t)p.stages * kWStageBytes;
    EpiScratch *epi = reinterpret_cast<EpiScratch *>(h_smem + (size_t)p.stages * h_stage);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t tmem_cols = 2 * p.acc_cols;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 4);
        }
        mbar_init(&drain_bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    if (warp == 1 && lane == 0) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_h);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_dep_wait();  // barriers and TMEM are set up; now the inputs
    const uint32_t tmem = tmem_slot;
    const int total = p.pass_tiles * p.n_tok_tiles * p.k_splits;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t issued = 0, s = 0, ph = 1;  // the first pass finds every stage free
            bool ok = true;
            for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
                const Item item = decode(p, w);
                const int kb0 = item.ks * p.kb_per_split;
                const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                const int wrow = item.wt * kGemmTileW, hrow = item.nt * p.bn;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&empty_bar[s], ph, &abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    uint8_t *ws = w_smem + s * kWStageBytes;
                    uint8_t *hs = h_smem + s * h_stage;
                    const int k0 = kb * kGemmStageK;  // boxes past `hidden` read zeros
                    mbar_arrive_expect_tx(&full_bar[s], kWStageBytes + h_stage);
                    tma_load_2d(ws, &tm_w, &full_bar[s], k0, wrow);
                    tma_load_2d(ws + kWTileBytes, &tm_w, &full_bar[s], k0 + kGemmTileK, wrow);
                    tma_load_2d(hs, &tm_h, &full_bar[s], k0, hrow);
                    tma_load_2d(hs + h_sub, &tm_h, &full_bar[s], k0 + kGemmTileK, hrow);
                    ++issued;
                    if (++s == (uint32_t)p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // Never leave the CTA with copies still landing in its shared memory.
            drain_loads(full_bar, issued, (uint32_t)p.stages);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kGemmTileW, p.bn);
            const uint64_t wd0 = sw128_desc(smem_u32(w_smem)), hd0 = sw128_desc(smem_u32(h_smem));
            const uint32_t w_st = kWStageBytes >> 4, h_st = h_stage >> 4;  // descriptor units
            const uint32_t w_sub = kWTileBytes >> 4, h_sb = h_sub >> 4;
            uint32_t s = 0, ph = 0;
            int t = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < total; w += gridDim.x, ++t) {
                const Item item = decode(p, w);
                const int kb0 = item.ks * p.kb_per_split;
                const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                const int a = t & 1;
                if (!mbar_wait(&acc_empty[a], (((uint32_t)t >> 1) & 1u) ^ 1u, &abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)a * p.acc_cols;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full_bar[s], ph, &abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    mma_stage<false>(d_tmem, wd0 + s * w_st, hd0 + s * h_st, w_sub, h_sb, idesc,
                                     kb > kb0 ? 1u : 0u);
                    tc_commit(&empty_bar[s]);
                    if (++s == (uint32_t)p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(&acc_full[a]);
            }
            if (!ok) {
                // let the MMAs already issued finish before TMEM is released
                tc_commit(&drain_bar);
                mbar_wait_drain(&drain_bar, 0);
            }
        }
    } else {
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int row_in_tile = quarter * 32 + lane;
        EpiScratch &es = epi[warp - 2];
        int t = 0;
        for (int w = blockIdx.x; w < total; w += gridDim.x, ++t) {
            const Item item = decode(p, w);
            const int a = t & 1;
            const int m_tile = item.nt * p.bn;
            if (p.mode == kGemmFilter) {
                // the tile's thresholds, fetched while its MMAs still run
                for (int c = lane; c < 256; c += 32) {
                    const int m = m_tile + c;
                    const bool ok = c < p.bn && m < p.rows_h;
                    es.pre[c] = ok ? p.theta_pre[m] : INFINITY;
                    es.th[c] = ok ? p.theta[m] : ~0ull;
                }
                __syncwarp();
            }
            if (!mbar_wait(&acc_full[a], ((uint32_t)t >> 1) & 1u, &abort_flag, p.err)) break;
            tc_fence_after();
            const int64_t v = (int64_t)item.wt * p.unit + row_in_tile;
            const uint32_t tbase = tmem + (uint32_t)a * p.acc_cols + ((uint32_t)(quarter * 32) << 16);
            int nbuf = 0;
            for (int c0 = 0; c0 < p.bn; c0 += 32) {
                float z[32];
                tmem_ld32_wait(tbase + (uint32_t)c0, z);
                if (p.mode == kGemmFilter)
                    filter_chunk(p, z, v, m_tile + c0, c0, tbase + (uint32_t)c0, es, nbuf, lane);
                else
                    epilogue_chunk(p, z, v, row_in_tile, m_tile + c0, min(32, p.bn - c0), item, lane);
            }
            tc_fence_before();
            if (p.mode == kGemmFilter && nbuf > 0) flush_survivors(p, es, nbuf, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[a]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}


// ---------------------------------------------------------------------------
// CTA-pair variant (pilot and filter modes): the two CTAs of a cluster run
// one M = 256 MMA (tcgen05.mma.cta_group::2) over a 256-row weight unit.  Each
// CTA stages its 128 weight rows and half of the token tile, so the shared-
// memory traffic per SM for the token operand halves and more stages fit.
// The leader (rank 0) issues the MMAs; both CTAs' TMA loads complete on the
// leader's full barrier; the commits multicast to both CTAs' empty and
// accumulator-full barriers; both CTAs' epilogues (each reading its own 128
// TMEM lanes) arrive on the leader's accumulator-empty barrier.
// ---------------------------------------------------------------------------
template <bool NV>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tm_w,
                        const __grid_constant__ CUtensorMap tm_h,
                        const __grid_constant__ CUtensorMap tm_sfw,
                        const __grid_constant__ CUtensorMap tm_sfh, const GemmParams p) {
    extern __shared__ uint8_t dsmem[];
    __shared__ uint64_t full_bar[kGemmMaxStages];
    __shared__ uint64_t empty_bar[kGemmMaxStages];
    __shared__ uint64_t acc_full[2];
    __shared__ uint64_t acc_empty[2];
    __shared__ uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~static_cast<uintptr_t>(1023));
    const int half_bn = p.bn / 2;
    const uint32_t h_sub = (uint32_t)half_bn * kGemmTileK * 2;  // one box of this CTA's half of the tokens
    const uint32_t h_stage = 2 * h_sub;
    uint8_t *w_smem = smem;
    uint8_t *h_smem = smem + (size_t)p.stages * kWStageBytes;
    EpiScratchPair *epi =
        reinterpret_cast<EpiScratchPair *>(h_smem + (size_t)p.stages * h_stage);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const uint32_t tmem_cols = NV ? 512u : 2 * p.acc_cols;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 2 * kPairEpiWarps);  // every epilogue warp of the pair
        }
        mbar_init(&drain_bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc_pair(&tmem_slot, tmem_cols);
        tmem_relinquish_pair();
    }
    if (warp == 1 && lane == 0) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_h);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers exist before anyone signals them
    tc_fence_after();
    // Barriers and TMEM are set up; now the inputs.  The filter pass follows
    // the pilot select, which lets it start while the select runs: its loads
    // and MMAs read only the weights and the tokens, complete before the pilot
    // pass (and so the select) began, so only its epilogue (thresholds in,
    // candidates out) waits for the select.  (Letting the select, and so the
    // filter, start during the pilot pass was slower: the early filter CTAs
    // took bandwidth from the pilot.)
    if (p.mode != kGemmFilter || warp >= 2) grid_dep_wait();
    // The store modes let the next kernel be scheduled now: its CTAs take the
    // SMs this grid leaves idle (one CTA per SM here) and, as CTAs of this
    // grid exit, the rest, and they wait for this grid's results in their own
    // grid_dep_wait().
    if (p.mode == kGemmStoreRows || p.mode == kGemmStoreBf16) grid_dep_launch();
    const uint32_t tmem = tmem_slot;
    const int total = p.pass_tiles * p.n_tok_tiles * p.k_splits;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t issued = 0, s = 0, ph = 1;  // the first pass finds every stage free
            bool ok = true;
            for (int w = pair; w < total && ok; w += npairs) {
                const Item item = decode(p, w);
                const int wrow = item.wt * p.unit + (int)rank * kGemmTileW;
                const int hrow = item.nt * p.bn + (int)rank * half_bn;
                const int kb0 = item.ks * p.kb_per_split;
                const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&empty_bar[s], ph, &abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = mapa_shared(smem_u32(&full_bar[s]), 0);
                    if (leader)
                        mbar_arrive_expect_tx(&full_bar[s], 2 * (kWStageBytes + h_stage +
                                                                 (NV ? kNvSfStageBytes : 0u)));
                    uint8_t *ws = w_smem + s * kWStageBytes;
                    uint8_t *hs = h_smem + s * h_stage;
                    const int k0 = kb * 2 * p.box_k;  // boxes past `hidden` read zeros
                    tma_load_2d_pair(ws, &tm_w, fb, k0, wrow);
                    tma_load_2d_pair(ws + kWTileBytes, &tm_w, fb, k0 + p.box_k, wrow);
                    tma_load_2d_pair(hs, &tm_h, fb, k0, hrow);
                    tma_load_2d_pair(hs + h_sub, &tm_h, fb, k0 + p.box_k, hrow);
                    if (NV) {
                        // the stage's 8 scale tiles of this CTA's 128 weight rows and of
                        // the tile's tokens (rows of 256 bytes in the tensor maps)
                        uint8_t *sfs = smem + p.sf_off + (size_t)s * kNvSfStageBytes;
                        const int yw = 2 * ((item.wt * 2 + (int)rank) * p.sf_nw8 + kb * 8);
                        const int yh = 2 * (item.nt * p.sf_nw8 + kb * 8);
                        tma_load_2d_pair(sfs, &tm_sfw, fb, 0, yw);
                        tma_load_2d_pair(sfs + 4096, &tm_sfh, fb, 0, yh);
                    }
                    ++issued;
                    if (++s == (uint32_t)p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // the leader waits until the last loads of both CTAs have landed
            if (leader) drain_loads(full_bar, issued, (uint32_t)p.stages);
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            const uint32_t idesc = NV     ? idesc_nvfp4(2 * kGemmTileW, p.bn)
                                   : p.fp8 ? idesc_e4m3(2 * kGemmTileW, p.bn)
                                           : idesc_bf16(2 * kGemmTileW, p.bn);
            const uint64_t wd0 = sw128_desc(smem_u32(w_smem)), hd0 = sw128_desc(smem_u32(h_smem));
            const uint32_t w_st = kWStageBytes >> 4, h_st = h_stage >> 4;  // descriptor units
            const uint32_t w_sub = kWTileBytes >> 4, h_sb = h_sub >> 4;
            uint32_t s = 0, ph = 0;
            int t = 0;
            bool ok = true;
            for (int w = pair; w < total; w += npairs, ++t) {
                const int a = t & 1;
                if (!mbar_wait(&acc_empty[a], (((uint32_t)t >> 1) & 1u) ^ 1u, &abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)a * p.acc_cols;
                const Item item = decode(p, w);
                const int kb0 = item.ks * p.kb_per_split;
                const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full_bar[s], ph, &abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (NV) {
                        // the stage's scales into its TMEM slot, then its MMAs (in order;
                        // the slot's previous MMAs finished before this stage's loads began)
                        const uint32_t sft = tmem + kSfBase + s * kSfCols;
                        const uint32_t sfs = smem_u32(smem + p.sf_off) + s * kNvSfStageBytes;
#pragma unroll
                        for (int m = 0; m < 8; ++m) {
                            tc_cp_sf_pair(sft + 4u * (uint32_t)m, sfs + 512u * (uint32_t)m);
                            tc_cp_sf_pair(sft + 32u + 4u * (uint32_t)m,
                                          sfs + 4096u + 512u * (uint32_t)m);
                        }
                        mma_stage_nvfp4_pair(d_tmem, wd0 + s * w_st, hd0 + s * h_st, w_sub, h_sb,
                                             idesc, kb > kb0 ? 1u : 0u, sft);
                    }
                    else if (p.fp8)
                        mma_stage_f8_pair(d_tmem, wd0 + s * w_st, hd0 + s * h_st, w_sub, h_sb,
                                          idesc, kb > kb0 ? 1u : 0u);
                    else
                        mma_stage<true>(d_tmem, wd0 + s * w_st, hd0 + s * h_st, w_sub, h_sb,
                                        idesc, kb > kb0 ? 1u : 0u);
                    tc_commit_pair_mc(&empty_bar[s], 0x3);
                    if (++s == (uint32_t)p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit_pair_mc(&acc_full[a], 0x3);
            }
            if (!ok) {
                tc_commit_pair(&drain_bar);
                mbar_wait_drain(&drain_bar, 0);
            }
        }
    } else {
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int row_in_unit = (int)rank * kGemmTileW + quarter * 32 + lane;
        // the tile columns this warp takes: one half of them (the store modes
        // split any tile evenly in chunks of 32; the candidate modes keep
        // halves of kPairEpiCols, their scratch size)
        const bool store_mode = p.mode == kGemmStoreRows || p.mode == kGemmStoreBf16;
        const int half = store_mode ? (p.bn + 63) / 64 * 32 : kPairEpiCols;
        const int cb = ((warp - 2) / 4) * half;
        const int ce = min(p.bn, cb + half);
        // bf16 stores: the warp's transpose tile after the stages
        __nv_bfloat16 *bf_tile = reinterpret_cast<__nv_bfloat16 *>(
            h_smem + (size_t)p.stages * h_stage + (size_t)(warp - 2) * kBf16TileBytes);
        const bool bf_vec = (reinterpret_cast<uintptr_t>(p.out_bf16) & 15) == 0 && p.ldo % 8 == 0;
        EpiScratchPair &es = epi[warp - 2];
        const uint32_t acc_empty_leader[2] = {mapa_shared(smem_u32(&acc_empty[0]), 0),
                                              mapa_shared(smem_u32(&acc_empty[1]), 0)};
        // The candidates of one filter-style tile whose accumulator is full:
        // its tokens' thresholds, the chunks, then the buffer goes back.
        const auto load_thresholds = [&](const Item &item) {
            const int m_tile = item.nt * p.bn;
            for (int c = lane; c < kPairEpiCols; c += 32) {
                const int cc = cb + c;
                const int m = m_tile + cc;
                const bool ok = cc < p.bn && m < p.rows_h;
                es.pre[c] = ok ? __ldcg(p.theta_pre + m) : INFINITY;
                es.th[c] = ok ? __ldcg(p.theta + m) : ~0ull;
            }
            __syncwarp();
        };
        // fp8: this thread's weight-row scale; nvfp4: the weights' one scale
        const bool scaled = p.fp8 || NV;
        const auto row_scale = [&](int64_t v) {
            return p.fp8 ? (v < p.rows_w ? __ldg(p.w_scale + v) : 0.0f) : NV ? p.w_global : 1.0f;
        };
        const auto filter_tile = [&](const Item &item, int a) {
            const int m_tile = item.nt * p.bn;
            const int64_t v = (int64_t)item.wt * p.unit + row_in_unit;
            const float wsv = row_scale(v);
            const uint32_t tbase = tmem + (uint32_t)a * p.acc_cols + ((uint32_t)(quarter * 32) << 16);
            int nbuf = 0;
            for (int c0 = cb; c0 < ce; c0 += 32) {
                float z[32];
                tmem_ld32_wait(tbase + (uint32_t)c0, z);
                const float asc = scaled ? fp8_scale_chunk(p, z, m_tile + c0, wsv, lane) : 1.0f;
                filter_chunk(p, z, v, m_tile + c0, c0 - cb, tbase + (uint32_t)c0, es, nbuf, lane,
                             asc, wsv);
            }
            tc_fence_before();
            if (nbuf > 0) flush_survivors(p, es, nbuf, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty_leader[a]);
        };
        int t = 0;
        int w = pair;
        if (p.mode == kGemmFused) {
            // Phase A: the group maxima of this pair's pilot tiles (the first
            // in its order, at most two), whose accumulators stay in TMEM.
            int np = 0;
            bool ok = true;
            for (; w < total; w += npairs, ++t) {
                const Item item = decode(p, w);
                if (!item.pilot) break;
                const int a = t & 1;
                if (!mbar_wait(&acc_full[a], ((uint32_t)t >> 1) & 1u, &abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int64_t v = (int64_t)item.wt * p.unit + row_in_unit;
                const bool valid = v < p.rows_w && v < p.target_vocab;
                const uint32_t tbase =
                    tmem + (uint32_t)a * p.acc_cols + ((uint32_t)(quarter * 32) << 16);
                const int g = item.j * (p.unit / 32) + row_in_unit / 32;
                const float wsv = row_scale(v);
                for (int c0 = cb; c0 < ce; c0 += 32) {
                    float z[32];
                    tmem_ld32_wait(tbase + (uint32_t)c0, z);
                    if (scaled) fp8_scale_chunk(p, z, item.nt * p.bn + c0, wsv, lane);
                    group_max_chunk(p, z, valid, item.nt * p.bn + c0, min(32, p.bn - c0), g, lane);
                }
                counter_arrive(p.sync, lane);
                ++np;
            }
            // the thresholds of every row, then the pilot tiles' candidates
            ok = ok && fused_select(p, &abort_flag, lane) &&
                 counter_wait(p.sync + 1, gridDim.x * kPairEpiWarps, &abort_flag, p.err, lane);
            for (int i = 0; ok && i < np; ++i) {
                const Item item = decode(p, pair + i * npairs);
                load_thresholds(item);
                filter_tile(item, i & 1);
            }
            if (!ok) w = total;
        }
        for (; w < total; w += npairs, ++t) {
            const Item item = decode(p, w);
            const int a = t & 1;
            if (item.filter) load_thresholds(item);  // while the MMAs finish
            if (!mbar_wait(&acc_full[a], ((uint32_t)t >> 1) & 1u, &abort_flag, p.err)) break;
            tc_fence_after();
            if (item.filter) {
                filter_tile(item, a);
                continue;
            }
            const int m_tile = item.nt * p.bn;
            const int64_t v = (int64_t)item.wt * p.unit + row_in_unit;
            const float wsv = row_scale(v);
            const uint32_t tbase = tmem + (uint32_t)a * p.acc_cols + ((uint32_t)(quarter * 32) << 16);
            for (int c0 = cb; c0 < ce; c0 += 32) {
                float z[32];
                tmem_ld32_wait(tbase + (uint32_t)c0, z);
                if (scaled) fp8_scale_chunk(p, z, m_tile + c0, wsv, lane);
                if (p.mode == kGemmStoreBf16)
                    store_bf16_chunk(p, z, v - lane, m_tile + c0, min(32, p.bn - c0), bf_vec, bf_tile,
                                     lane);
                else
                    epilogue_chunk(p, z, v, row_in_unit, m_tile + c0, min(32, p.bn - c0), item, lane);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty_leader[a]);
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, tmem_cols);
    }
}

// Per-device caches; several host threads may fill them at once (the guarded
// calls are idempotent).
std::atomic<int> g_smem_set[64];
std::atomic<int> g_fused_pairs[2][64];  // [nvfp4][device]; 0: not yet asked; -1: none

dflash2_status set_gemm_attrs(const DeviceInfo &di) {
    if (di.device < 0 || di.device >= 64) return DFLASH2_ERR_CUDA;
    if (g_smem_set[di.device]) return DFLASH2_OK;
    if (cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kGemmSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_tc_pair_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kGemmSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_tc_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kGemmSmemBytes) != cudaSuccess) {
        cudaGetLastError();
        return DFLASH2_ERR_CUDA;
    }
    g_smem_set[di.device] = 1;
    return DFLASH2_OK;
}

// CTA pairs of the pair kernel (nv: its nvfp4 form) the device holds at once
// (its full shared memory, so one CTA per SM), or 0.
int fused_pairs(const DeviceInfo &di, bool nv = false) {
    if (di.device < 0 || di.device >= 64) return 0;
    std::atomic<int> &slot = g_fused_pairs[nv ? 1 : 0][di.device];
    if (slot == 0) {
        int n = 0;
        if (set_gemm_attrs(di) == DFLASH2_OK) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(di.sm_count / 2 * 2));
            cfg.blockDim = dim3(kPairThreads);
            cfg.dynamicSmemBytes = kGemmSmemBytes;
            const cudaError_t e =
                nv ? cudaOccupancyMaxActiveClusters(&n, gemm_tc_pair_kernel<true>, &cfg)
                   : cudaOccupancyMaxActiveClusters(&n, gemm_tc_pair_kernel<false>, &cfg);
            if (e != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
        }
        slot = n > 0 ? n : -1;
    }
    const int n = slot;
    return n > 0 ? n : 0;
}

}  // namespace

int fused_pair_count(const DeviceInfo &di, bool nv) { return fused_pairs(di, nv); }
int fused_epilogue_warps(const DeviceInfo &di, bool nv) {
    return fused_pairs(di, nv) * 2 * kPairEpiWarps;
}

dflash2_status launch_gemm_tc(const DeviceInfo &di, const void *w, const void *h, GemmParams p,
                              cudaStream_t st, bool pair) {
    if (p.bn < 16 || p.bn > 256 || p.bn % 16 != 0 || p.k_splits < 1) return DFLASH2_ERR_INVALID_ARG;
    if (p.rows_h <= 0 || p.rows_w <= 0 || p.hidden <= 0) return DFLASH2_OK;
    if (p.mode == kGemmStore) pair = false;  // the projection keeps one CTA per tile
    if (pair && di.sm_count < 2) return DFLASH2_ERR_UNSUPPORTED_DEVICE;  // the caller's layout assumes pairs
    if (p.fp8 && (!pair || p.hidden % 16 != 0)) return DFLASH2_ERR_INVALID_ARG;
    const bool nv = p.nvfp4 != 0;
    if (nv && (!pair || p.fp8 || p.bn > 128 || p.hidden % 64 != 0 || p.n_sf != p.hidden / 16 ||
               p.sf_nw8 != nvfp4_tile_cells(p.hidden) || !p.sfw || !p.sfh ||
               !aligned16(p.sfw) || !aligned16(p.sfh) ||
               (p.mode != kGemmPilot && p.mode != kGemmFilter && p.mode != kGemmFused)))
        return DFLASH2_ERR_INVALID_ARG;
    // The TMA boxes, the stages and their counts run over bytes of codes for
    // 8-bit and 4-bit operands: one 128-byte row holds 64 bf16, 128 E4M3 codes
    // or 256 E2M1 codes.
    const int64_t kdim = nv ? p.hidden / 2 : p.hidden;
    p.unit = pair ? 2 * kGemmTileW : kGemmTileW;
    p.n_tok_tiles = (p.rows_h + p.bn - 1) / p.bn;
    p.box_k = (p.fp8 || nv) ? 2 * kGemmTileK : kGemmTileK;
    p.num_kb = (int32_t)((kdim + 2 * p.box_k - 1) / (2 * p.box_k));
    p.kb_per_split = (p.num_kb + p.k_splits - 1) / p.k_splits;
    p.k_splits = (p.num_kb + p.kb_per_split - 1) / p.kb_per_split;  // every split gets >= 1 block
    p.n_wtiles = (p.rows_w + p.unit - 1) / p.unit;
    pilot_layout(p.n_wtiles, &p.n_pilot, &p.pilot_stride, p.unit);
    if (p.mode == kGemmPilot)
        p.pass_tiles = p.n_pilot;
    else if (p.mode == kGemmFilter)
        p.pass_tiles = p.n_wtiles - p.n_pilot;
    else
        p.pass_tiles = p.n_wtiles;
    if (p.pass_tiles <= 0) return DFLASH2_OK;
    if (p.mode != kGemmStore && p.mode != kGemmStoreRows) {
        p.k_splits = 1;
        p.kb_per_split = p.num_kb;
    }
    if (p.mode == kGemmStoreRows && (!pair || p.fp8 || p.ldo % 4 != 0)) return DFLASH2_ERR_INVALID_ARG;
    // Work order: the pairs take consecutive items, token tiles fastest, so a
    // weight unit is read from DRAM once while every token tile passes over it
    // from L2.  When the token tiles' rows exceed what the L2 keeps beside the
    // weight units in flight, they go in groups, each group over the whole
    // pass: the weights are read once per group, the tokens once.  (The fused
    // mode keeps one group: its pilot items come first.)
    p.tok_group = p.n_tok_tiles;
    if (p.mode != kGemmFused) {
        const double tile_bytes = (double)p.bn * (double)kdim * ((p.fp8 || nv) ? 1.0 : 2.0);
        const int64_t groups = (int64_t)((p.n_tok_tiles * tile_bytes + kTokGroupBytes - 1) / kTokGroupBytes);
        if (groups > 1) p.tok_group = (int32_t)((p.n_tok_tiles + groups - 1) / groups);
    }
    uint32_t acc = 32;
    while (acc < (uint32_t)p.bn) acc <<= 1;
    p.acc_cols = acc;
    const uint32_t h_rows = pair ? (uint32_t)p.bn / 2 : (uint32_t)p.bn;
    const uint32_t stage_bytes = kWStageBytes + h_rows * kGemmStageK * 2;  // same bytes for fp8
    const bool fused = p.mode == kGemmFused;
    if (fused && !pair) return DFLASH2_ERR_INVALID_ARG;
    const size_t epi_bytes = p.mode == kGemmFilter || fused
                                 ? (pair ? kPairEpiWarps * sizeof(EpiScratchPair)
                                         : 4 * sizeof(EpiScratch))
                             : p.mode == kGemmStoreBf16 && pair ? (size_t)kPairEpiWarps * kBf16TileBytes
                                                                 : 0;
    int stages = (int)((kGemmSmemBytes - 1024 - epi_bytes) / stage_bytes);
    if (stages > kGemmMaxStages) stages = kGemmMaxStages;
    if (nv) {
        // the TMEM scale columns hold kNvStages; each stage brings its scales
        stages = (int)((kGemmSmemBytes - 1024 - epi_bytes) / (stage_bytes + kNvSfStageBytes));
        if (stages < kNvStages) return DFLASH2_ERR_INVALID_ARG;
        stages = kNvStages;
    }
    if (stages < 2) return DFLASH2_ERR_INVALID_ARG;  // bn <= 256 always leaves room for two
    p.stages = stages;
    p.sf_off = (int32_t)((size_t)stages * stage_bytes + epi_bytes);  // after the epilogue scratch
    const size_t smem = (size_t)stages * stage_bytes + epi_bytes +
                        (nv ? (size_t)stages * kNvSfStageBytes : 0) + 1024;

    CUtensorMap tm_w, tm_h;
    const uint32_t eb = (p.fp8 || nv) ? 1 : 2;
    dflash2_status s =
        encode_tmap_2d(&tm_w, w, (uint64_t)p.rows_w, (uint64_t)kdim, kGemmTileW, eb);
    if (s != DFLASH2_OK) return s;
    s = encode_tmap_2d(&tm_h, h, (uint64_t)p.rows_h, (uint64_t)kdim, h_rows, eb);
    if (s != DFLASH2_OK) return s;
    CUtensorMap tm_sfw = tm_w, tm_sfh = tm_h;
    if (nv) {
        // the scale tiles as rows of 256 bytes; a stage's 8 tiles are 16 rows
        const uint64_t rw = nvfp4_tiles_bytes(p.rows_w, p.hidden, kGemmTileW) / 256;
        const uint64_t rh = nvfp4_tiles_bytes(p.rows_h, p.hidden, p.bn) / 256;
        s = encode_tmap_bytes_2d(&tm_sfw, p.sfw, rw, 256, 256, 16);
        if (s != DFLASH2_OK) return s;
        s = encode_tmap_bytes_2d(&tm_sfh, p.sfh, rh, 256, 256, 16);
        if (s != DFLASH2_OK) return s;
    }

    s = set_gemm_attrs(di);
    if (s != DFLASH2_OK) return s;
    const int64_t total = (int64_t)p.pass_tiles * p.n_tok_tiles * p.k_splits;
    if (fused) {
        // every CTA resident at once (its warps wait on one another): a
        // cooperative launch of at most the pairs the device holds together
        const int64_t pairs_max = fused_pairs(di, nv);
        if (pairs_max < 1) return DFLASH2_ERR_UNSUPPORTED_DEVICE;
        const int pairs = (int)(total < pairs_max ? total : pairs_max);
        // a pair keeps its pilot accumulators until the select: two at most
        if ((int64_t)p.n_pilot * p.n_tok_tiles > 2LL * pairs) return DFLASH2_ERR_INVALID_ARG;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(2 * pairs));
        cfg.blockDim = dim3(kPairThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeCooperative;
        attr[1].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        if (nv)
            cudaLaunchKernelEx(&cfg, gemm_tc_pair_kernel<true>, tm_w, tm_h, tm_sfw, tm_sfh, p);
        else
            cudaLaunchKernelEx(&cfg, gemm_tc_pair_kernel<false>, tm_w, tm_h, tm_w, tm_h, p);
        return launch_status();
    }
    if (pair) {
        const int64_t pairs_max = di.sm_count / 2;
        const int pairs = (int)(total < pairs_max ? total : pairs_max);
        if (nv)
            launch_k(gemm_tc_pair_kernel<true>, 2 * pairs, kPairThreads, smem, st, tm_w, tm_h,
                     tm_sfw, tm_sfh, p);
        else
            launch_k(gemm_tc_pair_kernel<false>, 2 * pairs, kPairThreads, smem, st, tm_w, tm_h,
                     tm_w, tm_h, p);
    } else {
        const int grid = (int)(total < di.sm_count ? total : di.sm_count);
        launch_k(gemm_tc_kernel, grid, 192, smem, st, tm_w, tm_h, p);
    }
    return launch_status();
}

}  // namespace dflash2
