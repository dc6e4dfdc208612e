// Internal launch interfaces shared between the translation units.
#pragma once

#include "common.cuh"

namespace dflash2 {

// ---- tcgen05 GEMM (gemm_tc.cu) ----------------------------------------------
// C[m, v] = sum_j h[m, j] * w[v, j] with w and h row-major bf16 (K-major).
// The weight rows form the MMA's M side in tiles of 128 rows; the h rows
// (tokens) form the N side in tiles of `bn` rows.
enum GemmMode : int32_t {
    kGemmStore = 0,   // write fp32 C (split-K partials) to out
    kGemmPilot = 1,   // write the transformed, masked u of the pilot tiles to out
    kGemmFilter = 2,  // append (u, id) keys that reach the row's threshold
    kGemmStoreBf16 = 3,  // write C rounded to bf16 (nearest-even) to out_bf16, no split
    // pilot, select and filter in one cooperative launch: the pilot tiles come
    // first (at most two per CTA pair) and their epilogues write group maxima,
    // the epilogue warps then derive every row's threshold while the MMAs run
    // on, and every tile's candidates (the pilot tiles' from the accumulators
    // they kept) are taken against the thresholds
    kGemmFused = 4,
    // fp32 C row by row, split over hidden: out[ks * split_stride + v * ldo + m]
    // for weight row v and token m (CTA pairs).  The selector projection of a
    // large batch runs with the tokens as the weight side (256 per pair), so
    // each CTA streams 128 token rows and stages half of the small projection
    // matrix.
    kGemmStoreRows = 5,
};

constexpr int kGemmTileW = 128;  // weight rows per tile (MMA M)
constexpr int kGemmTileK = 64;   // hidden elements per TMA box (one 128-byte swizzle row)
constexpr int kGemmStageK = 128; // hidden elements per pipeline stage (two boxes per operand)
constexpr int kGemmMaxStages = 8;
constexpr int kPilotTiles = 64;  // pilot weight tiles (of 128 rows) sampled across the vocab, at most

struct GemmParams {
    // problem
    int32_t rows_w;  // weight rows (draft vocab, or selector rank)
    int32_t rows_h;  // token rows
    int32_t hidden;
    int32_t mode;
    // tiling (filled by launch_gemm_tc except bn / k_splits)
    int32_t bn;       // token tile, multiple of 16 in [16, 256]
    int32_t k_splits; // store mode: number of hidden splits (>= 1)
    int32_t n_tok_tiles;
    int32_t num_kb;       // pipeline stages (kGemmStageK hidden elements each) over hidden
    int32_t kb_per_split;
    int32_t n_wtiles;
    int32_t n_pilot;
    int32_t pilot_stride;
    int32_t pass_tiles;
    int32_t unit;     // weight rows per work unit: 128 (one CTA) or 256 (a CTA pair)
    int32_t tok_group; // token tiles per group of the work order (filled by launch_gemm_tc)
    int32_t stages;
    uint32_t acc_cols;
    // epilogue
    int64_t target_vocab;
    float mult;
    float cap;
    float *out;            // store: [k_splits][rows_h][ldo]; store-rows: [k_splits][rows_w][ldo]; pilot: [rows_h][ldo]
    __nv_bfloat16 *out_bf16;  // store-bf16: [rows_h][ldo]
    int64_t ldo;
    int64_t split_stride;
    const uint64_t *theta; // filter: per-row threshold key
    const float *theta_pre; // filter: per-row bound on mult * z below which u cannot reach theta
    uint32_t *cnt;         // filter: per-row candidate count
    uint64_t *cand;        // filter: [rows_h][cand_cap] keys
    int32_t cand_cap;
    int32_t *err;
    // fused: the pilot tiles' group maxima (order bits of the largest logit
    // of each 32 consecutive vocab rows of a pilot unit) [rows_h][ld_pmax];
    // top_k; two grid counters (pilot warps done, select warps done), zero at
    // launch
    uint32_t *pmax;
    int64_t ld_pmax;
    int32_t top_k;
    uint32_t *sync;
    // fp8: E4M3 operands (kind::f8f6f4; a box covers 128 hidden elements, a
    // stage 256); C = acc * (a_scale[m] * w_scale[v]) before the epilogue
    int32_t fp8;
    int32_t box_k;  // hidden elements per TMA box (filled by launch_gemm_tc)
    const float *a_scale;
    const float *w_scale;
    // nvfp4: E2M1 codes, two per byte (kind::mxf4nvf4 with one E4M3 scale per
    // 16 elements, the scales in TMEM; CTA pairs, bn <= 128).  hidden counts
    // elements; the codes rows are hidden / 2 bytes.  sfw [rows_w][n_sf] and
    // sfh [rows_h][n_sf] hold the scales (n_sf = hidden / 16, a multiple of
    // 4); C = acc * (a_scale[m] * w_global) before the epilogue.
    int32_t nvfp4;
    int32_t n_sf;
    const uint8_t *sfw;  // weight scales in scale tiles of 128 rows (nvfp4_tiles_bytes)
    const uint8_t *sfh;  // token scales in scale tiles of bn rows
    float w_global;
    int32_t sf_nw8;  // 4-scale cells per row in the scale tiles (a multiple of 8)
    int32_t sf_off;  // the scale stages' offset in dynamic shared memory (filled by launch_gemm_tc)
};

// NVFP4 scale tiles: the layout in which the block-scaled GEMM copies a
// stage's scales (TMA) and hands them to TMEM (tcgen05.cp 32x128b.warpx4).
// Rows go in blocks of `block_rows` (<= 128); a row's scales in cells of 4
// (one cell per MMA of 64 elements), nw8 = cells per row rounded up to a
// multiple of 8.  Tile (rb, w) is 512 bytes at (rb * nw8 + w) * 512: row
// rb * block_rows + l + 32 j (l < 32, j < 4) has its cell w at byte l * 16 +
// j * 4.  Cells of rows past the end or past block_rows, and past the row's
// scales, are zero.
inline int32_t nvfp4_tile_cells(int32_t hidden) { return (hidden / 64 + 7) / 8 * 8; }
inline size_t nvfp4_tiles_bytes(int64_t rows, int32_t hidden, int32_t block_rows) {
    return (size_t)((rows + block_rows - 1) / block_rows) * nvfp4_tile_cells(hidden) * 512;
}
dflash2_status launch_nvfp4_tile_scales(const uint8_t *scales, int64_t rows, int32_t hidden,
                                        int32_t block_rows, uint8_t *tiles, cudaStream_t st);

// Pilot tiling of a weight matrix with n_wtiles units of unit_rows rows:
// n_pilot units spaced pilot_stride apart, from unit 0.  A larger pilot gives
// a tighter threshold (fewer filter survivors, about K * vocab / pilot rows
// per token) at the cost of a larger one-wave pilot GEMM; measured on the
// bf16 workloads, about a sixteenth of the vocab, between 8 units and 8192
// rows, balances the two (every unit when the vocab has fewer than 8).
inline void pilot_layout(int64_t n_wtiles, int32_t *n_pilot, int32_t *stride, int unit_rows = 128) {
    const int64_t max_units = (int64_t)kPilotTiles * kGemmTileW / unit_rows;
    int64_t np = (n_wtiles + 15) / 16;
    if (np < 8) np = 8;
    if (np > max_units) np = max_units;
    if (np > n_wtiles) np = n_wtiles;
    if (np < 1) np = 1;
    *n_pilot = (int32_t)np;
    *stride = (int32_t)(n_wtiles / np);
}

// pair: run the pilot / filter / fused modes on CTA pairs (2-CTA MMA, 256-row units).
dflash2_status launch_gemm_tc(const DeviceInfo &di, const void *w, const void *h, GemmParams p,
                              cudaStream_t st, bool pair = false);

// Per-row E4M3 quantization (quant.cu): q [rows, cols] codes, d [rows] scales.
dflash2_status launch_quant_rows_e4m3(const void *x, int32_t dtype, int64_t rows, int32_t cols,
                                      uint8_t *q, float *d, cudaStream_t st);
// Per-row NVFP4 quantization (quant.cu): codes [rows, cols / 2] (element 2i in
// the low nibble), E4M3 block scales [rows, cols / 16], fp32 second-level
// scales g [rows]; cols a multiple of 16.
dflash2_status launch_quant_rows_nvfp4(const void *x, int32_t dtype, int64_t rows, int32_t cols,
                                       uint8_t *codes, uint8_t *scales, float *g, cudaStream_t st);

// CTA pairs of one fused launch (every CTA resident at once) and their
// epilogue warps, or 0 when the device cannot hold such a launch.  Host-side,
// cached per device.
int fused_pair_count(const DeviceInfo &di, bool nvfp4 = false);
int fused_epilogue_warps(const DeviceInfo &di, bool nvfp4 = false);

}  // namespace dflash2
