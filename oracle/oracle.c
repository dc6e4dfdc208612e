/*
 * Plain, slow CPU oracle for the DFlash2 draft-proposal hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that tests, the smoke check and the benchmark's
 * CPU-baseline leg can compare the CUDA library against an obviously correct
 * restatement of the method.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * Conventions
 *   - Every floating-point accumulation runs in double from the exact input
 *     values (bf16 and fp32 inputs widen exactly to double) and is rounded once
 *     at the output.
 *   - Where floating point decides an integer (top-K membership, the walk's
 *     argmax and inverse-CDF draw) the decision is taken in fp32, the precision
 *     of the sglang Triton walk ("[Spec] DFlash2: local convolution + candidate
 *     selector", _selector_walk_kernel, which loads the scores as float32).
 *   - dtype 0 = fp32 (float arrays), dtype 1 = bf16 (uint16 bit patterns).
 *   - Parallelism is OpenMP over independent rows only; it cannot change a
 *     result because no reduction crosses threads.
 *
 * Every function below is pinned by the CPU tests (tests/test_oracle_*.py)
 * against brute force, closed forms, invariants or library special cases.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* ---- element access ---------------------------------------------------- */

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *p, int64_t i, int dtype)
{
    if (dtype == ORACLE_BF16)
        return bf16_bits_to_double(((const uint16_t *)p)[i]);
    return (double)((const float *)p)[i];
}

/*
 * Round a double to the nearest bf16 (ties to even) in ONE step.  Going
 * through float first would round twice.  The value is scaled by a power of
 * two so that it carries exactly 8 significant bits before the binary point;
 * nearbyint() then rounds half-to-even in the default rounding mode.  Power of
 * two scaling is exact, so the only rounding is the one in nearbyint().
 */
uint16_t oracle_round_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int e;
    frexp(a, &e); /* a = f * 2^e with f in [0.5, 1) */
    int sh = 8 - e; /* a * 2^sh lies in [128, 256) */
    if (e - 8 < -133)
        sh = 133; /* below the normal range bf16 steps by 2^-133 */
    double q = nearbyint(ldexp(a, sh));
    double r = ldexp(q, -sh);
    const double bf16_max = 3.3895313892515355e38; /* (2 - 2^-7) * 2^127 */
    if (r > bf16_max)
        return sign | 0x7F80;
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return sign | (uint16_t)(bits >> 16);
}

static void store_elem(void *p, int64_t i, double v, int dtype)
{
    if (dtype == ORACLE_BF16)
        ((uint16_t *)p)[i] = oracle_round_bf16(v);
    else
        ((float *)p)[i] = (float)v; /* one round-to-nearest-even */
}

/* ---- (1) block-causal grouped dynamic depthwise conv --------------------
 * sglang "[Spec] DFlash2: local convolution + candidate selector",
 * _grouped_conv: hidden is split into (groups, group_size); the coefficient of
 * tap t for channel c of token i is base[t, c] + delta[i, t, c / group_size];
 * tap t reads the token t rows earlier and is zeroed unless the in-block
 * position (i mod block_size) is at least t.
 *
 *   out[i, c] = sum_{t < taps, pos(i) >= t} (base[t,c] + delta[i,t,c/gs]) * x[i-t, c]
 *
 * x, out: [n, hidden]; base: [taps, hidden]; delta row i starts at
 * i * delta_row_stride and holds [taps, hidden / gs].
 */
int oracle_conv(const void *x, const void *base, const void *delta,
                int64_t delta_row_stride, void *out, int64_t n, int32_t hidden,
                int32_t group_size, int32_t taps, int32_t block_size,
                int32_t dtype)
{
    if (n < 0 || hidden <= 0 || group_size <= 0 || hidden % group_size ||
        taps <= 0 || block_size <= 0)
        return 1;
    const int64_t groups = hidden / group_size;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        const int64_t pos = i % block_size;
        for (int32_t c = 0; c < hidden; ++c) {
            double acc = 0.0;
            for (int32_t t = 0; t < taps; ++t) {
                if (pos < t)
                    continue; /* this tap would cross the block start */
                double coef =
                    load_elem(base, (int64_t)t * hidden + c, dtype) +
                    load_elem(delta,
                              i * delta_row_stride + (int64_t)t * groups +
                                  c / group_size,
                              dtype);
                acc += coef * load_elem(x, (i - t) * hidden + c, dtype);
            }
            store_elem(out, i * hidden + c, acc, dtype);
        }
    }
    return 0;
}

/* ---- (2)+(3) unary logits ------------------------------------------------
 * z[m, v] = sum_j h[m, j] * lm_head[v, j]   (lm_head in nn.Linear layout)
 * u = cap * tanh(mult * z / cap) when cap > 0, else mult * z
 *   (output_multiplier / final_logit_softcapping of DFlashDraftConfig in the
 *   DFlash2 PR, which names the two fields but prints no formula; this is
 *   the soft-capping reading used throughout)
 * u = -inf for padded vocab rows v >= target_vocab: the vLLM DSpark
 *   padded-vocab review asks that [target_vocab, draft_vocab) be masked
 *   before any top-k.
 * Rows listed in `rows` (all rows when rows == NULL) are evaluated; u_out is
 * [n_sel, draft_vocab] doubles.
 */
void oracle_unary_rows(const void *h, const void *lm_head, const int64_t *rows,
                       int64_t n_sel, int32_t hidden, int64_t draft_vocab,
                       int64_t target_vocab, double mult, double cap,
                       int32_t dtype, double *u_out)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < n_sel; ++r) {
        for (int64_t v = 0; v < draft_vocab; ++v) {
            const int64_t m = rows ? rows[r] : r;
            double u;
            if (v >= target_vocab) {
                u = -INFINITY;
            } else {
                double z = 0.0;
                for (int32_t j = 0; j < hidden; ++j)
                    z += load_elem(h, m * hidden + j, dtype) *
                         load_elem(lm_head, v * hidden + j, dtype);
                u = cap > 0.0 ? cap * tanh(mult * z / cap) : mult * z;
            }
            u_out[r * draft_vocab + v] = u;
        }
    }
}

/* ---- (4) top-K ------------------------------------------------------------
 * Per row, the K best (u, id) pairs with u taken in fp32: a full sort by u
 * descending, equal u by smaller vocab id first, then the first K.  The order
 * matters downstream: the walk's greedy tie rule picks the lowest candidate
 * index and its inverse-CDF scans candidates in index order.
 */
typedef struct {
    float u;
    int64_t id;
} oracle_pair;

static int pair_order(const void *pa, const void *pb)
{
    const oracle_pair *a = (const oracle_pair *)pa;
    const oracle_pair *b = (const oracle_pair *)pb;
    if (a->u > b->u)
        return -1;
    if (a->u < b->u)
        return 1;
    return (a->id > b->id) - (a->id < b->id);
}

int oracle_topk(const double *u, int64_t n_rows, int64_t draft_vocab,
                int32_t k, int64_t *ids, float *vals)
{
    if (k <= 0 || k > draft_vocab)
        return 1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        oracle_pair *p =
            (oracle_pair *)malloc((size_t)draft_vocab * sizeof(oracle_pair));
        if (!p) {
#pragma omp atomic write
            bad = 1;
            continue;
        }
        for (int64_t v = 0; v < draft_vocab; ++v) {
            p[v].u = (float)u[r * draft_vocab + v];
            p[v].id = v;
        }
        qsort(p, (size_t)draft_vocab, sizeof(oracle_pair), pair_order);
        for (int32_t i = 0; i < k; ++i) {
            ids[r * k + i] = p[i].id;
            vals[r * k + i] = p[i].u;
        }
        free(p);
    }
    return bad;
}

/* ---- (5) selector projection -----------------------------------------------
 * project(h) of the selector edge formula, read as an nn.Linear(hidden, rank)
 * without bias: g[m, j] = sum_i h[m, i] * proj[j, i], proj stored [rank, hidden].
 */
void oracle_project(const void *h, const void *proj, int64_t rows,
                    int32_t hidden, int32_t rank, int32_t dtype, double *g)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < rows; ++m) {
        for (int32_t j = 0; j < rank; ++j) {
            double acc = 0.0;
            for (int32_t i = 0; i < hidden; ++i)
                acc += load_elem(h, m * hidden + i, dtype) *
                       load_elem(proj, (int64_t)j * hidden + i, dtype);
            g[m * rank + j] = acc;
        }
    }
}

/* ---- (6) selector lattice ------------------------------------------------
 * The sglang DFlash2 PR body scores adjacent transitions as
 *   edge(p -> c) = < A[p] (elementwise *) project(h), B[c] > + unary[c].
 * scores[b, s, kp, kc] is the edge from predecessor kp to candidate kc of
 * slot s, matching the [batch, slots, K, K] layout the Triton walk indexes
 * ((row*slots + slot)*K + previous)*K + k.  Slot 0's predecessor is the
 * verified anchor token, so every kp row of slot 0 holds the anchor's edges.
 * A and B are [table_rows, rank] indexed by draft ids.  An id outside
 * [0, table_rows) counts as an error and contributes a zero table row.
 * Returns the number of out-of-range ids met.
 */
int64_t oracle_lattice(const double *g, const void *A, const void *B,
                       int64_t table_rows, const int64_t *anchors,
                       const int64_t *cand, const float *cand_u, int32_t batch,
                       int32_t slots, int32_t rank, int32_t k, int32_t dtype,
                       float *scores)
{
    int64_t errors = 0;
#pragma omp parallel for collapse(2) schedule(static) reduction(+ : errors)
    for (int32_t b = 0; b < batch; ++b) {
        for (int32_t s = 0; s < slots; ++s) {
            const int64_t bs_row = (int64_t)b * slots + s;
            for (int32_t kp = 0; kp < k; ++kp) {
                int64_t p = s == 0 ? anchors[b] : cand[(bs_row - 1) * k + kp];
                int p_ok = p >= 0 && p < table_rows;
                if (!p_ok && (s > 0 || kp == 0))
                    errors += 1;
                for (int32_t kc = 0; kc < k; ++kc) {
                    int64_t c = cand[bs_row * k + kc];
                    int c_ok = c >= 0 && c < table_rows;
                    if (!c_ok && kp == 0)
                        errors += 1;
                    double acc = 0.0;
                    if (p_ok && c_ok) {
                        for (int32_t j = 0; j < rank; ++j)
                            acc += load_elem(A, p * rank + j, dtype) *
                                   g[bs_row * rank + j] *
                                   load_elem(B, c * rank + j, dtype);
                    }
                    acc += (double)cand_u[bs_row * k + kc];
                    scores[(bs_row * k + kp) * k + kc] = (float)acc;
                }
            }
        }
    }
    return errors;
}

/* ---- (7) selector walk -------------------------------------------------------
 * Follows the sglang _selector_walk_kernel step by step, in fp32:
 *   previous = 0 (the anchor row) at slot 0;
 *   scores = lattice row `previous` of this slot;
 *   greedy row:  index = smallest k with scores[k] == max(scores); q = one-hot;
 *   sampled row: scaled = scores / T; e = exp(scaled - max(scaled));
 *                p = e / sum(e); cdf = cumulative sum of p;
 *                index = #{k : uniform >= cdf[k]}, capped at K - 1; q = p;
 *   token = candidate[index]; previous = index.
 * T is first clamped to at least 1e-5 (stage_sampling_params of the same PR).
 * The sums run left to right in fp32; exp is taken in double and rounded to
 * fp32 once (a correctly rounded fp32 exp for all practical purposes).
 * chosen (nullable) receives the candidate index per (b, s).
 */
void oracle_walk(const float *scores, const int64_t *cand, const float *uniforms,
                 const float *temperatures, const uint8_t *greedy, int32_t batch,
                 int32_t slots, int32_t k, int64_t *tokens, float *q,
                 int32_t *chosen)
{
#pragma omp parallel for schedule(static)
    for (int32_t b = 0; b < batch; ++b) {
        float t = temperatures[b];
        if (!(t >= 1e-5f))
            t = 1e-5f;
        const int is_greedy = greedy[b] != 0;
        float *scaled = (float *)malloc((size_t)k * sizeof(float));
        int32_t previous = 0;
        for (int32_t s = 0; s < slots; ++s) {
            const int64_t bs_row = (int64_t)b * slots + s;
            const float *row = scores + (bs_row * k + previous) * k;
            float *qr = q + bs_row * k;
            int32_t index = 0;
            if (is_greedy) {
                float best = row[0];
                for (int32_t i = 1; i < k; ++i)
                    if (row[i] > best)
                        best = row[i];
                index = k;
                for (int32_t i = 0; i < k; ++i)
                    if (row[i] == best && i < index)
                        index = i;
                for (int32_t i = 0; i < k; ++i)
                    qr[i] = i == index ? 1.0f : 0.0f;
            } else {
                float mx = -INFINITY;
                for (int32_t i = 0; i < k; ++i) {
                    scaled[i] = row[i] / t;
                    if (scaled[i] > mx)
                        mx = scaled[i];
                }
                float total = 0.0f;
                for (int32_t i = 0; i < k; ++i) {
                    float d = scaled[i] - mx;
                    qr[i] = (float)exp((double)d);
                    total += qr[i];
                }
                for (int32_t i = 0; i < k; ++i)
                    qr[i] = qr[i] / total;
                const float uni = uniforms[bs_row];
                float cdf = 0.0f;
                index = 0;
                for (int32_t i = 0; i < k; ++i) {
                    cdf += qr[i];
                    if (uni >= cdf)
                        index += 1;
                }
                if (index > k - 1)
                    index = k - 1;
            }
            tokens[bs_row] = cand[bs_row * k + index];
            if (chosen)
                chosen[bs_row] = index;
            previous = index;
        }
        free(scaled);
    }
}

/* ---- (8) draft-to-target id remap -----------------------------------------
 * vLLM Qwen3DSparkForCausalLM.map_draft_to_target: d2t holds OFFSETS, so the
 * target id is draft + d2t[draft]; with no table (draft vocab >= target vocab,
 * the padded-vocab case) the map is the identity.  Ids that are not valid
 * draft ids, or that land outside [0, target_vocab), count as errors and are
 * written as 0.  Returns the number of errors.
 */
int64_t oracle_d2t(const int64_t *draft_ids, const int64_t *d2t, int64_t n,
                   int64_t draft_vocab, int64_t target_vocab, int64_t *out)
{
    int64_t errors = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t d = draft_ids[i];
        if (d < 0 || d >= draft_vocab) {
            out[i] = 0;
            errors += 1;
            continue;
        }
        int64_t t = d2t ? d + d2t[d] : d;
        if (t < 0 || t >= target_vocab) {
            out[i] = 0;
            errors += 1;
            continue;
        }
        out[i] = t;
    }
    return errors;
}

/* ---- (9) counter-based uniforms --------------------------------------------
 * The sglang DFlash2 sampler (_SelectorDraftSampler) draws the walk's
 * uniforms inside the captured graph from a Philox generator whose state
 * advances at every replay.  The generator here is Philox4x64 with 10 rounds
 * as defined by Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3" (SC 2011): a 4-word counter and a 2-word key; a round
 * multiplies words 0 and 2 by two fixed odd constants, the new words are
 * (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)), and the
 * key then advances by two fixed Weyl increments.
 *
 * Uniform i is word (i mod 4) of the block at counter (base + i / 4, 0, 0, 0)
 * under key (seed, 0), mapped to [0, 1) as (word >> 40) * 2^-24 (exact in
 * fp32).
 */
void oracle_philox4x64(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4])
{
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
    uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        unsigned __int128 p0 = (unsigned __int128)M0 * c0;
        unsigned __int128 p1 = (unsigned __int128)M1 * c2;
        uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
        uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
        k0 += W0;
        k1 += W1;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

void oracle_philox_uniforms(uint64_t seed, uint64_t base, int64_t n, float *out)
{
    const uint64_t key[2] = {seed, 0};
    for (int64_t i = 0; i < n; ++i) {
        const uint64_t ctr[4] = {base + (uint64_t)(i / 4), 0, 0, 0};
        uint64_t words[4];
        oracle_philox4x64(ctr, key, words);
        out[i] = (float)((double)(words[i % 4] >> 40) * 0x1p-24);
    }
}

/* ---- (10) kernel projection of the grouped conv ---------------------------
 * DFlashGroupedConv (sglang DFlash2 PR) derives the dynamic coefficients of
 * both of its convolutions from one bias-free linear map of the input,
 * nn.Linear(hidden, 2 * taps * groups), whose weight is
 * w_kp[2 * taps * groups, hidden]:
 *
 *   coef[i, r] = sum_j x[i, j] * w_kp[r, j],   r = (side * taps + t) * groups + g
 *
 * stored in the layer's dtype, as the Linear's output is.  prepare() convolves
 * the input with side 0 of coef and side 0 of base_kernel[2, taps, hidden];
 * finish() convolves the sublayer's output with side 1 of both.  Both are
 * oracle_conv with delta_row_stride = 2 * taps * groups (see oracle/__init__.py).
 */
void oracle_kernel_projection(const void *x, const void *w_kp, int64_t n, int32_t hidden,
                              int32_t out_features, int32_t dtype, void *coef)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        for (int32_t r = 0; r < out_features; ++r) {
            double acc = 0.0;
            for (int32_t j = 0; j < hidden; ++j)
                acc += load_elem(x, i * hidden + j, dtype) *
                       load_elem(w_kp, (int64_t)r * hidden + j, dtype);
            store_elem(coef, i * (int64_t)out_features + r, acc, dtype);
        }
    }
}

/* ---- (11) lossless verification of a proposed block ------------------------
 * The consumer of the walk's q.  The pages do not print it; this is the
 * standard speculative-sampling rule (Leviathan, Kalman and Matias, "Fast
 * inference from transformers via speculative decoding", 2023; Chen et al.,
 * "Accelerating large language model decoding with speculative sampling",
 * 2023).  For request b with S drafted tokens and S + 1 target positions:
 *
 *   T' = max(T_b, 1e-5) (as the walk clamps), p_s = softmax(logits[b, s, :] / T')
 *   for s = 0 .. S-1, in order:
 *     x = draft[b, s] (a target id); k = the candidate with cand[b, s, k] == x
 *     greedy row:  accept iff x == argmax_y logits[b, s, y] (smallest y on ties)
 *     sampled row: accept iff r[b, s] * q[b, s, k] < p_s(x)
 *                  (probability min(1, p_s(x) / q[b, s, k]))
 *     on the first rejection emit one token and stop:
 *       greedy:  argmax_y logits[b, s, y]
 *       sampled: from res(y) = max(0, p_s(y) - qt(y)), where qt(y) = q[b, s, k]
 *                if y = cand[b, s, k] and 0 elsewhere, by inverse CDF with
 *                u = r[b, S]: y = min { y : sum_{y' <= y} res(y') > u * sum res }
 *   if every slot is accepted, emit the bonus token from position S the same
 *   way with res = p_S (greedy: argmax).
 *
 * Arithmetic in double from the exact logits (bf16 widened); the uniforms,
 * q and T are the fp32 inputs.  Outputs: accept_len[b] = accepted drafts;
 * out_tokens[b, 0 .. S] = the accepted drafts, then the emitted token, then -1.
 * A draft that is not among its slot's candidates counts as an error and
 * leaves that request's outputs at accept_len 0 and all -1.  Returns the
 * number of errors.
 */
static int64_t argmax_row(const void *logits, int64_t off, int64_t vocab, int dtype)
{
    int64_t best = 0;
    double bv = load_elem(logits, off, dtype);
    for (int64_t y = 1; y < vocab; ++y) {
        double v = load_elem(logits, off + y, dtype);
        if (v > bv) {
            bv = v;
            best = y;
        }
    }
    return best;
}

/* p_s(y) for every y of one position, in double */
static void softmax_row(const void *logits, int64_t off, int64_t vocab, double temp, int dtype,
                        double *p)
{
    double m = -INFINITY;
    for (int64_t y = 0; y < vocab; ++y) {
        double z = load_elem(logits, off + y, dtype) / temp;
        if (z > m)
            m = z;
    }
    double sum = 0.0;
    for (int64_t y = 0; y < vocab; ++y) {
        p[y] = exp(load_elem(logits, off + y, dtype) / temp - m);
        sum += p[y];
    }
    for (int64_t y = 0; y < vocab; ++y)
        p[y] /= sum;
}

/* inverse CDF over res[0, vocab) with threshold u * total */
static int64_t inverse_cdf(const double *res, int64_t vocab, double u)
{
    double total = 0.0;
    for (int64_t y = 0; y < vocab; ++y)
        total += res[y];
    const double target = u * total;
    double c = 0.0;
    int64_t last_pos = -1;
    for (int64_t y = 0; y < vocab; ++y) {
        if (res[y] > 0.0)
            last_pos = y;
        c += res[y];
        if (c > target && res[y] > 0.0)
            return y;
    }
    return last_pos; /* only reached through rounding at the very top */
}

int64_t oracle_verify(const void *logits, const float *temperatures, const uint8_t *greedy,
                      const int64_t *draft, const int64_t *cand, const float *q,
                      const float *r, int32_t batch, int32_t slots, int32_t top_k,
                      int64_t vocab, int32_t dtype, int64_t *accept_len, int64_t *out_tokens)
{
    int64_t errors = 0;
#pragma omp parallel for schedule(dynamic) reduction(+ : errors)
    for (int32_t b = 0; b < batch; ++b) {
        int64_t *out = out_tokens + (int64_t)b * (slots + 1);
        for (int32_t s = 0; s <= slots; ++s)
            out[s] = -1;
        accept_len[b] = 0;
        const double temp = (double)(temperatures[b] > 1e-5f ? temperatures[b] : 1e-5f);
        double *p = (double *)malloc(sizeof(double) * (size_t)vocab);
        int bad = 0, done = 0;
        int32_t s = 0;
        for (; s < slots && !done; ++s) {
            const int64_t off = ((int64_t)b * (slots + 1) + s) * vocab;
            const int64_t x = draft[(int64_t)b * slots + s];
            const int64_t *cs = cand + ((int64_t)b * slots + s) * top_k;
            const float *qs = q + ((int64_t)b * slots + s) * top_k;
            int32_t k = -1;
            for (int32_t j = 0; j < top_k; ++j)
                if (cs[j] == x) {
                    k = j;
                    break;
                }
            if (k < 0 || x < 0 || x >= vocab) {
                bad = 1;
                break;
            }
            if (greedy[b]) {
                const int64_t y = argmax_row(logits, off, vocab, dtype);
                if (y == x) {
                    out[s] = x;
                    continue;
                }
                out[s] = y;
                done = 1;
                break;
            }
            softmax_row(logits, off, vocab, temp, dtype, p);
            if ((double)r[(int64_t)b * (slots + 1) + s] * (double)qs[k] < p[x]) {
                out[s] = x;
                continue;
            }
            for (int32_t j = 0; j < top_k; ++j) { /* residual: subtract q on its candidates */
                const int64_t y = cs[j];
                if (y >= 0 && y < vocab)
                    p[y] = p[y] - (double)qs[j] > 0.0 ? p[y] - (double)qs[j] : 0.0;
            }
            out[s] = inverse_cdf(p, vocab, (double)r[(int64_t)b * (slots + 1) + slots]);
            done = 1;
            break;
        }
        if (bad) {
            for (int32_t j = 0; j <= slots; ++j)
                out[j] = -1;
            errors += 1;
        } else {
            accept_len[b] = s; /* s drafts accepted when the loop stopped at slot s */
            if (!done) {       /* all accepted: the bonus token from position S */
                const int64_t off = ((int64_t)b * (slots + 1) + slots) * vocab;
                if (greedy[b]) {
                    out[slots] = argmax_row(logits, off, vocab, dtype);
                } else {
                    softmax_row(logits, off, vocab, temp, dtype, p);
                    out[slots] = inverse_cdf(p, vocab, (double)r[(int64_t)b * (slots + 1) + slots]);
                }
            }
        }
        free(p);
    }
    return errors;
}

/* ---- (10) FP8 lm_head: E4M3 codes and W8A8 logits -------------------------
 * The quantized-head path asked for beside the pages' method (sglang DFlash2
 * PR: a quantized lm_head makes the selector fall back; the vLLM DSpark
 * review's drafts ship NVFP4 heads).  Plain definitions:
 *   - E4M3 ("e4m3fn" of the OCP 8-bit floating point formats): sign bit,
 *     4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds
 *     the subnormals m * 2^-9 (m = 0..7); no infinities; codes 0x7F / 0xFF are
 *     NaN; the largest finite value is 448.  Encoding rounds to nearest, ties
 *     to the even code, and saturates at +-448.
 *   - Per-row activation quantization (W8A8 with dynamic per-token scales):
 *     amax = max_j |h[m, j]| in fp32, inv = 448 / amax and d = amax / 448 in
 *     fp32 (amax == 0: every code 0, d = 1), q[m, j] = E4M3(h[m, j] * inv)
 *     with the product rounded to fp32 first.  These decide integer codes, so
 *     they run in fp32, the precision of the kernel.
 *   - Logits: z[m, v] = d[m] * s_w[v] * sum_j dec(q_h[m, j]) * dec(q_w[v, j]),
 *     the sum in double (exact: each product has at most 8 significant bits
 *     within 2^-18 .. 2^17), then the transform and mask of (3).
 */
double oracle_e4m3_decode(uint8_t c)
{
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

uint8_t oracle_e4m3_encode(float x)
{
    if (x != x)
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 464.0) /* at or past the midpoint above 448: saturate */
        return sign | 0x7E;
    if (a < ldexp(1.0, -6)) { /* subnormal: steps of 2^-9; m = 8 is the smallest normal */
        const double m = nearbyint(ldexp(a, 9));
        return sign | (uint8_t)m;
    }
    int e;
    (void)frexp(a, &e); /* a = f * 2^e with f in [0.5, 1): unbiased exponent e - 1 */
    e -= 1;
    double m = nearbyint(ldexp(a, 3 - e)); /* in [8, 16] */
    if (m == 16.0) {
        m = 8.0;
        e += 1;
    }
    const int code = ((e + 7) << 3) | ((int)m - 8);
    return sign | (uint8_t)(code > 0x7E ? 0x7E : code);
}

void oracle_quantize_rows_e4m3(const void *h, int64_t rows, int32_t hidden, int32_t dtype,
                               uint8_t *q, float *d)
{
    for (int64_t m = 0; m < rows; ++m) {
        float amax = 0.0f;
        for (int32_t j = 0; j < hidden; ++j) {
            const float a = fabsf((float)load_elem(h, m * hidden + j, dtype));
            if (a > amax)
                amax = a;
        }
        if (amax == 0.0f) {
            memset(q + m * hidden, 0, (size_t)hidden);
            d[m] = 1.0f;
            continue;
        }
        const float inv = 448.0f / amax; /* fp32 division, rounded once */
        const float dm = amax / 448.0f;
        d[m] = dm;
        for (int32_t j = 0; j < hidden; ++j) {
            const float x = (float)load_elem(h, m * hidden + j, dtype) * inv;
            q[m * hidden + j] = oracle_e4m3_encode(x);
        }
    }
}

void oracle_unary_rows_fp8(const uint8_t *qh, const float *dh, const uint8_t *qw,
                           const float *sw, const int64_t *rows, int64_t n_sel, int32_t hidden,
                           int64_t draft_vocab, int64_t target_vocab, double mult, double cap,
                           double *u_out)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < n_sel; ++r) {
        for (int64_t v = 0; v < draft_vocab; ++v) {
            const int64_t m = rows ? rows[r] : r;
            double u;
            if (v >= target_vocab) {
                u = -INFINITY;
            } else {
                double acc = 0.0;
                for (int32_t j = 0; j < hidden; ++j)
                    acc += oracle_e4m3_decode(qh[m * hidden + j]) *
                           oracle_e4m3_decode(qw[v * hidden + j]);
                const double z = (double)dh[m] * (double)sw[v] * acc;
                u = cap > 0.0 ? cap * tanh(mult * z / cap) : mult * z;
            }
            u_out[r * draft_vocab + v] = u;
        }
    }
}

/* ---- (11) NVFP4 lm_head: E2M1 codes with E4M3 block scales ----------------
 * The block-scaled 4-bit head (the vLLM DSpark review's padded-vocab draft
 * is an NVFP4 checkpoint; the sglang DFlash2 PR rejects quantized heads).
 * Plain definitions:
 *   - E2M1 element (the FP4 element of the OCP microscaling formats): sign
 *     bit, 2 exponent bits with bias 1, 1 mantissa bit; exponent field 0
 *     holds 0 and 0.5; the magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6; no
 *     infinities or NaN.  Encoding rounds to nearest, ties to the even code
 *     (mantissa bit 0), and saturates at 6.  Codes are 4 bits; two per byte,
 *     element 2i in the low nibble and element 2i+1 in the high nibble.
 *   - Every 16 consecutive elements along hidden share one scale, a
 *     non-negative E4M3 code (section 10's format), and every row of the
 *     activations (dynamic) or the whole weight tensor shares an fp32
 *     second-level scale.
 *   - Quantizing a row (activations) or a tensor (weights) X with amax A over
 *     it, all in fp32 (the values decide integer codes):
 *       enc = 2688 / A and g = A / 2688 (2688 = 6 * 448; A == 0: both 1);
 *       block b: a_b = max |x| over its 16 elements,
 *                s_b = E4M3((a_b / 6) * enc), each operation rounded;
 *                s_b == 0: the block's codes are 0; else
 *                r_b = enc / dec(s_b) and q_j = E2M1(x_j * r_b).
 *     Dequantized element: g * dec(s_b) * dec(q_j).
 *   - Logits: z[m, v] = g_h[m] * g_w * sum_b dec(s_h[m, b]) * dec(s_w[v, b])
 *     * sum_{j in b} dec(q_h[m, j]) * dec(q_w[v, j]), the sums in double
 *     (exact: each term has at most 9 significant bits), then the transform
 *     and mask of (3).
 */
double oracle_e2m1_decode(uint8_t c)
{
    const int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

uint8_t oracle_e2m1_encode(float x)
{
    const uint8_t sign = signbit(x) ? 0x8 : 0x0;
    const double a = fabs((double)x);
    if (a < 1.0) /* 0 and 0.5: steps of 0.5; 2 steps is the smallest normal, 1.0 */
        return sign | (uint8_t)nearbyint(2.0 * a);
    int e;
    (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): unbiased exponent e - 1 */
    e -= 1;
    double m = nearbyint(ldexp(a, 1 - e)); /* in [2, 4] */
    if (m == 4.0) {
        m = 2.0;
        e += 1;
    }
    if (e > 2) /* past 6 (or the midpoint 7 rounding up): saturate */
        return sign | 0x7;
    return sign | (uint8_t)(((e + 1) << 1) | ((int)m - 2));
}

/* Quantize rows x [rows, cols] (cols a multiple of 16) to packed codes
 * [rows, cols / 2], block scales [rows, cols / 16] and second-level scales
 * g: one per row (per_tensor == 0) or one for the whole tensor (g[0]). */
void oracle_quantize_nvfp4(const void *x, int64_t rows, int32_t cols, int32_t dtype,
                           int32_t per_tensor, uint8_t *codes, uint8_t *scales, float *g)
{
    float amax_t = 0.0f;
    if (per_tensor)
        for (int64_t i = 0; i < rows * (int64_t)cols; ++i) {
            const float a = fabsf((float)load_elem(x, i, dtype));
            if (a > amax_t)
                amax_t = a;
        }
    for (int64_t m = 0; m < rows; ++m) {
        float amax = amax_t;
        if (!per_tensor) {
            amax = 0.0f;
            for (int32_t j = 0; j < cols; ++j) {
                const float a = fabsf((float)load_elem(x, m * cols + j, dtype));
                if (a > amax)
                    amax = a;
            }
        }
        const float enc = amax == 0.0f ? 1.0f : 2688.0f / amax;
        const float gm = amax == 0.0f ? 1.0f : amax / 2688.0f;
        if (!per_tensor)
            g[m] = gm;
        else if (m == 0)
            g[0] = gm;
        for (int32_t b = 0; b < cols / 16; ++b) {
            float ab = 0.0f;
            for (int32_t j = 16 * b; j < 16 * b + 16; ++j) {
                const float a = fabsf((float)load_elem(x, m * cols + j, dtype));
                if (a > ab)
                    ab = a;
            }
            float t = ab / 6.0f;
            t = t * enc;
            const uint8_t sb = oracle_e4m3_encode(t);
            scales[m * (cols / 16) + b] = sb;
            const float dsb = (float)oracle_e4m3_decode(sb);
            const float r = dsb == 0.0f ? 0.0f : enc / dsb;
            for (int32_t j = 16 * b; j < 16 * b + 16; j += 2) {
                uint8_t lo = 0, hi = 0;
                if (dsb != 0.0f) {
                    lo = oracle_e2m1_encode((float)load_elem(x, m * cols + j, dtype) * r);
                    hi = oracle_e2m1_encode((float)load_elem(x, m * cols + j + 1, dtype) * r);
                }
                codes[m * (cols / 2) + j / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

void oracle_unary_rows_nvfp4(const uint8_t *qh, const uint8_t *sh, const float *gh,
                             const uint8_t *qw, const uint8_t *sw, float gw, const int64_t *rows,
                             int64_t n_sel, int32_t hidden, int64_t draft_vocab,
                             int64_t target_vocab, double mult, double cap, double *u_out)
{
    const int32_t nb = hidden / 16, hb = hidden / 2;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < n_sel; ++r) {
        for (int64_t v = 0; v < draft_vocab; ++v) {
            const int64_t m = rows ? rows[r] : r;
            double u;
            if (v >= target_vocab) {
                u = -INFINITY;
            } else {
                double acc = 0.0;
                for (int32_t b = 0; b < nb; ++b) {
                    double blk = 0.0;
                    for (int32_t j = 16 * b; j < 16 * b + 16; ++j) {
                        const uint8_t ch = (qh[m * hb + j / 2] >> (4 * (j & 1))) & 15;
                        const uint8_t cw = (qw[v * hb + j / 2] >> (4 * (j & 1))) & 15;
                        blk += oracle_e2m1_decode(ch) * oracle_e2m1_decode(cw);
                    }
                    acc += oracle_e4m3_decode(sh[m * nb + b]) * oracle_e4m3_decode(sw[v * nb + b]) *
                           blk;
                }
                const double z = (double)gh[m] * (double)gw * acc;
                u = cap > 0.0 ? cap * tanh(mult * z / cap) : mult * z;
            }
            u_out[r * draft_vocab + v] = u;
        }
    }
}

/* Threads the OpenMP loops above use: n > 0 sets them, n <= 0 only asks.
 * Returns the count now in force (1 without OpenMP).  Timing aid only. */
int oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
