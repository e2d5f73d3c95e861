/*
 * fp64 CPU oracle of one mixture-of-experts (MoE) layer, of the grouped-query
 * decode attention of the model's full-attention layers and of the Gated
 * DeltaNet scan of its linear-attention layers (the last two at the end).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * Source of the method: the page "Perplexity libera o Lily" (noticiai.com.br):
 *   - section "O modelo em tres formatos de carga": a router scores 256 experts
 *     and selects eight, plus one shared expert that sees every token;
 *   - section "Prefill e decode: onde estao os ganhos": 4-bit group-wise affine
 *     weights, each group of 64 weights sharing one bf16 scale and one bf16 bias,
 *     rebuilt before the GEMM, FP32 accumulation; on-GPU histogram, prefix scan,
 *     scatter and block map of the routing.
 * Readings where the page is silent (all also stated in the design notes):
 *   - softmax over the E logits, keep the top k, renormalise over the k
 *     (which equals a softmax over the k selected logits); lower expert index
 *     first among equal logits; slots ordered by descending logit;
 *   - the shared expert is added with weight 1.0, no gate;
 *   - q is the unsigned nibble, low nibble = even k; groups run along the
 *     reduction dimension;  w = q * scale + bias;
 *   - experts are SwiGLU:  y = Wd (silu(Wg x) * (Wu x)),  silu(z) = z/(1+e^-z).
 *
 * Everything is computed in double precision, plainly, one token at a time.
 * Nothing is rounded to bf16: the oracle is the exact result (up to fp64
 * rounding) that the GPU path approximates.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> double (exact). */
static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Element k of a packed row: byte k/2, low nibble for even k, high for odd k. */
static int nibble_at(const uint8_t *row, int64_t k)
{
    uint8_t byte = row[k / 2];
    return (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
}

/* One dequantised weight: w[n][k] = q[n][k] * scale[n][k/G] + bias[n][k/G]. */
static double weight_at(const uint8_t *q, const uint16_t *scale, const uint16_t *bias,
                        int64_t K, int64_t G, int64_t n, int64_t k)
{
    int64_t ng = K / G;
    double s = bf16_value(scale[n * ng + k / G]);
    double b = bf16_value(bias[n * ng + k / G]);
    return (double)nibble_at(q + n * (K / 2), k) * s + b;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Dequantise a whole [rows][K] matrix into w (row-major doubles). */
void oracle_dequant(const uint8_t *q, const uint16_t *scale, const uint16_t *bias,
                    int64_t rows, int64_t K, int64_t G, double *w)
{
    for (int64_t n = 0; n < rows; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = weight_at(q, scale, bias, K, G, n, k);
}

/* Router logits: l[t][e] = sum_k x[t][k] * Wr[e][k] + bias_r[e]  (bias_r may be NULL). */
void oracle_logits(const uint16_t *x, const uint16_t *wr, const float *bias_r,
                   int64_t T, int64_t d, int64_t E, double *logits)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int64_t k = 0; k < d; ++k)
                acc += bf16_value(x[t * d + k]) * bf16_value(wr[e * d + k]);
            if (bias_r) acc += (double)bias_r[e];
            logits[t * E + e] = acc;
        }
    }
}

typedef struct { double neg_logit; int32_t expert; } scored;

/* Ascending (-logit, expert): descending logit, lower index first on equal logits. */
static int scored_cmp(const void *pa, const void *pb)
{
    const scored *a = (const scored *)pa, *b = (const scored *)pb;
    if (a->neg_logit < b->neg_logit) return -1;
    if (a->neg_logit > b->neg_logit) return 1;
    return (a->expert > b->expert) - (a->expert < b->expert);
}

/*
 * Top-k selection and weights.  Sort all E (-logit, e) pairs, keep the first k.
 * Weights: w_j = exp(l_j - l_max) / sum_j' exp(l_j' - l_max) over the k kept,
 * which is the softmax over all E renormalised over the k kept.
 */
void oracle_select(const double *logits, int64_t T, int64_t E, int64_t k,
                   int32_t *idx, double *w)
{
#pragma omp parallel
    {
        scored *buf = (scored *)malloc(sizeof(scored) * (size_t)E);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t e = 0; e < E; ++e) {
                buf[e].neg_logit = -logits[t * E + e];
                buf[e].expert = (int32_t)e;
            }
            qsort(buf, (size_t)E, sizeof(scored), scored_cmp);
            double lmax = -buf[0].neg_logit, denom = 0.0;
            for (int64_t j = 0; j < k; ++j) denom += exp(-buf[j].neg_logit - lmax);
            for (int64_t j = 0; j < k; ++j) {
                idx[t * k + j] = buf[j].expert;
                w[t * k + j] = exp(-buf[j].neg_logit - lmax) / denom;
            }
        }
        free(buf);
    }
}

/*
 * Routing tables from the selection idx[T][k]:
 *   counts[e]  = number of (t, j) with idx[t][j] == e                 (histogram)
 *   offsets    = exclusive prefix sum of counts, offsets[E] = T*k     (scan)
 *   perm[offsets[e] + r] = t*k + j for the r-th assignment of expert e,
 *                          counted in ascending (t, j) order           (scatter)
 *   block map: for e ascending, b < ceil(counts[e]/BM):
 *              (e, offsets[e] + b*BM, min(BM, counts[e] - b*BM))       (block map)
 * block_map must hold at least sum_e ceil(counts[e]/BM) entries of 3 int32.
 */
void oracle_route_tables(const int32_t *idx, int64_t T, int64_t E, int64_t k, int64_t BM,
                         int32_t *counts, int32_t *offsets, int32_t *perm,
                         int32_t *block_map, int32_t *n_blocks)
{
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t a = 0; a < T * k; ++a) counts[idx[a]] += 1;

    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];

    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    for (int64_t e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < k; ++j) {
            int32_t e = idx[t * k + j];
            perm[cursor[e]] = (int32_t)(t * k + j);
            cursor[e] += 1;
        }
    free(cursor);

    int32_t nb = 0;
    for (int64_t e = 0; e < E; ++e)
        for (int64_t start = 0; start < counts[e]; start += BM) {
            int64_t rows = counts[e] - start < BM ? counts[e] - start : BM;
            block_map[3 * nb + 0] = (int32_t)e;
            block_map[3 * nb + 1] = (int32_t)(offsets[e] + start);
            block_map[3 * nb + 2] = (int32_t)rows;
            nb += 1;
        }
    *n_blocks = nb;
}

/* One layer's weights.  Routed experts are stacked by expert. */
typedef struct {
    int64_t d, E, I, I_shared, G;
    const uint8_t *gate_q, *up_q, *down_q;
    const uint16_t *gate_s, *gate_b, *up_s, *up_b, *down_s, *down_b;
    const uint8_t *sh_gate_q, *sh_up_q, *sh_down_q;
    const uint16_t *sh_gate_s, *sh_gate_b, *sh_up_s, *sh_up_b, *sh_down_s, *sh_down_b;
} oracle_layer;

static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * One SwiGLU expert on one token: y = Wd (silu(Wg x) * (Wu x)).
 * Wg, Wu: [Ie][d] (row offset r0 into the stacked arrays); Wd: [d][Ie] (row offset r0d).
 * h is scratch of Ie doubles.
 */
static void expert_apply(const oracle_layer *L, int shared, int64_t e, const double *x,
                         double *h, double *y)
{
    const int64_t d = L->d, G = L->G;
    const int64_t Ie = shared ? L->I_shared : L->I;
    const uint8_t *gq = shared ? L->sh_gate_q : L->gate_q;
    const uint16_t *gs = shared ? L->sh_gate_s : L->gate_s, *gb = shared ? L->sh_gate_b : L->gate_b;
    const uint8_t *uq = shared ? L->sh_up_q : L->up_q;
    const uint16_t *us = shared ? L->sh_up_s : L->up_s, *ub = shared ? L->sh_up_b : L->up_b;
    const uint8_t *dq = shared ? L->sh_down_q : L->down_q;
    const uint16_t *ds = shared ? L->sh_down_s : L->down_s, *db = shared ? L->sh_down_b : L->down_b;
    const int64_t r0 = shared ? 0 : e * Ie;   /* first gate/up row of this expert */
    const int64_t r0d = shared ? 0 : e * d;   /* first down row of this expert */

    for (int64_t i = 0; i < Ie; ++i) {
        double g = 0.0, u = 0.0;
        for (int64_t k = 0; k < d; ++k) {
            g += weight_at(gq, gs, gb, d, G, r0 + i, k) * x[k];
            u += weight_at(uq, us, ub, d, G, r0 + i, k) * x[k];
        }
        h[i] = silu(g) * u;
    }
    for (int64_t n = 0; n < d; ++n) {
        double acc = 0.0;
        for (int64_t i = 0; i < Ie; ++i)
            acc += weight_at(dq, ds, db, Ie, G, r0d + n, i) * h[i];
        y[n] = acc;
    }
}

/*
 * Layer output for a list of tokens:
 *   out[t] = sum_j w[t][j] * expert_{idx[t][j]}(x_t) + shared(x_t)
 * x: bf16 [T][d]; idx/w: [T][k]; tokens: n_tok indices into [0, T);
 * out: [n_tok][d] doubles, row i for token tokens[i].
 */
void oracle_moe_tokens(const oracle_layer *L, const uint16_t *x, int64_t k,
                       const int32_t *idx, const double *w,
                       const int64_t *tokens, int64_t n_tok, double *out)
{
    const int64_t d = L->d;
    const int64_t hmax = L->I > L->I_shared ? L->I : L->I_shared;
#pragma omp parallel
    {
        double *xv = (double *)malloc(sizeof(double) * (size_t)d);
        double *y = (double *)malloc(sizeof(double) * (size_t)d);
        double *h = (double *)malloc(sizeof(double) * (size_t)hmax);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_tok; ++i) {
            const int64_t t = tokens[i];
            double *o = out + i * d;
            for (int64_t c = 0; c < d; ++c) xv[c] = bf16_value(x[t * d + c]);
            expert_apply(L, 1, 0, xv, h, y);
            for (int64_t c = 0; c < d; ++c) o[c] = y[c];          /* shared, weight 1 */
            for (int64_t j = 0; j < k; ++j) {
                expert_apply(L, 0, idx[t * k + j], xv, h, y);
                for (int64_t c = 0; c < d; ++c) o[c] += w[t * k + j] * y[c];
            }
        }
        free(xv); free(y); free(h);
    }
}

/*
 * Parameter-free RMS normalisation used to chain decode layers:
 * xn[t] = out[t] / sqrt(mean_c(out[t][c]^2) + eps).
 */
void oracle_rms_norm(const double *out, int64_t T, int64_t d, double eps, double *xn)
{
    for (int64_t t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int64_t c = 0; c < d; ++c) ss += out[t * d + c] * out[t * d + c];
        double inv = 1.0 / sqrt(ss / (double)d + eps);
        for (int64_t c = 0; c < d; ++c) xn[t * d + c] = out[t * d + c] * inv;
    }
}

/*
 * Decode attention over a KV cache stored in fixed-size blocks (grouped-query
 * attention), one step for each of B sequences.
 *
 * Source of the method: the page "Perplexity libera o Lily" (noticiai.com.br):
 *   - section "O modelo em tres formatos de carga": the full-attention layers
 *     use grouped-query attention with 16 query heads and two KV heads, over a
 *     growing KV cache;
 *   - section "Prefill e decode: onde estao os ganhos": decode packs the query
 *     heads of a KV head together (GQA packing), reads the cache coalesced, and
 *     keeps it in a fixed-block layout.
 * Readings where the page is silent: plain scaled dot-product attention,
 *   o_h = sum_t softmax_t(scale * q_h . k_{g,t}) v_{g,t},  g = h / (H_q / H_kv),
 * with the caller's scale (1/sqrt(D) by default); K and V of token t of a
 * sequence sit in cache block block_table[t / bs], row t % bs of that block,
 * laid out [block][kv head][row][D].
 *
 * q: bf16 [B][H_q][D]; k_cache, v_cache: bf16 [n_blocks][H_kv][bs][D];
 * block_table: [B][max_blocks]; seq_lens: [B] (>= 1); out: [B][H_q][D] doubles.
 */
void oracle_attn_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_table, const int32_t *seq_lens,
                        int64_t B, int64_t H_q, int64_t H_kv, int64_t D, int64_t bs, int64_t max_blocks,
                        double scale, double *out)
{
    const int64_t group = H_q / H_kv;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t h = 0; h < H_q; ++h) {
            const int64_t g = h / group;
            const int64_t L = seq_lens[b];
            const uint16_t *qh = q + (b * H_q + h) * D;
            double *o = out + (b * H_q + h) * D;
            double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
            /* scores */
            double m = -INFINITY;
            for (int64_t t = 0; t < L; ++t) {
                const int64_t blk = block_table[b * max_blocks + t / bs];
                const uint16_t *kt = k_cache + ((blk * H_kv + g) * bs + t % bs) * D;
                double dot = 0.0;
                for (int64_t c = 0; c < D; ++c) dot += bf16_value(qh[c]) * bf16_value(kt[c]);
                s[t] = scale * dot;
                if (s[t] > m) m = s[t];
            }
            /* softmax weights and the weighted sum of values */
            double den = 0.0;
            for (int64_t t = 0; t < L; ++t) {
                s[t] = exp(s[t] - m);
                den += s[t];
            }
            for (int64_t c = 0; c < D; ++c) o[c] = 0.0;
            for (int64_t t = 0; t < L; ++t) {
                const int64_t blk = block_table[b * max_blocks + t / bs];
                const uint16_t *vt = v_cache + ((blk * H_kv + g) * bs + t % bs) * D;
                const double w = s[t] / den;
                for (int64_t c = 0; c < D; ++c) o[c] += w * bf16_value(vt[c]);
            }
            free(s);
        }
    }
}

/*
 * Gated DeltaNet scan: the fixed-size recurrence of the model's linear-attention
 * layers, over T tokens of one sequence.
 *
 * Source: the page "Perplexity libera o Lily" (noticiai.com.br), section "O
 * modelo em tres formatos de carga" (30 Gated DeltaNet layers: a recurrence of
 * fixed size) and section "Prefill e decode: onde estao os ganhos" (a scan
 * with the recurrent state held in registers).  The page gives no formula;
 * the reading is the gated delta rule of Gated DeltaNet.  Per value head h
 * (key head hk = h / (H_v / H_k)), state S (d_v x d_k), token t:
 *   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T
 *       (= S_{t-1} alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T)
 *   o_t = scale S_t q_t
 * q, k: bf16 [T][H_k][d_k]; v: bf16 [T][H_v][d_v]; alpha, beta: f32 [T][H_v];
 * S0: [H_v][d_v][d_k] doubles or NULL (zeros); o: [T][H_v][d_v] doubles;
 * S_out: [H_v][d_v][d_k] doubles (the state after the last token).
 */
void oracle_gdn_scan(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                     const float *beta, const double *S0, int64_t T, int64_t H_k, int64_t H_v, int64_t dk,
                     int64_t dv, double scale, double *o, double *S_out)
{
    const int64_t group = H_v / H_k;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t h = 0; h < H_v; ++h) {
        const int64_t hk = h / group;
        double *S = S_out + h * dv * dk;
        double *kv = (double *)malloc(sizeof(double) * (size_t)dk);
        double *qv = (double *)malloc(sizeof(double) * (size_t)dk);
        for (int64_t i = 0; i < dv * dk; ++i) S[i] = S0 ? S0[h * dv * dk + i] : 0.0;
        for (int64_t t = 0; t < T; ++t) {
            const double a = (double)alpha[t * H_v + h], b = (double)beta[t * H_v + h];
            for (int64_t j = 0; j < dk; ++j) {
                kv[j] = bf16_value(k[(t * H_k + hk) * dk + j]);
                qv[j] = bf16_value(q[(t * H_k + hk) * dk + j]);
            }
            for (int64_t i = 0; i < dv; ++i) {
                double *row = S + i * dk;
                double u = 0.0;                                   /* (S_{t-1} k_t)_i */
                for (int64_t j = 0; j < dk; ++j) u += row[j] * kv[j];
                const double c = b * (bf16_value(v[(t * H_v + h) * dv + i]) - a * u);
                double oi = 0.0;
                for (int64_t j = 0; j < dk; ++j) {
                    row[j] = a * row[j] + c * kv[j];
                    oi += row[j] * qv[j];
                }
                o[(t * H_v + h) * dv + i] = scale * oi;
            }
        }
        free(kv);
        free(qv);
    }
}
