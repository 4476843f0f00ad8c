/*
 * k3da_oracle.c -- fp64 CPU oracle of the K3 DFlash drafter block attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition that the CUDA path is checked against.  Only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark may load it; the
 * product path never does.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes follows the page "[None][feat] Share Kimi K3 FP4 modeling
 * and add NVFP4 support on SM103" (NVIDIA/TensorRT-LLM PR #20532):
 *   - the commit adding the drafter block attention ops k3_drafter_attn and
 *     k3_drafter_attn_qknorm: every draft token of a request attends densely
 *     (non-causally) to the request's paged context (HND pages of 64 tokens)
 *     and to its own block's K/V, which come from qkv and are never written
 *     to the pool; GQA with 6 query heads per KV head; head_dim 64; the
 *     fused variant applies per-head q/k RMSNorm and NeoX RoPE first;
 *   - the commit adding the contracts of both ops and the drafter's
 *     fused_qk_norm_rope cell: eps 1e-5, RoPE base 10000, NeoX pairing,
 *     head layouts 6/1 and 24/4, context lengths 0..2041, int32 and int64
 *     positions.
 * Steps the pages leave open take their plainest reading:
 *   - RMSNorm is x * (mean(x^2) + eps)^(-1/2) * w over the 64 dims of one
 *     head, with one weight vector for q and one for k shared by all heads;
 *   - NeoX RoPE rotates the pairs (j, j + D/2) by pos * base^(-2j/D), over
 *     the whole head;
 *   - qkv rows are token-major, request r's token i in row r*B + i, holding
 *     the Hq query heads, then the Hkv key heads, then the Hkv value heads;
 *   - query head h reads KV head h / (Hq/Hkv);
 *   - the pool is [page][K=0,V=1][kv_head][slot 0..63][dim];
 *   - context token c of request r sits in page table[r*S + c/64], slot c%64;
 *   - context keys are used as stored (already normalised and roped); only
 *     the block's q and k are normalised and roped by the fused variant;
 *     block values are used raw.
 *
 * Every floating-point step is fp64: bf16 inputs widen exactly, nothing is
 * rounded, softmax subtracts the row maximum, and the output is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an fp32. */
static double bf16_bits_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* RMSNorm of one head row x[0..D), scaled elementwise by w (fp64). */
void k3o_rmsnorm(const double *x, const double *w, int D, double eps, double *y)
{
    double sum_sq = 0.0;
    for (int j = 0; j < D; ++j)
        sum_sq += x[j] * x[j];
    double mean_sq = sum_sq / (double)D;
    double inv_rms = 1.0 / sqrt(mean_sq + eps);
    for (int j = 0; j < D; ++j)
        y[j] = x[j] * inv_rms * w[j];
}

/* NeoX rotary embedding of one head row at position pos: dimension j (for
 * j < D/2) pairs with j + D/2 and both turn by the angle pos * base^(-2j/D). */
void k3o_rope_neox(const double *x, int D, double pos, double base, double *y)
{
    int half = D / 2;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)D);
    for (int j = 0; j < half; ++j) {
        double inv_freq = pow(base, -2.0 * (double)j / (double)D);
        double theta = pos * inv_freq;
        double c = cos(theta), s = sin(theta);
        double lo = x[j], hi = x[j + half];
        tmp[j] = lo * c - hi * s;
        tmp[j + half] = hi * c + lo * s;
    }
    memcpy(y, tmp, sizeof(double) * (size_t)D);
    free(tmp);
}

/*
 * YaRN frequencies ("YaRN: Efficient Context Window Extension of Large
 * Language Models", Peng et al. 2023, the "NTK-by-parts" interpolation with
 * its ramp): pair j of the plain table turns at theta_j = base^(-2j/D), with
 * wavelength lambda_j = 2 pi / theta_j, and sees r_j = orig_len / lambda_j
 * wavelengths in the original context.  gamma = 0 below r = alpha, 1 above
 * r = beta, linear in between; the new frequency is
 * (1 - gamma) * theta_j / factor + gamma * theta_j.  factor 1 is the plain
 * table.
 */
void k3o_yarn_inv_freq(double *inv_freq, int D, double base, double factor, double orig_len,
                       double alpha, double beta)
{
    const double two_pi = 6.283185307179586476925286766559;
    for (int j = 0; j < D / 2; ++j) {
        double theta = pow(base, -2.0 * (double)j / (double)D);
        if (factor == 1.0) {
            inv_freq[j] = theta;
            continue;
        }
        double wavelength = two_pi / theta;
        double r = orig_len / wavelength;
        double gamma;
        if (r < alpha)
            gamma = 0.0;
        else if (r > beta)
            gamma = 1.0;
        else
            gamma = (r - alpha) / (beta - alpha);
        inv_freq[j] = (1.0 - gamma) * theta / factor + gamma * theta;
    }
}

/* Rotary embedding of one head row with an explicit frequency table: pair
 * (j, j + D/2) turns by pos * inv_freq[j]; both outputs are multiplied by
 * mscale (YaRN's attention temperature, sqrt(1/t), applied to q and k). */
void k3o_rope_table(const double *x, int D, double pos, const double *inv_freq, double mscale,
                    double *y)
{
    int half = D / 2;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)D);
    for (int j = 0; j < half; ++j) {
        double theta = pos * inv_freq[j];
        double c = cos(theta), s = sin(theta);
        double lo = x[j], hi = x[j + half];
        tmp[j] = (lo * c - hi * s) * mscale;
        tmp[j + half] = (hi * c + lo * s) * mscale;
    }
    memcpy(y, tmp, sizeof(double) * (size_t)D);
    free(tmp);
}

/* Error codes of k3o_attn. */
enum {
    K3O_OK = 0,
    K3O_BAD_SHAPE = 1,
    K3O_BAD_LENGTH = 2,
    K3O_BAD_PAGE = 3,
    K3O_NO_MEMORY = 4
};

/*
 * The whole op, for R requests of B block tokens each (T = R*B rows).
 *
 *   out        [T, Hq*D] fp64, written
 *   qkv        [T, (Hq + 2*Hkv)*D] bf16 bits
 *   pool       [num_pages, 2, Hkv, page_size, D] bf16 bits
 *   page_table [R, page_stride] int32
 *   ctx_lens   [R] int32
 *   qknorm     0: q and block k are used as given; 1: RMSNorm then RoPE
 *   positions  [T] int64 (read only when qknorm)
 *   q_w, k_w   [D] bf16 bits (read only when qknorm)
 *
 * Returns K3O_OK, or an error code without a meaningful output when a length
 * or a page id that would be read is out of range.
 */
static int attn_core(double *out, const uint16_t *qkv, const uint16_t *pool,
                     int64_t num_pages, const int32_t *page_table, int page_stride,
                     const int32_t *ctx_lens, int R, int B, int Hq, int Hkv, int D,
                     int page_size, double scale, int qknorm, const int64_t *positions,
                     const uint16_t *q_w, const uint16_t *k_w, double eps, double base,
                     const double *inv_freq, double mscale)
{
    if (R < 1 || B < 1 || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || D < 2 ||
        D % 2 != 0 || page_size < 1 || page_stride < 1)
        return K3O_BAD_SHAPE;
    const int G = Hq / Hkv;
    const int64_t row_w = (int64_t)(Hq + 2 * Hkv) * D;

    double *wq = (double *)malloc(sizeof(double) * (size_t)D);
    double *wk = (double *)malloc(sizeof(double) * (size_t)D);
    double *raw = (double *)malloc(sizeof(double) * (size_t)D);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)D);
    double *q = (double *)malloc(sizeof(double) * (size_t)D);
    if (!wq || !wk || !raw || !tmp || !q) {
        free(wq); free(wk); free(raw); free(tmp); free(q);
        return K3O_NO_MEMORY;
    }
    for (int j = 0; j < D; ++j) {
        wq[j] = qknorm ? bf16_bits_to_f64(q_w[j]) : 1.0;
        wk[j] = qknorm ? bf16_bits_to_f64(k_w[j]) : 1.0;
    }

    int status = K3O_OK;
    for (int r = 0; r < R && status == K3O_OK; ++r) {
        const int64_t L = ctx_lens[r];
        if (L < 0 || L > (int64_t)page_stride * page_size) {
            status = K3O_BAD_LENGTH;
            break;
        }
        const int64_t nkeys = L + B;
        double *K = (double *)malloc(sizeof(double) * (size_t)(nkeys * D));
        double *V = (double *)malloc(sizeof(double) * (size_t)(nkeys * D));
        double *s = (double *)malloc(sizeof(double) * (size_t)nkeys);
        if (!K || !V || !s) {
            free(K); free(V); free(s);
            status = K3O_NO_MEMORY;
            break;
        }
        for (int g = 0; g < Hkv && status == K3O_OK; ++g) {
            /* Key and value set of (request r, kv head g): the context first,
             * gathered through the page table, then the B block tokens. */
            for (int64_t c = 0; c < L; ++c) {
                int64_t page = page_table[(int64_t)r * page_stride + c / page_size];
                int64_t slot = c % page_size;
                if (page < 0 || page >= num_pages) {
                    status = K3O_BAD_PAGE;
                    break;
                }
                const uint16_t *kp =
                    pool + (((page * 2 + 0) * Hkv + g) * page_size + slot) * D;
                const uint16_t *vp =
                    pool + (((page * 2 + 1) * Hkv + g) * page_size + slot) * D;
                for (int j = 0; j < D; ++j) {
                    K[c * D + j] = bf16_bits_to_f64(kp[j]);
                    V[c * D + j] = bf16_bits_to_f64(vp[j]);
                }
            }
            if (status != K3O_OK)
                break;
            for (int jb = 0; jb < B; ++jb) {
                const int64_t t = (int64_t)r * B + jb;
                const uint16_t *kr = qkv + t * row_w + (int64_t)(Hq + g) * D;
                const uint16_t *vr = qkv + t * row_w + (int64_t)(Hq + Hkv + g) * D;
                for (int j = 0; j < D; ++j)
                    raw[j] = bf16_bits_to_f64(kr[j]);
                double *kdst = K + (L + jb) * D;
                if (qknorm) {
                    k3o_rmsnorm(raw, wk, D, eps, tmp);
                    if (inv_freq)
                        k3o_rope_table(tmp, D, (double)positions[t], inv_freq, mscale, kdst);
                    else
                        k3o_rope_neox(tmp, D, (double)positions[t], base, kdst);
                } else {
                    memcpy(kdst, raw, sizeof(double) * (size_t)D);
                }
                for (int j = 0; j < D; ++j)
                    V[(L + jb) * D + j] = bf16_bits_to_f64(vr[j]);
            }
            /* Every query head of this kv head, every block token. */
            for (int hl = 0; hl < G; ++hl) {
                const int h = g * G + hl;
                for (int i = 0; i < B; ++i) {
                    const int64_t t = (int64_t)r * B + i;
                    const uint16_t *qr = qkv + t * row_w + (int64_t)h * D;
                    for (int j = 0; j < D; ++j)
                        raw[j] = bf16_bits_to_f64(qr[j]);
                    if (qknorm) {
                        k3o_rmsnorm(raw, wq, D, eps, tmp);
                        if (inv_freq)
                            k3o_rope_table(tmp, D, (double)positions[t], inv_freq, mscale, q);
                        else
                            k3o_rope_neox(tmp, D, (double)positions[t], base, q);
                    } else {
                        memcpy(q, raw, sizeof(double) * (size_t)D);
                    }
                    double m = -INFINITY;
                    for (int64_t k = 0; k < nkeys; ++k) {
                        double dot = 0.0;
                        for (int j = 0; j < D; ++j)
                            dot += q[j] * K[k * D + j];
                        s[k] = scale * dot;
                        if (s[k] > m)
                            m = s[k];
                    }
                    double denom = 0.0;
                    for (int64_t k = 0; k < nkeys; ++k) {
                        s[k] = exp(s[k] - m);
                        denom += s[k];
                    }
                    double *o = out + t * (int64_t)Hq * D + (int64_t)h * D;
                    for (int j = 0; j < D; ++j) {
                        double acc = 0.0;
                        for (int64_t k = 0; k < nkeys; ++k)
                            acc += s[k] * V[k * D + j];
                        o[j] = acc / denom;
                    }
                }
            }
        }
        free(K); free(V); free(s);
    }
    free(wq); free(wk); free(raw); free(tmp); free(q);
    return status;
}

int k3o_attn(double *out, const uint16_t *qkv, const uint16_t *pool,
             int64_t num_pages, const int32_t *page_table, int page_stride,
             const int32_t *ctx_lens, int R, int B, int Hq, int Hkv, int D,
             int page_size, double scale, int qknorm, const int64_t *positions,
             const uint16_t *q_w, const uint16_t *k_w, double eps, double base)
{
    return attn_core(out, qkv, pool, num_pages, page_table, page_stride, ctx_lens, R, B, Hq, Hkv,
                     D, page_size, scale, qknorm, positions, q_w, k_w, eps, base, NULL, 1.0);
}

/*
 * The fused variant with YaRN RoPE: as k3o_attn with qknorm = 1, but the
 * block's q and k turn by the YaRN frequencies of k3o_yarn_inv_freq
 * (factor, orig_len, alpha = beta_slow, beta = beta_fast) and are scaled by
 * mscale.  factor 1 and mscale 1 give k3o_attn's fused result.
 */
int k3o_attn_yarn(double *out, const uint16_t *qkv, const uint16_t *pool,
                  int64_t num_pages, const int32_t *page_table, int page_stride,
                  const int32_t *ctx_lens, int R, int B, int Hq, int Hkv, int D,
                  int page_size, double scale, const int64_t *positions,
                  const uint16_t *q_w, const uint16_t *k_w, double eps, double base,
                  double factor, double orig_len, double beta_fast, double beta_slow,
                  double mscale)
{
    if (D < 2 || D % 2 != 0)
        return K3O_BAD_SHAPE;
    double *inv = (double *)malloc(sizeof(double) * (size_t)(D / 2));
    if (!inv)
        return K3O_NO_MEMORY;
    k3o_yarn_inv_freq(inv, D, base, factor, orig_len, beta_slow, beta_fast);
    int st = attn_core(out, qkv, pool, num_pages, page_table, page_stride, ctx_lens, R, B, Hq, Hkv,
                       D, page_size, scale, 1, positions, q_w, k_w, eps, base, inv, mscale);
    free(inv);
    return st;
}

/*
 * The drafter's fused q/k norm + RoPE cell on its own (the fused_qk_norm_rope
 * cell of the commit adding the ops' contracts), for T tokens of qkv:
 *
 *   out        [T, (Hq + 2*Hkv)*D] fp64, written: query head rows become
 *              rope(rmsnorm(q, q_w), pos_t), key head rows
 *              rope(rmsnorm(k, k_w), pos_t), value head rows are copied
 *   qkv        [T, (Hq + 2*Hkv)*D] bf16 bits (the layout of k3o_attn)
 *   positions  [T] int64
 *   q_w, k_w   [D] bf16 bits
 *
 * Returns K3O_OK, K3O_BAD_SHAPE or K3O_NO_MEMORY.
 */
static int norm_rope_core(double *out, const uint16_t *qkv, int T, int Hq, int Hkv, int D,
                          const int64_t *positions, const uint16_t *q_w, const uint16_t *k_w,
                          double eps, double base, const double *inv_freq, double mscale)
{
    if (T < 1 || Hq < 1 || Hkv < 1 || D < 2 || (D % 2) != 0)
        return K3O_BAD_SHAPE;
    const int heads = Hq + 2 * Hkv;
    double *wq = (double *)malloc(sizeof(double) * (size_t)D);
    double *wk = (double *)malloc(sizeof(double) * (size_t)D);
    double *raw = (double *)malloc(sizeof(double) * (size_t)D);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)D);
    if (!wq || !wk || !raw || !tmp) {
        free(wq); free(wk); free(raw); free(tmp);
        return K3O_NO_MEMORY;
    }
    for (int j = 0; j < D; ++j) {
        wq[j] = bf16_bits_to_f64(q_w[j]);
        wk[j] = bf16_bits_to_f64(k_w[j]);
    }
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < heads; ++h) {
            const uint16_t *src = qkv + ((size_t)t * heads + h) * D;
            double *dst = out + ((size_t)t * heads + h) * D;
            for (int j = 0; j < D; ++j)
                raw[j] = bf16_bits_to_f64(src[j]);
            if (h < Hq + Hkv) {
                k3o_rmsnorm(raw, h < Hq ? wq : wk, D, eps, tmp);
                if (inv_freq)
                    k3o_rope_table(tmp, D, (double)positions[t], inv_freq, mscale, dst);
                else
                    k3o_rope_neox(tmp, D, (double)positions[t], base, dst);
            } else {
                memcpy(dst, raw, sizeof(double) * (size_t)D);
            }
        }
    }
    free(wq); free(wk); free(raw); free(tmp);
    return K3O_OK;
}

int k3o_qk_norm_rope(double *out, const uint16_t *qkv, int T, int Hq, int Hkv, int D,
                     const int64_t *positions, const uint16_t *q_w, const uint16_t *k_w,
                     double eps, double base)
{
    return norm_rope_core(out, qkv, T, Hq, Hkv, D, positions, q_w, k_w, eps, base, NULL, 1.0);
}

/* The cell with YaRN RoPE (see k3o_attn_yarn). */
int k3o_qk_norm_rope_yarn(double *out, const uint16_t *qkv, int T, int Hq, int Hkv, int D,
                          const int64_t *positions, const uint16_t *q_w, const uint16_t *k_w,
                          double eps, double base, double factor, double orig_len,
                          double beta_fast, double beta_slow, double mscale)
{
    if (D < 2 || D % 2 != 0)
        return K3O_BAD_SHAPE;
    double *inv = (double *)malloc(sizeof(double) * (size_t)(D / 2));
    if (!inv)
        return K3O_NO_MEMORY;
    k3o_yarn_inv_freq(inv, D, base, factor, orig_len, beta_slow, beta_fast);
    int st = norm_rope_core(out, qkv, T, Hq, Hkv, D, positions, q_w, k_w, eps, base, inv, mscale);
    free(inv);
    return st;
}
