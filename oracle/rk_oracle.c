/*
 * rk_oracle.c -- float64 CPU oracle for deterministic paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file; only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg use it.  It shares no code, header, table
 * or constant generator with the CUDA path.
 *
 * What it computes (the plain definition, step by step, in float64):
 *
 *   "WS2 PR7 Fused Attention Backend Alignment", section "Current
 *   Implementation": the strict control materialises the logical paged K/V
 *   (block table -> logical token order) before any arithmetic, and the
 *   output is restored to out [B, Hq, Sq, D] with an attention-domain LSE of
 *   shape [B, Hq, Sq].
 *
 *   Same page, section "FlashInfer RoPE Fusion": pre-RoPE Q and a pre-RoPE K
 *   cache are rotated with the Llama rotate-half (non-interleaved) rule,
 *   theta = 1e6, rope_scale = 1.0, rotary_dim = head_dim.
 *
 *   "Add FlashInfer RoPE-fused paged attention scaffold" (PR #279), boundary
 *   table: GQA packing fixed from the head layout, FP32 attention-domain LSE.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - softmax scale: 1/sqrt(D) unless the caller passes another one;
 *   - LSE: natural log of the sum of exp of the *scaled* scores;
 *   - key t of row b sits at logical position t and is visible to a query at
 *     position p iff t <= p and t < kv_len[b];
 *   - query head h reads KV head h / (Hq / Hkv);
 *   - rotation angle of pair i at position p: p * theta^(-2i/D) / rope_scale;
 *   - a query with no visible key gets out = 0 and lse = -inf.
 *
 * The arithmetic for one output is exactly the definition: gather, convert
 * to float64, rotate, score every visible key, subtract the maximum, sum the
 * exponentials in ascending key order, divide.  Queries are distributed over
 * OpenMP threads; that changes nothing inside any one output.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_E_ARG 1
#define ORACLE_E_PAGE 2
#define ORACLE_E_NOMEM 3

/* Input element types accepted for q / k_cache / v_cache. */
#define ORACLE_F64 0
#define ORACLE_BF16 1 /* raw bfloat16 bit patterns (uint16) */

static double to_f64(const void *base, int64_t idx, int dtype) {
    if (dtype == ORACLE_BF16) {
        uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f; /* exact: every bfloat16 is a float32 */
    }
    return ((const double *)base)[idx];
}

/* Inverse frequency of rotation pair i:  theta^(-2i/D). */
static double inv_freq(int i, int D, double theta) {
    return pow(theta, -2.0 * (double)i / (double)D);
}

/*
 * Rotate-half RoPE of one D-vector x at position pos (float64 in and out).
 * For i < D/2:  y[i]       = x[i] cos(a_i) - x[i + D/2] sin(a_i)
 *               y[i + D/2] = x[i + D/2] cos(a_i) + x[i] sin(a_i)
 * with a_i = pos * theta^(-2i/D) / rope_scale.
 */
void rk_oracle_rope(const double *x, int D, double pos, double theta,
                    double rope_scale, double *y) {
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        double a = pos * inv_freq(i, D, theta) / rope_scale;
        double c = cos(a), s = sin(a);
        double lo = x[i], hi = x[i + half];
        y[i] = lo * c - hi * s;
        y[i + half] = hi * c + lo * s;
    }
}

/*
 * Materialise the logical cache of one row: dst[h][t][d] = cache[page][slot][h][d]
 * with page = block_table[b, t / page_size], slot = t % page_size, for
 * t < kv_len[b].  Returns ORACLE_E_PAGE if a needed page id is outside
 * [0, num_pages).
 */
int rk_oracle_materialize_row(const void *cache, int dtype, int num_pages,
                              int page_size, int Hkv, int D,
                              const int32_t *block_table, int W,
                              const int32_t *kv_lens, int b, double *dst) {
    int n = kv_lens[b];
    if (n < 0 || n > W * page_size) return ORACLE_E_ARG;
    for (int t = 0; t < n; ++t) {
        int page = block_table[(int64_t)b * W + t / page_size];
        int slot = t % page_size;
        if (page < 0 || page >= num_pages) return ORACLE_E_PAGE;
        for (int h = 0; h < Hkv; ++h) {
            int64_t src = (((int64_t)page * page_size + slot) * Hkv + h) * D;
            double *out = dst + ((int64_t)h * n + t) * D;
            for (int d = 0; d < D; ++d) out[d] = to_f64(cache, src + d, dtype);
        }
    }
    return ORACLE_OK;
}

/* One unit of work: row b, KV head kh, queries s in [s0, s1). */
typedef struct {
    int b, kh, s0, s1;
} task_t;

/*
 * Paged causal attention with fused RoPE, float64.
 *
 *   q            [B, Hq, Sq, D]      (dtype qkv_dtype)
 *   k_cache      [num_pages, page_size, Hkv, D]
 *   v_cache      [num_pages, page_size, Hkv, D]
 *   block_table  [B, W] int32
 *   kv_lens      [B] int32
 *   position_ids [B, Sq] int32
 *   out          [B, Hq, Sq, D] float64
 *   lse          [B, Hq, Sq] float64
 *
 * row_mask: optional [B, Sq] uint8; when non-NULL only queries with a
 * non-zero entry are computed (the others are left untouched).
 */
int rk_oracle_attention(int B, int Sq, int Hq, int Hkv, int D, int page_size,
                        int num_pages, int W, const void *q,
                        const void *k_cache, const void *v_cache,
                        int qkv_dtype, const int32_t *block_table,
                        const int32_t *kv_lens, const int32_t *position_ids,
                        double rope_theta, double rope_scale, double sm_scale,
                        const uint8_t *row_mask, double *out, double *lse,
                        int nthreads) {
    if (B < 0 || Sq < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || (D % 2) ||
        page_size <= 0 || W < 0 || Hq % Hkv)
        return ORACLE_E_ARG;
    const int G = Hq / Hkv;
    const int CHUNK = 64;
    int nchunks = (Sq + CHUNK - 1) / CHUNK;
    int64_t ntask = (int64_t)B * Hkv * nchunks;
    task_t *tasks = (task_t *)malloc(sizeof(task_t) * (size_t)(ntask > 0 ? ntask : 1));
    if (!tasks) return ORACLE_E_NOMEM;
    int64_t k = 0;
    for (int b = 0; b < B; ++b)
        for (int kh = 0; kh < Hkv; ++kh)
            for (int c = 0; c < nchunks; ++c) {
                tasks[k].b = b;
                tasks[k].kh = kh;
                tasks[k].s0 = c * CHUNK;
                tasks[k].s1 = (c + 1) * CHUNK < Sq ? (c + 1) * CHUNK : Sq;
                ++k;
            }
    int err = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t ti = 0; ti < ntask; ++ti) {
        const task_t tk = tasks[ti];
        const int b = tk.b, kh = tk.kh;
        const int n_kv = kv_lens[b];
        if (n_kv < 0 || n_kv > W * page_size) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            err = ORACLE_E_ARG;
            continue;
        }
        /* Number of keys any query of this chunk may see. */
        int need = 0;
        for (int s = tk.s0; s < tk.s1; ++s) {
            if (row_mask && !row_mask[(int64_t)b * Sq + s]) continue;
            int p = position_ids[(int64_t)b * Sq + s];
            int nv = p < 0 ? 0 : (p + 1 < n_kv ? p + 1 : n_kv);
            if (nv > need) need = nv;
        }
        double *kr = (double *)malloc(sizeof(double) * ((size_t)need * D + 1));
        double *vr = (double *)malloc(sizeof(double) * ((size_t)need * D + 1));
        double *tmp = (double *)malloc(sizeof(double) * (size_t)D);
        double *qr = (double *)malloc(sizeof(double) * (size_t)D);
        double *sc = (double *)malloc(sizeof(double) * ((size_t)need + 1));
        if (!kr || !vr || !tmp || !qr || !sc) {
            free(kr); free(vr); free(tmp); free(qr); free(sc);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            err = ORACLE_E_NOMEM;
            continue;
        }
        /* Step 1: gather logical K/V for t < need; rotate K at position t. */
        int bad = 0;
        for (int t = 0; t < need && !bad; ++t) {
            int page = block_table[(int64_t)b * W + t / page_size];
            int slot = t % page_size;
            if (page < 0 || page >= num_pages) { bad = 1; break; }
            int64_t src = (((int64_t)page * page_size + slot) * Hkv + kh) * D;
            for (int d = 0; d < D; ++d) {
                tmp[d] = to_f64(k_cache, src + d, qkv_dtype);
                vr[(int64_t)t * D + d] = to_f64(v_cache, src + d, qkv_dtype);
            }
            rk_oracle_rope(tmp, D, (double)t, rope_theta, rope_scale,
                           kr + (int64_t)t * D);
        }
        if (bad) {
            free(kr); free(vr); free(tmp); free(qr); free(sc);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            err = ORACLE_E_PAGE;
            continue;
        }
        /* Step 2: every query head of this KV head's group, every query. */
        for (int g = 0; g < G; ++g) {
            const int h = kh * G + g;
            for (int s = tk.s0; s < tk.s1; ++s) {
                if (row_mask && !row_mask[(int64_t)b * Sq + s]) continue;
                const int p = position_ids[(int64_t)b * Sq + s];
                const int nv = p < 0 ? 0 : (p + 1 < n_kv ? p + 1 : n_kv);
                const int64_t qoff = (((int64_t)b * Hq + h) * Sq + s) * D;
                double *o = out + qoff;
                double *l = lse + ((int64_t)b * Hq + h) * Sq + s;
                if (nv == 0) {
                    for (int d = 0; d < D; ++d) o[d] = 0.0;
                    *l = -INFINITY;
                    continue;
                }
                for (int d = 0; d < D; ++d) tmp[d] = to_f64(q, qoff + d, qkv_dtype);
                rk_oracle_rope(tmp, D, (double)p, rope_theta, rope_scale, qr);
                double m = -INFINITY;
                for (int t = 0; t < nv; ++t) {
                    double acc = 0.0;
                    const double *kt = kr + (int64_t)t * D;
                    for (int d = 0; d < D; ++d) acc += qr[d] * kt[d];
                    sc[t] = acc * sm_scale;
                    if (sc[t] > m) m = sc[t];
                }
                double sum = 0.0;
                for (int t = 0; t < nv; ++t) {
                    sc[t] = exp(sc[t] - m);
                    sum += sc[t];
                }
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                for (int t = 0; t < nv; ++t) {
                    const double w = sc[t] / sum;
                    const double *vt = vr + (int64_t)t * D;
                    for (int d = 0; d < D; ++d) o[d] += w * vt[d];
                }
                *l = m + log(sum);
            }
        }
        free(kr); free(vr); free(tmp); free(qr); free(sc);
    }
    free(tasks);
    return err;
}

/*
 * Gradient of the same attention, float64: "Add FlashInfer RoPE-fused paged
 * attention scaffold", scope table, Backward row (dropout 0, deterministic
 * backward).  For the scalar L = sum over (b, h, s, d) of dout * out, with
 * out as computed by rk_oracle_attention, it returns dL/dq, dL/dk_cache and
 * dL/dv_cache.  Per query (rotated q' at position p, visible keys t < nv,
 * rotated keys k'_t):
 *
 *   s_t   = sm_scale * (q' . k'_t),   P_t = exp(s_t - lse),   out = sum_t P_t v_t
 *   Dq    = dout . out
 *   dP_t  = dout . v_t,               dS_t = P_t (dP_t - Dq)
 *   dv_t += P_t dout                  dk'_t += sm_scale dS_t q'
 *   dq'   = sm_scale sum_t dS_t k'_t
 *
 * and the rotation is undone with its transpose (rotation by the negative
 * angle): dq = R(p)^T dq', dk_t = R(t)^T dk'_t.  The derivation is the chain
 * rule through the softmax (d softmax_t / d s_u = P_t (delta_tu - P_u)).
 *
 * Outputs: dq [B, Hq, Sq, D]; dk, dv in the cache layout [num_pages,
 * page_size, Hkv, D].  For every row the pages of its first ceil(kv_len / P)
 * table entries are written in full (slots at or past kv_len get 0); other
 * pages are left untouched.  mag_dq / mag_dk / mag_dv (optional, same
 * layouts) receive the sums of the absolute values of the terms of each
 * output element (after the rotation: |R^T x|_i <= |x_i| + |x_(i +- D/2)|),
 * from which rounding-error bounds of other implementations are derived.
 * sens_dq / sens_dk (optional) receive, per element, the sum of the absolute
 * values of its terms' dependence on Dq scaled by A = sum_d |dout_d out_d|
 * (the bound on a relative change of every out element entering Dq):
 * sum_t sm_scale P_t |k'_t| A for dq', sum_q sm_scale P_t |q'| A for dk'.
 * Work is split over (b, KV head): each unit owns its keys' dk / dv.
 */
int rk_oracle_attention_backward(int B, int Sq, int Hq, int Hkv, int D, int page_size,
                                 int num_pages, int W, const void *q, const void *k_cache,
                                 const void *v_cache, int qkv_dtype, const void *dout,
                                 int dout_dtype, const int32_t *block_table,
                                 const int32_t *kv_lens, const int32_t *position_ids,
                                 double rope_theta, double rope_scale, double sm_scale,
                                 double *dq, double *dk, double *dv, double *mag_dq,
                                 double *mag_dk, double *mag_dv, double *sens_dq,
                                 double *sens_dk, int nthreads) {
    if (B < 0 || Sq < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || (D % 2) ||
        page_size <= 0 || W < 0 || Hq % Hkv)
        return ORACLE_E_ARG;
    const int G = Hq / Hkv, half = D / 2;
    const int64_t units = (int64_t)B * Hkv;
    int err = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        const int b = (int)(u / Hkv), kh = (int)(u % Hkv);
        const int n = kv_lens[b];
        if (n < 0 || n > W * page_size) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            err = ORACLE_E_ARG;
            continue;
        }
        const size_t nd = (size_t)n * D + 1;
        double *kr = (double *)malloc(sizeof(double) * nd);   /* rotated keys */
        double *vr = (double *)malloc(sizeof(double) * nd);
        double *gk = (double *)calloc(nd, sizeof(double));    /* dk' (rotated domain) */
        double *gv = (double *)calloc(nd, sizeof(double));
        double *mk = (double *)calloc(nd, sizeof(double));    /* magnitudes of dk' terms */
        double *mv = (double *)calloc(nd, sizeof(double));
        double *sk = (double *)calloc(nd, sizeof(double));    /* Dq sensitivity of dk' */
        double *pr = (double *)malloc(sizeof(double) * ((size_t)n + 1));
        double *ds = (double *)malloc(sizeof(double) * ((size_t)n + 1));
        double *tmp = (double *)malloc(sizeof(double) * (size_t)D);
        double *qr = (double *)malloc(sizeof(double) * (size_t)D);
        double *go = (double *)malloc(sizeof(double) * (size_t)D);
        double *ov = (double *)malloc(sizeof(double) * (size_t)D);
        double *gq = (double *)malloc(sizeof(double) * (size_t)D);
        double *mq = (double *)malloc(sizeof(double) * (size_t)D);
        double *sq = (double *)malloc(sizeof(double) * (size_t)D);
        if (!kr || !vr || !gk || !gv || !mk || !mv || !sk || !pr || !ds || !tmp || !qr || !go || !ov || !gq ||
            !mq || !sq) {
            free(kr); free(vr); free(gk); free(gv); free(mk); free(mv); free(sk); free(pr); free(ds);
            free(tmp); free(qr); free(go); free(ov); free(gq); free(mq); free(sq);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            err = ORACLE_E_NOMEM;
            continue;
        }
        int bad = 0;
        for (int t = 0; t < n && !bad; ++t) {
            int page = block_table[(int64_t)b * W + t / page_size];
            if (page < 0 || page >= num_pages) { bad = 1; break; }
            int64_t src = (((int64_t)page * page_size + t % page_size) * Hkv + kh) * D;
            for (int d = 0; d < D; ++d) {
                tmp[d] = to_f64(k_cache, src + d, qkv_dtype);
                vr[(int64_t)t * D + d] = to_f64(v_cache, src + d, qkv_dtype);
            }
            rk_oracle_rope(tmp, D, (double)t, rope_theta, rope_scale, kr + (int64_t)t * D);
        }
        for (int g = 0; g < G && !bad; ++g) {
            const int h = kh * G + g;
            for (int s = 0; s < Sq; ++s) {
                const int p = position_ids[(int64_t)b * Sq + s];
                const int nv = p < 0 ? 0 : (p + 1 < n ? p + 1 : n);
                const int64_t qoff = (((int64_t)b * Hq + h) * Sq + s) * D;
                if (nv == 0) {  /* out = 0 does not depend on anything */
                    for (int d = 0; d < D; ++d) {
                        dq[qoff + d] = 0.0;
                        if (mag_dq) mag_dq[qoff + d] = 0.0;
                        if (sens_dq) sens_dq[qoff + d] = 0.0;
                    }
                    continue;
                }
                for (int d = 0; d < D; ++d) tmp[d] = to_f64(q, qoff + d, qkv_dtype);
                rk_oracle_rope(tmp, D, (double)p, rope_theta, rope_scale, qr);
                for (int d = 0; d < D; ++d) go[d] = to_f64(dout, qoff + d, dout_dtype);
                /* forward again: probabilities and the output */
                double m = -INFINITY;
                for (int t = 0; t < nv; ++t) {
                    double acc = 0.0;
                    const double *kt = kr + (int64_t)t * D;
                    for (int d = 0; d < D; ++d) acc += qr[d] * kt[d];
                    pr[t] = acc * sm_scale;
                    if (pr[t] > m) m = pr[t];
                }
                double sum = 0.0;
                for (int t = 0; t < nv; ++t) {
                    pr[t] = exp(pr[t] - m);
                    sum += pr[t];
                }
                for (int d = 0; d < D; ++d) ov[d] = 0.0;
                for (int t = 0; t < nv; ++t) {
                    pr[t] /= sum;
                    const double *vt = vr + (int64_t)t * D;
                    for (int d = 0; d < D; ++d) ov[d] += pr[t] * vt[d];
                }
                double Dq = 0.0, A = 0.0;
                for (int d = 0; d < D; ++d) {
                    Dq += go[d] * ov[d];
                    A += fabs(go[d] * ov[d]);
                }
                /* softmax gradient */
                for (int t = 0; t < nv; ++t) {
                    double dp = 0.0;
                    const double *vt = vr + (int64_t)t * D;
                    for (int d = 0; d < D; ++d) dp += go[d] * vt[d];
                    ds[t] = pr[t] * (dp - Dq);
                }
                /* dq' and its magnitudes; dk', dv accumulate over queries */
                for (int d = 0; d < D; ++d) { gq[d] = 0.0; mq[d] = 0.0; sq[d] = 0.0; }
                for (int t = 0; t < nv; ++t) {
                    const double *kt = kr + (int64_t)t * D;
                    double *gkt = gk + (int64_t)t * D, *gvt = gv + (int64_t)t * D;
                    double *mkt = mk + (int64_t)t * D, *mvt = mv + (int64_t)t * D;
                    double *skt = sk + (int64_t)t * D;
                    const double w = sm_scale * ds[t], aw = fabs(w), ws = sm_scale * pr[t] * A;
                    for (int d = 0; d < D; ++d) {
                        gq[d] += w * kt[d];
                        mq[d] += aw * fabs(kt[d]);
                        sq[d] += ws * fabs(kt[d]);
                        gkt[d] += w * qr[d];
                        mkt[d] += aw * fabs(qr[d]);
                        skt[d] += ws * fabs(qr[d]);
                        gvt[d] += pr[t] * go[d];
                        mvt[d] += pr[t] * fabs(go[d]);
                    }
                }
                /* back to the pre-rotation domain: dq = R(p)^T dq' */
                for (int d = 0; d < D; ++d) tmp[d] = gq[d];
                rk_oracle_rope(tmp, D, -(double)p, rope_theta, rope_scale, dq + qoff);
                for (int i = 0; i < half; ++i) {
                    const double a = mq[i] + mq[i + half], c = sq[i] + sq[i + half];
                    if (mag_dq) { mag_dq[qoff + i] = a; mag_dq[qoff + i + half] = a; }
                    if (sens_dq) { sens_dq[qoff + i] = c; sens_dq[qoff + i + half] = c; }
                }
            }
        }
        if (!bad) {
            /* write the row's pages: dk_t = R(t)^T dk'_t, dv_t; 0 past kv_len */
            const int npages = (n + page_size - 1) / page_size;
            for (int t = 0; t < npages * page_size; ++t) {
                int page = block_table[(int64_t)b * W + t / page_size];
                int64_t dst = (((int64_t)page * page_size + t % page_size) * Hkv + kh) * D;
                if (t < n) {
                    rk_oracle_rope(gk + (int64_t)t * D, D, -(double)t, rope_theta, rope_scale, dk + dst);
                    for (int d = 0; d < D; ++d) dv[dst + d] = gv[(int64_t)t * D + d];
                    for (int i = 0; i < half; ++i) {
                        const double a = mk[(int64_t)t * D + i] + mk[(int64_t)t * D + i + half];
                        const double c = sk[(int64_t)t * D + i] + sk[(int64_t)t * D + i + half];
                        if (mag_dk) { mag_dk[dst + i] = a; mag_dk[dst + i + half] = a; }
                        if (sens_dk) { sens_dk[dst + i] = c; sens_dk[dst + i + half] = c; }
                    }
                    if (mag_dv)
                        for (int d = 0; d < D; ++d) mag_dv[dst + d] = mv[(int64_t)t * D + d];
                } else {
                    for (int d = 0; d < D; ++d) {
                        dk[dst + d] = 0.0;
                        dv[dst + d] = 0.0;
                        if (mag_dk) mag_dk[dst + d] = 0.0;
                        if (mag_dv) mag_dv[dst + d] = 0.0;
                        if (sens_dk) sens_dk[dst + d] = 0.0;
                    }
                }
            }
        }
        free(kr); free(vr); free(gk); free(gv); free(mk); free(mv); free(sk); free(pr); free(ds);
        free(tmp); free(qr); free(go); free(ov); free(gq); free(mq); free(sq);
        if (bad) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            err = ORACLE_E_PAGE;
        }
    }
    return err;
}

/* Threads OpenMP will use for a parallel region (1 without OpenMP). */
int rk_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
