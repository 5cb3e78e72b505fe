/*
 * lowram_oracle.c -- plain, slow, fp64 CPU oracle for LowRAM compressed decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this file; only the
 * test suite, the smoke check and the CPU-baseline leg of the benchmark do.  It shares no code,
 * header, table or constant with the CUDA library: every step is written out here from its
 * definition, in double precision, in the order the method describes it.
 *
 * Sources (web pages about arXiv:2611.07025, cited by page title and section):
 *   [ABS]  "LowRAM: Low-Rank Keys and Amortised Values for Composable KV Cache Compression at
 *          Test-Time" -- arXiv listing, section Abstract.
 *   [ZH]   "LowRAM compresses KV cache with low-rank keys and amortised values" -- Key facts.
 *   [CB]   "LowRAM: predict values from keys, store only the misses" -- TL;DR, the flowchart
 *          "Values are mostly a function of keys", Key points.
 *   [EX]   "LowRAM Paper: Amortised Values and Low-Rank Keys for KV Compression" -- sections
 *          "Value cache amortisation in plain language", "Asymmetric key compression with xKV",
 *          "Step-by-step mental model for one decoding session".
 *
 * Where the pages leave a step open, this file takes the reading the library documents:
 *   - selection: per (sequence, kv-head) the S tokens with the largest key, where the key of a token
 *     is the largest scaled logit over the q-heads that share the kv-head; ties go to the lower
 *     token index; unselected tokens are left out of the softmax;
 *   - predictor: a 2-layer MLP with SiLU, input = the rebuilt pre-RoPE key;
 *   - RoPE: rotate-half, w_i = theta^(-2i/d), angle = position * w_i; q arrives already rotated;
 *   - residual ranking: L2 norm over d of (true value - predicted value), ties to the lower index.
 *
 * Layouts (the library's interface layouts; all arrays row-major, fp64 here):
 *   q      [B, H_q, d]            coef  [B, T, r]          pos [B, T] (NULL -> t)
 *   basis  [H_kv*d, r]            row h*d+i holds the r coefficients of key feature (h, i)
 *   w1     [H_kv, m, d]  b1 [H_kv, m]      hidden_j = sum_i w1[h,j,i] * k_pre[i] + b1[h,j]
 *   w2     [H_kv, d, m]  b2 [H_kv, d]      v_i      = sum_j w2[h,i,j] * silu(hidden_j) + b2[h,i]
 *   res_idx [B, H_kv, n_res] (strictly ascending token indices)   res_val [B, H_kv, n_res, d]
 *   out [B, H_q, d]  lse [B, H_q]  key [B, H_kv, T]  sel [B, H_kv, min(S,T)] (ascending)
 * q-head hq reads kv-head hq / (H_q / H_kv).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int B, T, H_q, H_kv, d, r, m, S, n_res;
    double rope_theta;
    double sm_scale; /* <= 0 selects 1/sqrt(d) */
} lro_dims;

enum { LRO_OK = 0, LRO_BAD_ARG = 1, LRO_BAD_INDEX = 2, LRO_NO_MEMORY = 3 };

static double scale_of(const lro_dims* D) { return D->sm_scale > 0 ? D->sm_scale : 1.0 / sqrt((double)D->d); }

/* ---------------------------------------------------------------------------------------------
 * Storage rounding.  Round-to-nearest-even from fp64, written from the IEEE 754 definitions of the
 * two 16-bit formats: bfloat16 keeps 8 significant bits and fp32's exponent range, binary16 keeps
 * 11 significant bits with normal exponents down to -14.
 * ------------------------------------------------------------------------------------------- */
static double round_to_format(double x, int sig_bits, int min_normal_exp, double max_finite) {
    if (x == 0.0 || isnan(x) || isinf(x)) return x;
    int e;
    frexp(x, &e);                         /* |x| = f * 2^e, 0.5 <= f < 1: leading bit has weight 2^(e-1) */
    int lead = e - 1;
    if (lead < min_normal_exp) lead = min_normal_exp; /* subnormal: fixed quantum */
    double quantum = ldexp(1.0, lead - (sig_bits - 1));
    double y = nearbyint(x / quantum) * quantum;      /* default rounding mode: to nearest, ties to even */
    if (fabs(y) > max_finite) y = copysign(INFINITY, x);
    return y;
}

double lro_round_bf16_scalar(double x) { return round_to_format(x, 8, -126, 3.38953138925153547590470800371487866880e+38); }
double lro_round_f16_scalar(double x) { return round_to_format(x, 11, -14, 65504.0); }
double lro_round_f32_scalar(double x) { return (double)(float)x; }

void lro_round_bf16(int64_t n, const double* x, double* y) { for (int64_t i = 0; i < n; ++i) y[i] = lro_round_bf16_scalar(x[i]); }
void lro_round_f32(int64_t n, const double* x, double* y) { for (int64_t i = 0; i < n; ++i) y[i] = lro_round_f32_scalar(x[i]); }

/* ---------------------------------------------------------------------------------------------
 * Quantised storage for the composed setting ("composes with quantisation and eviction" [ABS];
 * [EX] "Step-by-step mental model", step 3).  The pages give no format; the library's formats:
 *   int4 coefficients: groups of 32 consecutive entries of one row; scale = fp16(amax / 7);
 *     code = clamp(round_even(x / scale), -7, 7); two's-complement nibbles, even entry in the
 *     low nibble; amax = 0 gives scale 0 and codes 0.
 *   int8 residuals: one scale per d-vector; scale = fp16(amax / 127); code = clamp(round_even(x /
 *     scale), -127, 127).
 * ------------------------------------------------------------------------------------------- */
static int quant_code(double x, double scale, int qmax) {
    if (scale == 0.0) return 0;
    double c = nearbyint(x / scale);
    if (c > qmax) c = qmax;
    if (c < -qmax) c = -qmax;
    return (int)c;
}

void lro_quant_int4_g32(int64_t rows, int r, const double* x, uint8_t* packed, double* scales) {
    const int groups = r / 32;
    for (int64_t i = 0; i < rows; ++i) {
        for (int g = 0; g < groups; ++g) {
            const double* xs = x + i * r + g * 32;
            double amax = 0.0;
            for (int k = 0; k < 32; ++k) if (fabs(xs[k]) > amax) amax = fabs(xs[k]);
            double s = lro_round_f16_scalar(amax / 7.0);
            scales[i * groups + g] = s;
            for (int k = 0; k < 32; k += 2) {
                int lo = quant_code(xs[k], s, 7), hi = quant_code(xs[k + 1], s, 7);
                packed[i * (r / 2) + (g * 32 + k) / 2] = (uint8_t)((lo & 0xF) | ((hi & 0xF) << 4));
            }
        }
    }
}

void lro_dequant_int4_g32(int64_t rows, int r, const uint8_t* packed, const double* scales, double* x) {
    const int groups = r / 32;
    for (int64_t i = 0; i < rows; ++i)
        for (int k = 0; k < r; ++k) {
            uint8_t byte = packed[i * (r / 2) + k / 2];
            int nib = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            int code = nib >= 8 ? nib - 16 : nib;
            x[i * r + k] = code * scales[i * groups + k / 32];
        }
}

void lro_quant_int8_vec(int64_t rows, int d, const double* x, int8_t* codes, double* scales) {
    for (int64_t i = 0; i < rows; ++i) {
        double amax = 0.0;
        for (int k = 0; k < d; ++k) if (fabs(x[i * d + k]) > amax) amax = fabs(x[i * d + k]);
        double s = lro_round_f16_scalar(amax / 127.0);
        scales[i] = s;
        for (int k = 0; k < d; ++k) codes[i * d + k] = (int8_t)quant_code(x[i * d + k], s, 127);
    }
}

void lro_dequant_int8_vec(int64_t rows, int d, const int8_t* codes, const double* scales, double* x) {
    for (int64_t i = 0; i < rows; ++i)
        for (int k = 0; k < d; ++k) x[i * d + k] = codes[i * d + k] * scales[i];
}

/* ---------------------------------------------------------------------------------------------
 * RoPE.  [EX] "Asymmetric key compression with xKV": rotary position embedding is inverted before
 * the keys are compressed and applied again during attention.  Rotate-half convention: feature
 * pairs (i, i + d/2), frequency w_i = theta^(-2i/d), angle = pos * w_i.  inverse != 0 rotates by
 * the negative angle.
 * ------------------------------------------------------------------------------------------- */
void lro_rope_angles(int d, double theta, double pos, double* cos_out, double* sin_out) {
    for (int i = 0; i < d / 2; ++i) {
        double w = pow(theta, -2.0 * i / d);
        cos_out[i] = cos(pos * w);
        sin_out[i] = sin(pos * w);
    }
}

void lro_rope(int d, double theta, double pos, const double* x, double* y, int inverse) {
    const int h = d / 2;
    for (int i = 0; i < h; ++i) {
        double w = pow(theta, -2.0 * i / d);
        double c = cos(pos * w), s = sin(pos * w);
        if (inverse) s = -s;
        double a = x[i], b = x[i + h];
        y[i] = a * c - b * s;
        y[i + h] = b * c + a * s;
    }
}

/* Rotate n d-vectors, row i at position pos[i] (a batch of lro_rope calls). */
void lro_rope_rows(int64_t n, int d, double theta, const int32_t* pos, const double* x, double* y, int inverse) {
    for (int64_t i = 0; i < n; ++i) lro_rope(d, theta, (double)pos[i], x + i * d, y + i * d, inverse);
}

/* ---------------------------------------------------------------------------------------------
 * Key rebuild from the cross-layer low-rank factors ([EX] "Asymmetric key compression with xKV";
 * [ABS] "cross-layer low-rank key compression"): the pre-RoPE key of feature (h, i) of token t is
 * the dot product of the token's latent coefficients with row h*d+i of the layer's basis.
 * ------------------------------------------------------------------------------------------- */
static void rebuild_key(const lro_dims* D, const double* coef_row, const double* basis, int h, double* k_pre) {
    for (int i = 0; i < D->d; ++i) {
        const double* brow = basis + ((int64_t)h * D->d + i) * D->r;
        double acc = 0.0;
        for (int k = 0; k < D->r; ++k) acc += coef_row[k] * brow[k];
        k_pre[i] = acc;
    }
}

/* ---------------------------------------------------------------------------------------------
 * Value predictor ([ABS] "fits a lightweight per-head predictor"; [EX] "Value cache amortisation in
 * plain language": a small per-head MLP mapping each token's key vector to its value vector).
 * Two layers, SiLU(x) = x / (1 + e^-x) between them; biases may be NULL (zero).
 * ------------------------------------------------------------------------------------------- */
static double silu(double x) { return x / (1.0 + exp(-x)); }

void lro_mlp(int d, int m, const double* w1, const double* b1, const double* w2, const double* b2,
             const double* k_pre, double* hidden_scratch, double* v_out) {
    for (int j = 0; j < m; ++j) {
        double acc = b1 ? b1[j] : 0.0;
        for (int i = 0; i < d; ++i) acc += w1[(int64_t)j * d + i] * k_pre[i];
        hidden_scratch[j] = silu(acc);
    }
    for (int i = 0; i < d; ++i) {
        double acc = b2 ? b2[i] : 0.0;
        for (int j = 0; j < m; ++j) acc += w2[(int64_t)i * m + j] * hidden_scratch[j];
        v_out[i] = acc;
    }
}

/* ---------------------------------------------------------------------------------------------
 * Ordering used by both selections (tokens by score, and residual tokens by error): larger value
 * first, equal values by lower token index.  A full sort, so the prefix of length n is the exact
 * top-n set under that total order.
 * ------------------------------------------------------------------------------------------- */
typedef struct { double v; int32_t t; } scored;

static int by_value_desc_then_index(const void* pa, const void* pb) {
    const scored* a = (const scored*)pa;
    const scored* b = (const scored*)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->t > b->t) - (a->t < b->t);
}

static int by_index_asc(const void* pa, const void* pb) {
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a > b) - (a < b);
}

/* top-n of v[0..T) under the ordering above, returned ascending by token index in out[0..n). */
static int top_n_ascending(int T, const double* v, int n, int32_t* out) {
    scored* s = (scored*)malloc(sizeof(scored) * (size_t)(T > 0 ? T : 1));
    if (!s) return LRO_NO_MEMORY;
    for (int t = 0; t < T; ++t) { s[t].v = v[t]; s[t].t = t; }
    qsort(s, (size_t)T, sizeof(scored), by_value_desc_then_index);
    for (int j = 0; j < n; ++j) out[j] = s[j].t;
    qsort(out, (size_t)n, sizeof(int32_t), by_index_asc);
    free(s);
    return LRO_OK;
}

void lro_top_n(int T, const double* v, int n, int32_t* out) { top_n_ascending(T, v, n, out); }

static int check_dims(const lro_dims* D) {
    if (D->B < 0 || D->T < 0 || D->H_q <= 0 || D->H_kv <= 0 || D->d <= 0 || D->r <= 0 || D->m <= 0) return LRO_BAD_ARG;
    if (D->H_q % D->H_kv != 0 || D->d % 2 != 0 || D->S < 0 || D->n_res < 0 || D->n_res > D->T) return LRO_BAD_ARG;
    return LRO_OK;
}

/* ---------------------------------------------------------------------------------------------
 * lro_decode -- one decode-step attention of one layer for all B sequences, read from the
 * compressed cache.  Steps, in the method's order ([ABS]: "reconstructing only a selected subset
 * of KV pairs at each decoding step"; [ZH] Key facts; [CB] flowchart; [EX] "Step-by-step mental
 * model", step 2):
 *   1. rebuild every token's pre-RoPE key from the latent coefficients and the layer basis;
 *   2. rotate it at the token's position (RoPE re-applied during attention);
 *   3. scaled logits s[hq, t] = q_hq . k_t * scale for the q-heads of the kv-head;
 *   4. selection key = max over those q-heads; keep the top min(S, T) tokens;
 *   5. for the kept tokens only: value = MLP(pre-RoPE key), plus the stored residual if the token is
 *      one of the worst-reconstructed ones ([CB] flowchart "Residual store: worst tokens only");
 *   6. softmax over the kept tokens and the weighted sum of their values; lse = log sum exp.
 * key, sel may be NULL.  Returns LRO_BAD_INDEX if a residual index is out of range or not strictly
 * ascending.
 * ------------------------------------------------------------------------------------------- */
int lro_decode(const lro_dims* D, const double* q, const double* coef, const int32_t* pos,
               const double* basis, const double* w1, const double* b1, const double* w2, const double* b2,
               const int32_t* res_idx, const double* res_val,
               double* out, double* lse, double* key, int32_t* sel, int n_threads) {
    int st = check_dims(D);
    if (st) return st;
    const int B = D->B, T = D->T, Hq = D->H_q, Hkv = D->H_kv, d = D->d, r = D->r, m = D->m;
    const int g = Hq / Hkv, S_eff = D->S < T ? D->S : T, n_res = D->n_res;
    const double scale = scale_of(D);
    int status = LRO_OK;
    (void)r;
    if (n_res > 0 && (!res_idx || !res_val)) return LRO_BAD_ARG;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif

#pragma omp parallel for schedule(dynamic) collapse(2)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hkv; ++h) {
            double* k_pre = (double*)malloc(sizeof(double) * (size_t)T * d);
            double* s = (double*)malloc(sizeof(double) * (size_t)g * (T > 0 ? T : 1));
            double* kv = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
            int32_t* chosen = (int32_t*)malloc(sizeof(int32_t) * (size_t)(S_eff > 0 ? S_eff : 1));
            double* k_rot = (double*)malloc(sizeof(double) * d);
            double* v = (double*)malloc(sizeof(double) * (size_t)(S_eff > 0 ? S_eff : 1) * d);
            double* hid = (double*)malloc(sizeof(double) * m);
            if (!k_pre || !s || !kv || !chosen || !k_rot || !v || !hid) {
#pragma omp atomic write
                status = LRO_NO_MEMORY;
                goto done;
            }
            const int32_t* ridx = res_idx ? res_idx + ((int64_t)b * Hkv + h) * n_res : NULL;
            for (int j = 0; j < n_res; ++j)
                if (ridx[j] < 0 || ridx[j] >= T || (j > 0 && ridx[j] <= ridx[j - 1])) {
#pragma omp atomic write
                    status = LRO_BAD_INDEX;
                }

            /* steps 1-4, every token */
            for (int t = 0; t < T; ++t) {
                const double* crow = coef + ((int64_t)b * T + t) * D->r;
                double p = pos ? (double)pos[(int64_t)b * T + t] : (double)t;
                rebuild_key(D, crow, basis, h, k_pre + (int64_t)t * d);
                lro_rope(d, D->rope_theta, p, k_pre + (int64_t)t * d, k_rot, 0);
                double best = -INFINITY;
                for (int jq = 0; jq < g; ++jq) {
                    const double* qv = q + ((int64_t)b * Hq + h * g + jq) * d;
                    double dot = 0.0;
                    for (int i = 0; i < d; ++i) dot += qv[i] * k_rot[i];
                    s[(int64_t)jq * T + t] = dot * scale;
                    if (dot * scale > best) best = dot * scale;
                }
                kv[t] = best;
                if (key) key[((int64_t)b * Hkv + h) * T + t] = best;
            }

            /* step 4: the selected subset */
            top_n_ascending(T, kv, S_eff, chosen);
            if (sel) memcpy(sel + ((int64_t)b * Hkv + h) * S_eff, chosen, sizeof(int32_t) * (size_t)S_eff);

            /* step 5: values for the selected tokens only */
            const double* w1h = w1 + (int64_t)h * m * d;
            const double* w2h = w2 + (int64_t)h * d * m;
            const double* b1h = b1 ? b1 + (int64_t)h * m : NULL;
            const double* b2h = b2 ? b2 + (int64_t)h * d : NULL;
            for (int j = 0; j < S_eff; ++j) {
                int t = chosen[j];
                lro_mlp(d, m, w1h, b1h, w2h, b2h, k_pre + (int64_t)t * d, hid, v + (int64_t)j * d);
                for (int jr = 0; jr < n_res; ++jr)
                    if (ridx[jr] == t) {
                        const double* rv = res_val + (((int64_t)b * Hkv + h) * n_res + jr) * d;
                        for (int i = 0; i < d; ++i) v[(int64_t)j * d + i] += rv[i];
                        break;
                    }
            }

            /* step 6: softmax over the selected tokens, per q-head */
            for (int jq = 0; jq < g; ++jq) {
                const int hq = h * g + jq;
                double* o = out + ((int64_t)b * Hq + hq) * d;
                for (int i = 0; i < d; ++i) o[i] = 0.0;
                if (S_eff == 0) {
                    if (lse) lse[(int64_t)b * Hq + hq] = -INFINITY;
                    continue;
                }
                double mx = -INFINITY;
                for (int j = 0; j < S_eff; ++j) if (s[(int64_t)jq * T + chosen[j]] > mx) mx = s[(int64_t)jq * T + chosen[j]];
                double den = 0.0;
                for (int j = 0; j < S_eff; ++j) {
                    double p = exp(s[(int64_t)jq * T + chosen[j]] - mx);
                    den += p;
                    for (int i = 0; i < d; ++i) o[i] += p * v[(int64_t)j * d + i];
                }
                for (int i = 0; i < d; ++i) o[i] /= den;
                if (lse) lse[(int64_t)b * Hq + hq] = mx + log(den);
            }
        done:
            free(k_pre); free(s); free(kv); free(chosen); free(k_rot); free(v); free(hid);
        }
    }
    return status;
}

/* ---------------------------------------------------------------------------------------------
 * lro_project -- write side, latent coefficients ([EX] "Step-by-step mental model", step 1: RoPE
 * inverted, keys compressed with shared low-rank bases across the layer group; "Asymmetric key
 * compression with xKV").  k_cat [B, T, G*H_kv*d] holds the G layers' keys of each token side by
 * side (layer-major, then head, then feature).  If keys_post_rope != 0 each d-slice is first
 * rotated back by its token's position.  proj [r, G*H_kv*d]: the caller's left inverse of the
 * group's stacked bases.  coef[b, t, k] = sum_n proj[k, n] * k_pre_cat[b, t, n], unrounded.
 * ------------------------------------------------------------------------------------------- */
int lro_project(int B, int T, int G, int H_kv, int d, int r, const double* k_cat, const int32_t* pos,
                int keys_post_rope, double theta, const double* proj, double* coef, int n_threads) {
    if (B < 0 || T < 0 || G <= 0 || H_kv <= 0 || d <= 0 || d % 2 || r <= 0) return LRO_BAD_ARG;
    const int64_t N = (int64_t)G * H_kv * d;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int status = LRO_OK;
#pragma omp parallel for schedule(dynamic) collapse(2)
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t) {
            double* kp = (double*)malloc(sizeof(double) * (size_t)N);
            if (!kp) {
#pragma omp atomic write
                status = LRO_NO_MEMORY;
                continue;
            }
            const double* kr = k_cat + ((int64_t)b * T + t) * N;
            double p = pos ? (double)pos[(int64_t)b * T + t] : (double)t;
            for (int64_t off = 0; off < N; off += d) {
                if (keys_post_rope) lro_rope(d, theta, p, kr + off, kp + off, 1);
                else memcpy(kp + off, kr + off, sizeof(double) * d);
            }
            for (int k = 0; k < r; ++k) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) acc += proj[k * N + n] * kp[n];
                coef[((int64_t)b * T + t) * r + k] = acc;
            }
            free(kp);
        }
    return status;
}

/* ---------------------------------------------------------------------------------------------
 * lro_residuals -- write side, one layer: predictor error and the worst-token residual list
 * ([ABS]: "stores residuals only for the tokens it reconstructs worst"; [EX] "Value cache
 * amortisation": score reconstruction error per token, keep sparse residuals for the worst).
 * The predictor runs on keys rebuilt from the *stored* coefficients (coef_stored), i.e. on exactly
 * what decode will see.  err[b,h,t] = || v[b,t,h,:] - MLP(k_pre) ||_2.  The n_res largest errors
 * (ties to the lower index) are kept, ascending by index, with residual v - MLP(k_pre) (unrounded)
 * in res_raw.  v layout [B, T, H_kv, d].  err may be NULL.
 * ------------------------------------------------------------------------------------------- */
int lro_residuals(const lro_dims* D, const double* coef_stored, const double* v,
                  const double* basis, const double* w1, const double* b1, const double* w2, const double* b2,
                  int32_t* res_idx, double* res_raw, double* err, int n_threads) {
    int st = check_dims(D);
    if (st) return st;
    const int B = D->B, T = D->T, Hkv = D->H_kv, d = D->d, m = D->m, n_res = D->n_res;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int status = LRO_OK;
#pragma omp parallel for schedule(dynamic) collapse(2)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hkv; ++h) {
            double* vhat = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * d);
            double* e = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
            double* kp = (double*)malloc(sizeof(double) * d);
            double* hid = (double*)malloc(sizeof(double) * m);
            int32_t* worst = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_res > 0 ? n_res : 1));
            if (!vhat || !e || !kp || !hid || !worst) {
#pragma omp atomic write
                status = LRO_NO_MEMORY;
            } else {
                for (int t = 0; t < T; ++t) {
                    rebuild_key(D, coef_stored + ((int64_t)b * T + t) * D->r, basis, h, kp);
                    lro_mlp(d, m, w1 + (int64_t)h * m * d, b1 ? b1 + (int64_t)h * m : NULL,
                            w2 + (int64_t)h * d * m, b2 ? b2 + (int64_t)h * d : NULL, kp, hid, vhat + (int64_t)t * d);
                    const double* vt = v + (((int64_t)b * T + t) * Hkv + h) * d;
                    double ss = 0.0;
                    for (int i = 0; i < d; ++i) {
                        double diff = vt[i] - vhat[(int64_t)t * d + i];
                        ss += diff * diff;
                    }
                    e[t] = sqrt(ss);
                    if (err) err[((int64_t)b * Hkv + h) * T + t] = e[t];
                }
                top_n_ascending(T, e, n_res, worst);
                for (int j = 0; j < n_res; ++j) {
                    int t = worst[j];
                    res_idx[((int64_t)b * Hkv + h) * n_res + j] = t;
                    const double* vt = v + (((int64_t)b * T + t) * Hkv + h) * d;
                    double* rr = res_raw + (((int64_t)b * Hkv + h) * n_res + j) * d;
                    for (int i = 0; i < d; ++i) rr[i] = vt[i] - vhat[(int64_t)t * d + i];
                }
            }
            free(vhat); free(e); free(kp); free(hid); free(worst);
        }
    return status;
}

/* ---------------------------------------------------------------------------------------------
 * lro_dense_decode -- plain softmax attention of one decode query per q-head over an explicit,
 * uncompressed, already rotated K and V ([B, T, H_kv, d] each).  The comparator the compressed path
 * is measured against, and the closed form it must reduce to when nothing is compressed.
 * ------------------------------------------------------------------------------------------- */
int lro_dense_decode(int B, int T, int H_q, int H_kv, int d, double sm_scale, const double* q,
                     const double* k, const double* v, double* out, double* lse, int n_threads) {
    if (B < 0 || T < 0 || H_q <= 0 || H_kv <= 0 || H_q % H_kv || d <= 0) return LRO_BAD_ARG;
    const int g = H_q / H_kv;
    const double scale = sm_scale > 0 ? sm_scale : 1.0 / sqrt((double)d);
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int status = LRO_OK;
#pragma omp parallel for schedule(dynamic) collapse(2)
    for (int b = 0; b < B; ++b)
        for (int hq = 0; hq < H_q; ++hq) {
            const int h = hq / g;
            const double* qv = q + ((int64_t)b * H_q + hq) * d;
            double* o = out + ((int64_t)b * H_q + hq) * d;
            double* s = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
            if (!s) {
#pragma omp atomic write
                status = LRO_NO_MEMORY;
                continue;
            }
            double mx = -INFINITY;
            for (int t = 0; t < T; ++t) {
                const double* kt = k + (((int64_t)b * T + t) * H_kv + h) * d;
                double dot = 0.0;
                for (int i = 0; i < d; ++i) dot += qv[i] * kt[i];
                s[t] = dot * scale;
                if (s[t] > mx) mx = s[t];
            }
            for (int i = 0; i < d; ++i) o[i] = 0.0;
            double den = 0.0;
            for (int t = 0; t < T; ++t) {
                double p = exp(s[t] - mx);
                den += p;
                const double* vt = v + (((int64_t)b * T + t) * H_kv + h) * d;
                for (int i = 0; i < d; ++i) o[i] += p * vt[i];
            }
            if (T > 0) for (int i = 0; i < d; ++i) o[i] /= den;
            if (lse) lse[(int64_t)b * H_q + hq] = T > 0 ? mx + log(den) : -INFINITY;
            free(s);
        }
    return status;
}

/* Keys of a layer for every token, pre-RoPE: [B, T, H_kv, d] (used to build explicit caches). */
int lro_rebuild_keys(const lro_dims* D, const double* coef, const double* basis, double* k_pre, int n_threads) {
    int st = check_dims(D);
    if (st) return st;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel for schedule(static) collapse(2)
    for (int b = 0; b < D->B; ++b)
        for (int t = 0; t < D->T; ++t)
            for (int h = 0; h < D->H_kv; ++h)
                rebuild_key(D, coef + ((int64_t)b * D->T + t) * D->r, basis, h,
                            k_pre + (((int64_t)b * D->T + t) * D->H_kv + h) * D->d);
    return LRO_OK;
}

/* Predicted values for every token of a layer: [B, T, H_kv, d] from pre-RoPE keys [B, T, H_kv, d]. */
int lro_predict_values(int B, int T, int H_kv, int d, int m, const double* k_pre, const double* w1, const double* b1,
                       const double* w2, const double* b2, double* v_out, int n_threads) {
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int status = LRO_OK;
#pragma omp parallel for schedule(static) collapse(2)
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t) {
            double* hid = (double*)malloc(sizeof(double) * m);
            if (!hid) {
#pragma omp atomic write
                status = LRO_NO_MEMORY;
                continue;
            }
            for (int h = 0; h < H_kv; ++h) {
                int64_t off = (((int64_t)b * T + t) * H_kv + h) * d;
                lro_mlp(d, m, w1 + (int64_t)h * m * d, b1 ? b1 + (int64_t)h * m : NULL, w2 + (int64_t)h * d * m,
                        b2 ? b2 + (int64_t)h * d : NULL, k_pre + off, hid, v_out + off);
            }
            free(hid);
        }
    return status;
}

int lro_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
