/*
 * lowram.h -- C ABI of liblowram.so: LowRAM compressed-cache decode attention on B300 (sm_103a).
 *
 * The method (web pages about arXiv:2611.07025, cited by page title and section):
 *   - "LowRAM: Low-Rank Keys and Amortised Values for Composable KV Cache Compression at Test-Time"
 *     (arXiv listing), Abstract: values are predicted from keys by a lightweight per-head predictor
 *     fitted at test time, residuals are stored only for the worst-reconstructed tokens, keys get
 *     cross-layer low-rank compression, and each decode step reconstructs only a selected subset of
 *     KV pairs.  It composes with quantisation and eviction.
 *   - "LowRAM Paper: Amortised Values and Low-Rank Keys for KV Compression", sections "Value cache
 *     amortisation in plain language" (per-head MLP, per-token error, sparse residuals for the
 *     worst), "Asymmetric key compression with xKV" (a layer group shares the token-side factor;
 *     RoPE is inverted before compression and re-applied during attention), "Step-by-step mental
 *     model for one decoding session" (prefill compresses; decode rebuilds on demand).
 *   - "LowRAM: predict values from keys, store only the misses", flowchart "Values are mostly a
 *     function of keys" (keys -> predictor -> predicted values + residual store -> attention on a
 *     subset rebuilt per step).
 * The pages fix neither the selection rule nor the predictor's shape.  This library fixes them:
 * exact-score top-S per (sequence, kv-head), where a token's score is the largest scaled logit over
 * the q-heads sharing the kv-head (ties to the lower token index; unselected tokens are left out of
 * the softmax), and a 2-layer MLP with SiLU on the rebuilt pre-RoPE key.
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller, row-major and contiguous, 16-byte
 *     aligned (LOWRAM_ERR_ALIGNMENT otherwise).  Arrays of pointers (one per layer of a group) are
 *     HOST arrays holding device pointers.  The library allocates no device memory: scratch comes
 *     from the caller's workspace, sized by the matching *_workspace_size query.  The library sees
 *     pointers and sizes only, never buffer extents: every buffer must hold at least the layout its
 *     argument documents (the Python binding checks element counts and sizes before each call).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).  Calls enqueue
 *     work on it and return without synchronising, after checking their arguments on the host.
 *   - Errors are return codes; no C++ exception crosses the ABI.  lowram_last_error() gives a
 *     message for the calling thread's last failing call.  Kernels that find bad data (positions or
 *     residual indices out of range or unordered) clamp, keep going, and set a sticky word in the
 *     workspace that lowram_get_error() reads and clears.  No kernel waits on another CTA.
 *   - q-head hq reads kv-head hq / (H_q / H_kv).
 *   - Calls over B sequences that give each sequence its own grid row (decode, compress, the
 *     comparator and the exact tail's attention, the attention mass) take B <= 65535 per call, and
 *     calls over B*T token rows take B*T < 2^31 (LOWRAM_ERR_UNSUPPORTED otherwise); split larger
 *     batches into several calls.
 */
#ifndef LOWRAM_H
#define LOWRAM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LOWRAM_API __attribute__((visibility("default")))
#else
#define LOWRAM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LOWRAM_OK = 0,
    LOWRAM_ERR_INVALID_ARG = 1,   /* a size, a dtype or a required pointer is wrong */
    LOWRAM_ERR_ALIGNMENT = 2,     /* a pointer is not 16-byte aligned */
    LOWRAM_ERR_UNSUPPORTED = 3,   /* valid, but not built for this shape or dtype combination */
    LOWRAM_ERR_WORKSPACE = 4,     /* workspace NULL, misaligned or smaller than the query's answer */
    LOWRAM_ERR_CUDA = 5,          /* a CUDA runtime call or a launch failed */
    LOWRAM_ERR_DEVICE_CHECK = 6   /* lowram_get_error: a kernel found out-of-range or unordered data */
} lowram_status;

typedef enum {
    LOWRAM_F32 = 0,        /* float32 */
    LOWRAM_BF16 = 1,       /* bfloat16 */
    LOWRAM_INT4_G32 = 2,   /* coefficients: int4 codes, two per byte (even entry in the low nibble,
                              two's complement, -7..7), plus one fp16 scale per 32 consecutive
                              entries of a row: value = code * scale */
    LOWRAM_INT8_VEC = 3    /* residuals: int8 codes (-127..127) plus one fp16 scale per d-vector */
} lowram_dtype;

/* Bits of the device check word returned by lowram_get_error(). */
#define LOWRAM_CHECK_POS_RANGE 1u      /* a position was < 0 or >= max_pos (clamped) */
#define LOWRAM_CHECK_RES_INDEX 2u      /* a residual index was out of range or not strictly ascending */
#define LOWRAM_CHECK_TIMEOUT 4u        /* a tensor-core pipeline wait gave up (internal error; results invalid) */
#define LOWRAM_CHECK_NOT_PD 8u         /* lowram_fit_basis: an iterate lost rank (keys of rank < r); results invalid */
#define LOWRAM_CHECK_LAYOUT 16u        /* a tensor-core kernel's shared-memory layout did not fit its launch's
                                          allocation (internal error): the kernel returned at once, touching no
                                          memory; results invalid */

/* ---------------------------------------------------------------------------------------------
 * Decode: one layer, all B sequences.
 * ------------------------------------------------------------------------------------------- */
typedef struct {
    int32_t B;          /* sequences */
    int32_t T;          /* stored tokens per sequence (after eviction, if any) */
    int32_t H_q, H_kv;  /* query heads, kv-heads; H_q % H_kv == 0, H_q / H_kv <= 8 */
    int32_t d;          /* head dim: 64 or 128 */
    int32_t r;          /* latent rank of the layer group: multiple of 32, <= 1024 */
    int32_t m;          /* predictor hidden width: multiple of 32, <= 256 */
    int32_t S;          /* tokens selected per (sequence, kv-head); min(S, T) are used */
    int32_t n_res;      /* stored residuals per (sequence, kv-head), 0 <= n_res <= T */
    int32_t act_dtype;  /* q, basis, w1, w2: LOWRAM_F32 or LOWRAM_BF16 */
    int32_t coef_dtype; /* LOWRAM_F32, LOWRAM_BF16 (both need act_dtype equal) or LOWRAM_INT4_G32 */
    int32_t res_dtype;  /* LOWRAM_F32, LOWRAM_BF16 or LOWRAM_INT8_VEC */
    int32_t max_pos;    /* rows of the RoPE tables: positions are in [0, max_pos) */
    float sm_scale;     /* softmax scale; <= 0 selects 1/sqrt(d) */
    int64_t basis_batch_stride; /* elements from sequence b's basis to b+1's; 0: one basis for every sequence.
                                   Else >= H_kv*d*r and a multiple of 8 (16-byte rows for the TMA maps) */
    int64_t mlp_batch_stride;   /* elements from sequence b's w1 (and w2) to b+1's; 0: one predictor for every
                                   sequence.  Else >= H_kv*m*d and a multiple of 8; b1, b2 (when given) are then
                                   [B, H_kv, m] and [B, H_kv, d] */
    uint32_t flags;             /* LOWRAM_FLAG_* bits; 0 for the defaults */
} lowram_decode_shape;

/* int4 caches with bf16 activations on the tensor cores: split each dequantised coefficient exactly into two bf16
 * terms (rank 2r: twice the key-rebuild work and a 4r-byte copy per token) instead of the default single fp16 term
 * (code * scale rounded to fp16, 2^-12 relative; the basis and the folded predictor weights taken in fp16). */
#define LOWRAM_FLAG_INT4_EXACT_SPLIT 1u

/* Workspace bytes lowram_decode_attn needs for this shape (a multiple of 256). */
LOWRAM_API lowram_status lowram_decode_workspace_size(const lowram_decode_shape* shape, size_t* bytes);

/* *yes = 1 if calls of this shape run the key pass and the value regeneration on the tensor cores
 * (tcgen05; bf16 caches, and int4 caches with bf16 activations: these are first dequantised into an fp16 copy in
 * the workspace, or with LOWRAM_FLAG_INT4_EXACT_SPLIT and r <= 512 split exactly into two bf16 terms,
 * coefficient = hi + lo, stored as a rank-2r bf16 cache), 0 if they run on the CUDA cores (float32 caches and
 * shapes the tensor-core kernels do not cover). */
LOWRAM_API lowram_status lowram_decode_uses_tensor_cores(const lowram_decode_shape* shape, int32_t* yes);

/*
 * lowram_decode_attn -- decode-step attention read directly from the compressed cache.
 * Steps (LowRAM abstract; "Step-by-step mental model", step 2; "Asymmetric key compression with
 * xKV"; flowchart "Values are mostly a function of keys"):
 *   1. every token's pre-RoPE key k_pre[t, h, :] = basis[h*d : h*d+d, :] . coef[b, t, :];
 *   2. k = RoPE(k_pre) at the token's position (rotate-half: pair (i, i+d/2) rotated by
 *      pos * theta^(-2i/d), read from the cos/sin tables);
 *   3. s[hq, t] = sm_scale * q[b, hq] . k; selection key[h, t] = max over the q-heads of kv-head h;
 *   4. keep the min(S, T) tokens with the largest key (ties to the lower index);
 *   5. for kept tokens only: v = w2[h] . SiLU(w1[h] . k_pre + b1[h]) + b2[h], plus res_val[b, h, j]
 *      when t == res_idx[b, h, j];
 *   6. out[b, hq] = softmax over the kept tokens of s[hq, .] applied to their values.
 * Arguments (device pointers; shapes use the fields of *shape):
 *   q          [B, H_q, d] act_dtype, already rotated at the query's own position
 *   coef       [B, T, r] coef_dtype; LOWRAM_INT4_G32: [B, T, r/2] bytes
 *   coef_scale LOWRAM_INT4_G32 only: [B, T, r/32] fp16 scales; else NULL
 *   pos        [B, T] int32 original positions (eviction); NULL means position t
 *   rope_cos, rope_sin  [d/2, max_pos] float32 each (frequency-major), see lowram_rope_table
 *   basis      [H_kv*d, r] act_dtype (row h*d+i: latent coefficients of key feature (h, i)); with
 *              basis_batch_stride != 0, sequence b's basis starts basis_batch_stride elements after b-1's
 *   w1         [H_kv, m, d] act_dtype;  b1 [H_kv, m] float32 or NULL
 *   w2         [H_kv, d, m] act_dtype;  b2 [H_kv, d] float32 or NULL; with mlp_batch_stride != 0, sequence
 *              b's w1 and w2 start mlp_batch_stride elements after b-1's, and b1, b2 are [B, H_kv, m], [B, H_kv, d]
 *              (a predictor fitted per prompt: the LowRAM abstract fits the small per-head predictor at test
 *              time)
 *   res_idx    [B, H_kv, n_res] int32, strictly ascending per (b, h), in [0, T)
 *   res_val    [B, H_kv, n_res, d] res_dtype
 *   res_scale  LOWRAM_INT8_VEC only: [B, H_kv, n_res] fp16; else NULL
 *   out        [B, H_q, d] float32 (written)
 *   lse        [B, H_q] float32 log-sum-exp of the kept scaled logits, or NULL
 *   sel_out    [B, H_kv, min(S,T)] int32 kept token indices, ascending, or NULL
 *   key_out    [B, H_kv, T] float32 selection keys, or NULL
 * With T == 0 or S == 0, out is zero and lse is -inf.
 */
LOWRAM_API lowram_status lowram_decode_attn(const lowram_decode_shape* shape, const void* q, const void* coef,
                                 const void* coef_scale, const int32_t* pos, const float* rope_cos,
                                 const float* rope_sin, const void* basis, const void* w1, const void* w2,
                                 const float* b1, const float* b2, const int32_t* res_idx, const void* res_val,
                                 const void* res_scale, float* out, float* lse, int32_t* sel_out, float* key_out,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * lowram_decode_attn_events -- lowram_decode_attn, plus timing marks: when `events` (a host array of five
 * cudaEvent_t, any of them NULL) is given, events[0] is recorded on `stream` before the key pass,
 * events[1] after it, events[2] after the top-S selection, events[3] after value regeneration and
 * events[4] after the softmax merge.  Same kernels, same results.
 */
LOWRAM_API lowram_status lowram_decode_attn_events(const lowram_decode_shape* shape, const void* q, const void* coef,
                                                   const void* coef_scale, const int32_t* pos, const float* rope_cos,
                                                   const float* rope_sin, const void* basis, const void* w1,
                                                   const void* w2, const float* b1, const float* b2,
                                                   const int32_t* res_idx, const void* res_val, const void* res_scale,
                                                   float* out, float* lse, int32_t* sel_out, float* key_out,
                                                   void* workspace, size_t workspace_bytes, void* stream,
                                                   void* const* events);

/*
 * lowram_decode_attn_static -- lowram_decode_attn for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for integration.  Some callers cannot
 * call cudaMalloc or pass a workspace: code running inside another runtime's memory pool or arena that
 * owns every allocation, plug-ins loaded by a host that gives them no allocator, and code paths that
 * must not allocate after setup.  This call takes the same inputs and outputs as lowram_decode_attn
 * (same meaning, layouts and results) but allocates nothing: its scratch lives in one file-scope device
 * array of 32 MiB that every GPU which loads the library holds until the process exits.
 *   - Shapes whose lowram_decode_workspace_size() exceeds 32 MiB are rejected with
 *     LOWRAM_ERR_WORKSPACE (lowram_last_error() says how much they need).
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress, once per
 *     device, with that device current).  Make that first call before any stream capture.
 *   - Every call shares the one array per device, which keeps the last call's contents: calls that
 *     overlap on the GPU (different streams, or threads without ordering) race and corrupt each other's
 *     results.  Order them on one stream.
 *   - The device check word (LOWRAM_CHECK_* bits, including LOWRAM_CHECK_TIMEOUT) lives in the array too.
 *     It starts clear, stays set across calls once a kernel sets it, and is read and cleared by
 *     lowram_decode_attn_static_get_error().
 *   - A failed address lookup (for example one attempted during a stream capture) returns LOWRAM_ERR_CUDA
 *     and is retried by the next call.
 */
LOWRAM_API lowram_status lowram_decode_attn_static(const lowram_decode_shape* shape, const void* q, const void* coef,
                                                   const void* coef_scale, const int32_t* pos, const float* rope_cos,
                                                   const float* rope_sin, const void* basis, const void* w1,
                                                   const void* w2, const float* b1, const float* b2,
                                                   const int32_t* res_idx, const void* res_val, const void* res_scale,
                                                   float* out, float* lse, int32_t* sel_out, float* key_out,
                                                   void* stream);

/*
 * lowram_decode_attn_static_get_error -- the device check word of lowram_decode_attn_static's scratch on the
 * current device, as lowram_get_error() gives it for a workspace: synchronises `stream`, stores the word in
 * *check_word, clears it, and returns LOWRAM_ERR_DEVICE_CHECK if it was set (LOWRAM_OK if clear).  Allocates
 * nothing.  Order it after the static calls it reports on (same stream).
 */
LOWRAM_API lowram_status lowram_decode_attn_static_get_error(void* stream, uint32_t* check_word);

/*
 * lowram_rope_table -- cos/sin tables of the rotary embedding re-applied at decode ("Asymmetric key
 * compression with xKV": RoPE is inverted before compression and re-applied during attention).
 * cos_out[i * max_pos + p] = cos(p * theta^(-2i/d)), sin_out likewise, i < d/2, p < max_pos.
 * Angles are formed and evaluated in fp64 on the device, then rounded to float32.
 */
LOWRAM_API lowram_status lowram_rope_table(int32_t d, double theta, int32_t max_pos, float* cos_out, float* sin_out,
                                void* stream);

/* ---------------------------------------------------------------------------------------------
 * Compress: the write side for one layer group (prefill).
 * ------------------------------------------------------------------------------------------- */
typedef struct {
    int32_t B, T;          /* sequences; stored tokens per sequence */
    int32_t G;             /* layers in the group, 1..16 */
    int32_t H_kv, d, r, m; /* kv-heads, head dim (64/128), latent rank (multiple of 32), hidden width */
    int32_t n_res;         /* residuals kept per (sequence, layer, kv-head) */
    int32_t act_dtype;     /* keys, values, basis, w1, w2: LOWRAM_F32 or LOWRAM_BF16 */
    int32_t coef_dtype;    /* output coefficients: LOWRAM_F32, LOWRAM_BF16 or LOWRAM_INT4_G32 */
    int32_t res_dtype;     /* output residuals: LOWRAM_F32, LOWRAM_BF16 or LOWRAM_INT8_VEC */
    int32_t keys_post_rope;/* 1: keys are given rotated at their positions and are rotated back first */
    int32_t max_pos;       /* rows of the RoPE tables (used when keys_post_rope == 1) */
} lowram_compress_shape;

LOWRAM_API lowram_status lowram_compress_workspace_size(const lowram_compress_shape* shape, size_t* bytes);

/*
 * lowram_compress -- latent coefficients and worst-token residual lists of one layer group.
 * Steps (LowRAM abstract: residuals are kept only for the tokens the predictor rebuilds worst; "Value
 * cache amortisation in plain language": scores the per-token reconstruction error and keeps sparse
 * residuals for the worst predictions; "Step-by-step mental model", step 1; "Asymmetric key
 * compression with xKV"):
 *   1. (keys_post_rope) rotate each key back by its position; concatenate the G layers' keys of a
 *      token: k_cat[b, t, :] of length G*H_kv*d (layer, then head, then feature);
 *   2. coef[b, t, k] = sum_n proj[k, n] * k_cat[b, t, n], stored as coef_dtype (round to nearest
 *      even; int4: per-32 fp16 scale = amax/7, codes round(x/scale) clamped to +-7);
 *   3. per layer l: rebuild keys from the STORED coefficients, predict values with the layer's
 *      MLP in float32, err[b, h, t] = || values[l][b, t, h, :] - prediction ||_2;
 *   4. keep the n_res largest errors per (b, h) (ties to the lower index), ascending by index, with
 *      residual values - prediction stored as res_dtype (int8: per-vector fp16 scale = amax/127).
 * Arguments:
 *   keys       [B, T, G, H_kv, d] act_dtype (pre-RoPE unless keys_post_rope)
 *   values     host array of G device pointers, each [B, T, H_kv, d] act_dtype
 *   proj       [r, G*H_kv*d] float32: a left inverse of the group's stacked bases (proj . W = I)
 *   pos        [B, T] int32 or NULL (position t); rope_cos/rope_sin as for decode, NULL unless
 *              keys_post_rope
 *   basis, w1, w2   host arrays of G device pointers, layouts as for decode; b1, b2 host arrays of G
 *              float32 device pointers, or NULL
 *   coef_out   [B, T, r] coef_dtype (int4: [B, T, r/2] bytes); coef_scale_out [B, T, r/32] fp16 for
 *              int4, else NULL
 *   res_idx_out, res_val_out, res_scale_out   host arrays of G device pointers: [B, H_kv, n_res]
 *              int32; [B, H_kv, n_res, d] res_dtype; [B, H_kv, n_res] fp16 (int8 only, else NULL)
 *   err_out    host array of G device pointers to [B, H_kv, T] float32, or NULL
 */
LOWRAM_API lowram_status lowram_compress(const lowram_compress_shape* shape, const void* keys, const void* const* values,
                              const float* proj, const int32_t* pos, const float* rope_cos, const float* rope_sin,
                              const void* const* basis, const void* const* w1, const void* const* w2,
                              const float* const* b1, const float* const* b2, void* coef_out, void* coef_scale_out,
                              int32_t* const* res_idx_out, void* const* res_val_out, void* const* res_scale_out,
                              float* const* err_out, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Heavy hitters from accumulated attention: which prompt tokens an evicted cache keeps ("LowRAM:
 * predict values from keys, store only the misses", Key points; the eviction composed with the
 * compressed cache keeps sinks, recent tokens and heavy hitters).  The plan is made before
 * compression: compress the kept tokens' keys and values with their positions (pos).
 * ------------------------------------------------------------------------------------------- */
LOWRAM_API lowram_status lowram_attention_mass_workspace_size(int32_t B, int32_t T, int32_t W, int32_t H_q, int32_t H_kv,
                                                              int32_t d, int32_t dtype, size_t* bytes);

/*
 * lowram_attention_mass -- attention mass each of the T prompt tokens receives from an observation
 * window of W queries per sequence: mass[b, t] = sum_i sum_hq softmax_t(scale q_win[b, i, hq] .
 * k[b, t, hq / g])[t], every window query attending all T tokens (no causal mask), so each row sums
 * to W * H_q.  q_win [B, W, H_q, d] and k [B, T, H_kv, d] rotated, in dtype (LOWRAM_F32 or
 * LOWRAM_BF16); mass_out [B, T] float32; sm_scale <= 0 means 1/sqrt(d).  H_q/H_kv in {1, 2, 4, 7, 8}.
 * bf16 logits run on the tensor cores (fp32 accumulation), float32 ones on CUDA cores.  Device check
 * word (lowram_get_error): LOWRAM_CHECK_TIMEOUT if a tensor-core pipeline wait gave up (mass_out is
 * then incomplete).
 */
LOWRAM_API lowram_status lowram_attention_mass(int32_t B, int32_t T, int32_t W, int32_t H_q, int32_t H_kv, int32_t d,
                                               int32_t dtype, float sm_scale, const void* q_win, const void* k,
                                               float* mass_out, void* workspace, size_t workspace_bytes, void* stream);

LOWRAM_API lowram_status lowram_evict_plan_workspace_size(int32_t B, int32_t T, size_t* bytes);

/*
 * lowram_evict_plan -- keep_out [B, T_keep] int32, ascending per sequence: tokens t < n_sink and
 * t >= T - n_recent, and the T_keep - n_sink - n_recent others of largest mass (ties to the lower
 * index; exact selection).  Requires n_sink + n_recent <= T_keep <= T (or T_keep = T).
 */
LOWRAM_API lowram_status lowram_evict_plan(int32_t B, int32_t T, int32_t n_sink, int32_t n_recent, int32_t T_keep,
                                           const float* mass, int32_t* keep_out, void* workspace,
                                           size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Test-time fit of the value predictor (LowRAM abstract: the predictor is fitted at test time;
 * "Value cache amortisation in plain language": values are predicted from pre-RoPE keys).  Per
 * kv-head h the predictor v_hat = w2 silu(w1 k + b1) + b2 is fitted to the prompt's (pre-RoPE key,
 * value) pairs by full-batch Adam on loss_h = 1/(N d) sum_t || v_hat(k_t) - v_t ||^2, N = B*T.
 * Parameters are float32 master copies: w1 [H_kv, m, d], b1 [H_kv, m], w2 [H_kv, d, m],
 * b2 [H_kv, d] (decode takes w1, w2 in the activation dtype: round them after the fit).
 * keys, values [B, T, H_kv, d] in dtype (LOWRAM_F32 or LOWRAM_BF16); d is 64 or 128, m a multiple
 * of 32 up to 256.  Float32 accuracy throughout.
 * ------------------------------------------------------------------------------------------- */

/* Loss [H_kv] and gradient of every head's predictor at the given parameters (outputs shaped like the
 * parameters; overwritten).  One fused CUDA-core kernel, no workspace. */
LOWRAM_API lowram_status lowram_predictor_grad(int32_t B, int32_t T, int32_t H_kv, int32_t d, int32_t m, int32_t dtype,
                                               const void* keys, const void* values, const float* w1, const float* b1,
                                               const float* w2, const float* b2, float* loss_out, float* g_w1,
                                               float* g_b1, float* g_w2, float* g_b2, void* stream);

/* Workspace bytes lowram_fit_predictor needs for B*T prompt tokens: the gradient and Adam's two moments of every
 * parameter, and the scratch of the tensor-core products (the keys' bf16 terms in two layouts, about 12*B*T*H_kv*d
 * bytes, plus per-head activations and their terms, about 40*B*T*max(d, m) bytes). */
LOWRAM_API lowram_status lowram_fit_predictor_workspace_size(int32_t B, int32_t T, int32_t H_kv, int32_t d, int32_t m,
                                                             size_t* bytes);

/*
 * lowram_fit_predictor -- `steps` Adam steps (Kingma and Ba, bias-corrected; moments start at zero)
 * from the parameters given, updated in place.  losses_out [steps, H_kv] float32 (the loss before each
 * step) or NULL.  The five products of each step's forward and backward pass run on the tensor cores
 * with the float32 operands split exactly into three bf16 terms (six bf16 products, float32
 * accumulation); a pipeline timeout sets LOWRAM_CHECK_TIMEOUT in the workspace's check word
 * (lowram_get_error).  B*T is at most 2,097,120 prompt tokens, here and in
 * lowram_fit_predictor_workspace_size.  Errors: LOWRAM_ERR_INVALID_ARG (shape, steps < 0, lr <= 0,
 * beta outside [0, 1), eps <= 0, NULL pointers), LOWRAM_ERR_UNSUPPORTED (d, m, B*T),
 * LOWRAM_ERR_ALIGNMENT, LOWRAM_ERR_WORKSPACE.
 */
LOWRAM_API lowram_status lowram_fit_predictor(int32_t B, int32_t T, int32_t H_kv, int32_t d, int32_t m, int32_t dtype,
                                              const void* keys, const void* values, int32_t steps, float lr,
                                              float beta1, float beta2, float eps, float* w1, float* b1, float* w2,
                                              float* b2, float* losses_out, void* workspace, size_t workspace_bytes,
                                              void* stream);

/* ---------------------------------------------------------------------------------------------
 * Fitted basis: the group's shared low-rank key basis from the prompt's keys (before compress).
 * ------------------------------------------------------------------------------------------- */
/* Workspace bytes lowram_fit_basis needs (a multiple of 256; about 10*B*T*D + 10*D*D bytes, D = G*H_kv*d: the
 * float32 keys and their bf16 terms, the Gram matrix and its terms).
 * Uses shape fields B, T, G, H_kv, d, r, act_dtype, keys_post_rope and max_pos. */
LOWRAM_API lowram_status lowram_fit_basis_workspace_size(const lowram_compress_shape* shape, size_t* bytes);

/*
 * lowram_fit_basis -- the cross-layer SVD of the RoPE-inverted keys ("Asymmetric key compression with
 * xKV": the G layers' keys are stacked and factored together, RoPE inverted first), producing the
 * `proj` and `basis` that lowram_compress takes.  With k_cat [N = B*T, D = G*H_kv*d] the tokens'
 * stacked keys (rotated back by their positions when keys_post_rope), the rank-r subspace of k_cat's
 * largest singular values is the span of the top-r eigenvectors of k_cat^T k_cat.  They are found by
 * `iters` steps of subspace iteration from a Gaussian start drawn from `seed`, each orthonormalised
 * by Cholesky QR (fp64 Cholesky), and a final Cholesky QR; Q [D, r] then has orthonormal columns.
 * The basis within the subspace is not ordered by singular value (the rebuilt keys do not depend on
 * it).  Accuracy depends on the spectral gap: the subspace converges like (sigma_{r+1}/sigma_r)^(2 iters).
 * Arguments:
 *   keys       [B, T, G, H_kv, d] act_dtype; pos [B, T] int32 or NULL; rope_cos/rope_sin as for
 *              decode, NULL unless keys_post_rope
 *   proj_out   [r, D] float32 = Q^T (proj . stacked basis = I to float32 accuracy)
 *   basis_out  host array of G device pointers, each [H_kv*d, r] act_dtype: layer l's block of Q
 * Errors: LOWRAM_ERR_INVALID_ARG / _UNSUPPORTED (shape: r a multiple of 32, 32 <= r <= min(1024, D),
 * D <= 16384, B*T >= r), LOWRAM_ERR_ALIGNMENT, LOWRAM_ERR_WORKSPACE.  Device check word:
 * LOWRAM_CHECK_NOT_PD if an iterate lost rank (keys of rank below r: the r-th eigenvalue of the Gram
 * matrix under 1e-5 of the largest), LOWRAM_CHECK_POS_RANGE.
 */
LOWRAM_API lowram_status lowram_fit_basis(const lowram_compress_shape* shape, const void* keys, const int32_t* pos,
                                          const float* rope_cos, const float* rope_sin, int32_t iters, uint64_t seed,
                                          float* proj_out, void* const* basis_out, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Comparator: the same kernel family on an uncompressed cache.
 * ------------------------------------------------------------------------------------------- */
LOWRAM_API lowram_status lowram_dense_workspace_size(int32_t B, int32_t T, int32_t H_q, int32_t H_kv, int32_t d, size_t* bytes);

/*
 * lowram_dense_decode_attn -- softmax attention of one decode query per q-head over an explicit,
 * already rotated key cache and a value cache, both [B, T, H_kv, d] in dtype (LOWRAM_BF16 or
 * LOWRAM_F32); q [B, H_q, d] in dtype; out [B, H_q, d] float32; lse [B, H_q] float32 or NULL.
 * This is the baseline the compressed cache replaces (LowRAM abstract: the KV cache's footprint
 * caps batch size and throughput).
 */
LOWRAM_API lowram_status lowram_dense_decode_attn(int32_t B, int32_t T, int32_t H_q, int32_t H_kv, int32_t d, int32_t dtype,
                                       float sm_scale, const void* q, const void* k, const void* v, float* out,
                                       float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Exact tail (LowRAM Paper: Amortised Values and Low-Rank Keys for KV Compression, step-by-step:
 * the prompt's cache is compressed; tokens decoded afterwards are appended).  The tokens generated
 * after compression stay explicit: their already rotated keys and their values live in tail buffers
 * tail_k, tail_v [B, T_cap, H_kv, d] (dtype), the same length t_len in every sequence.  A decode
 * step attends the compressed body (lowram_decode_attn with lse) and the tail
 * (lowram_tail_decode_attn), then merges the two with lowram_merge_attn; the result is attention
 * over body and tail together.
 * ------------------------------------------------------------------------------------------- */

/*
 * lowram_tail_append -- write one decoded token's rotated keys k_new and values v_new, each
 * [B, H_kv, d] in dtype (LOWRAM_BF16 or LOWRAM_F32), into row t (0 <= t < T_cap) of every
 * sequence's tail buffers.  d is 64 or 128; all pointers 16-byte aligned device memory owned by
 * the caller.  Errors: LOWRAM_ERR_INVALID_ARG (shape, dtype, t out of range, NULL pointer),
 * LOWRAM_ERR_ALIGNMENT.
 */
LOWRAM_API lowram_status lowram_tail_append(int32_t B, int32_t T_cap, int32_t H_kv, int32_t d, int32_t dtype, int32_t t,
                                            const void* k_new, const void* v_new, void* tail_k, void* tail_v,
                                            void* stream);

/*
 * lowram_tail_decode_attn -- softmax attention of q [B, H_q, d] (dtype) over the first t_len rows
 * (0 <= t_len <= T_cap) of the tail buffers, read in place; out [B, H_q, d] float32, lse [B, H_q]
 * float32 or NULL (-inf and a zero output when t_len = 0).  sm_scale <= 0 means 1/sqrt(d).  The
 * workspace is lowram_dense_workspace_size(B, t_len, H_q, H_kv, d) bytes.  Same kernels and errors
 * as lowram_dense_decode_attn.
 */
LOWRAM_API lowram_status lowram_tail_decode_attn(int32_t B, int32_t T_cap, int32_t t_len, int32_t H_q, int32_t H_kv,
                                                 int32_t d, int32_t dtype, float sm_scale, const void* q,
                                                 const void* tail_k, const void* tail_v, float* out, float* lse,
                                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * lowram_merge_attn -- combine two attention results of the same queries over disjoint token sets:
 * with W = max(lse_a, lse_b), a = exp(lse_a - W), b = exp(lse_b - W):
 *   out = (a out_a + b out_b) / (a + b),  lse = W + log(a + b);
 * an empty set has lse = -inf (both empty: out = 0, lse = -inf).  out_*, out [B, H_q, d] float32;
 * lse_*, lse [B, H_q] float32 (lse may be NULL).  out may be out_a or out_b and lse may be lse_a or
 * lse_b (in-place merge).  Errors: LOWRAM_ERR_INVALID_ARG, LOWRAM_ERR_ALIGNMENT.
 */
LOWRAM_API lowram_status lowram_merge_attn(int32_t B, int32_t H_q, int32_t d, const float* out_a, const float* lse_a,
                                           const float* out_b, const float* lse_b, float* out, float* lse,
                                           void* stream);

/* ---------------------------------------------------------------------------------------------
 * Status
 * ------------------------------------------------------------------------------------------- */
/* Synchronises `stream`, returns the device check word accumulated in `workspace` since it was last
 * cleared (LOWRAM_CHECK_* bits; 0 = no bad data), and clears it.  A fresh workspace must have its first
 * 256 bytes zeroed once (lowram_clear_error) before its first use. */
LOWRAM_API lowram_status lowram_get_error(void* workspace, void* stream, uint32_t* check_word);
/* Enqueues a clear of the device check word in `workspace`. */
LOWRAM_API lowram_status lowram_clear_error(void* workspace, void* stream);
LOWRAM_API const char* lowram_status_string(lowram_status status);
/* Message for the calling thread's most recent failing call ("" if none). */
LOWRAM_API const char* lowram_last_error(void);
/* Library version: major * 10000 + minor * 100 + patch. */
LOWRAM_API int32_t lowram_version(void);

/*
 * lowram_set_wait_limit -- testing aid for the failure path of the tensor-core value pass (no counterpart on
 * the pages).  Every pipeline wait of that kernel (TMA stage landed, MMA done) gives up after `cycles` SM
 * clock cycles; 0 restores the default (~1 s at 2 GHz).  A limit shorter than a wait legitimately takes makes
 * the kernel give up on purpose: it then drains what it issued, frees its tensor memory, returns, and sets
 * LOWRAM_CHECK_TIMEOUT in the workspace's check word; that call's out and lse are invalid.  Process-wide; not
 * thread-safe against concurrent decode calls.  Errors: LOWRAM_ERR_INVALID_ARG for cycles < 0.
 */
LOWRAM_API lowram_status lowram_set_wait_limit(int64_t cycles);

#ifdef __cplusplus
}
#endif
#endif /* LOWRAM_H */
