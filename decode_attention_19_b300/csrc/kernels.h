// kernels.h -- host launchers of liblowram.so's kernels (internal; the public ABI is include/lowram.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/lowram.h"

namespace lowram {

void set_error_message(const char* fmt, ...);

// Internal coefficient dtype of the decode kernels' view of a shape: an fp16 copy of an int4 cache's dequantised
// coefficients in the workspace (the key and value passes then take fp16 operands: that copy, an fp16 copy of the
// basis, and the folded predictor weights in fp16).  Not a public lowram_dtype.
constexpr int32_t kCoefF16 = 100;

// Everything a decode call needs, already validated by the ABI layer.
struct DecodeArgs {
    lowram_decode_shape s;
    int g, S_eff;
    float scale;
    const void* q;
    const void* coef;
    const void* coef_scale;
    const int32_t* pos;
    const float* rope_cos;
    const float* rope_sin;
    const void* basis;
    const void* w1;
    const void* w2;
    const float* b1;
    const float* b2;
    const int32_t* res_idx;
    const void* res_val;
    const void* res_scale;
    float* out;
    float* lse;
    // scratch (carved from the workspace, or the caller's test hooks)
    float* key;
    int32_t* sel;
    float* partial;
    int n_chunks;        // partial chunks per (b, q-head)
    int PW;              // floats per partial record
    float* sall;         // [B, T, H_q] scaled logits of every q-head (tensor-core path), or null
    int32_t* hit;        // [B, H_kv, S_eff] residual row of each selected token or -1 (tensor-core path), or null
    void* fold;          // [copies, H_kv, m, r] bf16: w1[h] . basis_h, folded by the selection kernel (tensor-core
                         // path); one copy per sequence when a basis or a predictor is given per sequence
    long long wait_cycles;   // pipeline wait limit of the value pass in SM cycles; 0 = the default
    uint32_t* check;
};

// The value predictor's first layer folded into the basis (tensor-core value pass): F[h] = w1[h] . basis_h,
// [H_kv, m, r] bf16, made by spare CTAs of the selection kernel.
struct FoldArgs {
    const __nv_bfloat16* w1;      // [H_kv, m, d] (sequence c's at c * mlp_stride)
    const __nv_bfloat16* basis;   // [H_kv*d, r] (sequence c's at c * basis_stride)
    void* F;                      // [copies, H_kv, m, r] bf16 (fp16 with f16_out); null: no folding
    int H_kv, d, m, r;
    int copies;                   // 1, or B when a basis or a predictor is given per sequence
    int64_t basis_stride, mlp_stride;
    bool f16_out;
};

// Chunk (selected tokens per vregen CTA) used by each path.
constexpr int kSimtChunk = 32;

cudaError_t launch_rope_table(int d, double theta, int max_pos, float* cos_out, float* sin_out, cudaStream_t st);

// K1: selection keys of every token (CUDA-core path; any dtype)
cudaError_t launch_score_simt(const DecodeArgs& a, cudaStream_t st);
// K2: exact top-n per problem row (values [P][T] -> ascending indices [P][n]).  For the value pass it can also
// write hit[row][j] = position of token out[row][j] in the row's ascending residual list res_idx[row][0..n_res)
// or -1, checking the list (LOWRAM_CHECK_RES_INDEX into check).
// With `fold`, spare CTAs of the same launch also compute the folded weights (they do not wait for the kernel before).
cudaError_t launch_select_topn(int P, int T, int n_keep, const float* values, int32_t* out, cudaStream_t st,
                               int32_t* hit = nullptr, const int32_t* res_idx = nullptr,
                               int n_res = 0, uint32_t* check = nullptr, const FoldArgs* fold = nullptr);
size_t select_scratch_bytes(int P, int T, int n_keep);
// K3: value regeneration + softmax partials for selected chunks of 32 (CUDA-core path)
cudaError_t launch_vregen_simt(const DecodeArgs& a, cudaStream_t st);
// K4: merge partials -> out, lse
cudaError_t launch_merge(int B, int H_q, int n_chunks, int d, const float* partial, float* out, float* lse,
                         cudaStream_t st);

// Tensor-core path (bf16 caches): which of K1 / K3 cover a shape.  K3 on the tensor cores needs K1 on them
// too (it reads the scaled logits K1 stores) and writes partial records of tc_partial_width floats: the
// softmax-weighted value sum [d], the chunk's max logit and weight sum (the layout launch_merge reads).
bool tc_score_supported(const lowram_decode_shape& s);
bool tc_vregen_supported(const lowram_decode_shape& s);
int tc_partial_width(const lowram_decode_shape& s);
constexpr int kTcChunk = 128;
cudaError_t launch_score_tc(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_vregen_tc(const DecodeArgs& a, cudaStream_t st);
// int4 caches on the tensor-core path: the exact split of the dequantised coefficients into bf16 [hi | lo]
// ([rows, 2r]), and the basis with its columns repeated ([rows, 2r]); see dequant.cu
cudaError_t launch_int4_split(const void* codes, const void* scales, int64_t rows, int r, void* out, cudaStream_t st);
// int4 caches, default: out [rows, r] fp16 = fp16(code * scale); and an fp16 copy of bf16 basis rows (batched)
// fp16(code * scale) of an int4 cache [rows, r] and fp16 copies of `wbatches` bf16 bases [wrows, r] (basis c at
// c * wstride elements of W), in one launch.
cudaError_t launch_int4_f16_copies(const void* codes, const void* scales, int64_t rows, int r, void* out,
                                   const void* W, int64_t wrows, int wbatches, int64_t wstride, void* wout,
                                   cudaStream_t st);

cudaError_t launch_dup_cols(const void* W, int64_t rows, int r, void* out, cudaStream_t st, int batches = 1,
                            int64_t batch_stride = 0);

// Write side
struct CompressArgs {
    lowram_compress_shape s;
    const void* keys;
    const void* values[16];
    const float* proj;
    const int32_t* pos;
    const float* rope_cos;
    const float* rope_sin;
    const void* basis[16];
    const void* w1[16];
    const void* w2[16];
    const float* b1[16];
    const float* b2[16];
    void* coef_out;
    void* coef_scale_out;
    int32_t* res_idx_out[16];
    void* res_val_out[16];
    void* res_scale_out[16];
    float* err_out[16];
    float* err_scratch;
    uint32_t* check;
};
cudaError_t launch_project(const CompressArgs& a, cudaStream_t st);
cudaError_t launch_predict_err(const CompressArgs& a, int layer, float* err, cudaStream_t st);
cudaError_t launch_residual_rows(const CompressArgs& a, int layer, cudaStream_t st);

// Comparator (and the exact tail): token splits, and partial records per (sequence, q-head) that launch_dense
// writes; sequence b's K/V rows start at token b * Ts
int dense_splits(int B, int T, int H_kv, int H_q, int d, int dtype);   // token splits of one comparator call
int dense_records_max(int B, int T, int H_kv, int H_q, int d);       // most splits any dtype takes (workspace)
cudaError_t launch_dense(int B, int T, int Ts, int H_q, int H_kv, int d, int dtype, float scale, const void* q,
                         const void* k, const void* v, float* partial, int n_split, cudaStream_t st);

// Fitted basis (fit.cu): top-r eigenvectors of the RoPE-inverted keys' Gram matrix by subspace iteration
struct FitArgs {
    int B, T, G, H_kv, d, r, max_pos, post_rope, iters;
    bool bf16;
    uint64_t seed;
    const void* keys;            // [B, T, G, H_kv, d]
    const int32_t* pos;          // [B, T] or null
    const float* rope_cos;
    const float* rope_sin;
    float* proj_out;             // [r, G*H_kv*d]
    void* basis_out[16];         // G x [H_kv*d, r]
    void* scratch;               // fit_workspace_bytes
    uint32_t* check;
};
size_t fit_workspace_bytes(int64_t N, int D, int r);
cudaError_t launch_fit_basis(const FitArgs& f, cudaStream_t st);
// tc_fit.cu: float32 products of the fit on the tensor cores through an exact three-term bf16 split.
// launch_split3 writes the h, m, l terms of src [R, Cc] (float32, or bf16 when src_bf16; row stride lds), or of its
// transpose, as [out_rows, out_cols] bf16, zero past the source.  launch_split_gemm_tc sets C[M, N] (row stride ldc)
// = A B^T from the terms of A [Mp, Kp] and B [Np, Kp] (Mp and Np multiples of 128, Kp of 64); sym: A = B and only
// the tiles meeting the upper triangle run, each writing its upper entries and their mirrors.
cudaError_t launch_split3(const void* src, bool src_bf16, int R, int Cc, int64_t lds, bool transpose, int out_rows,
                          int out_cols, void* const out[3], cudaStream_t st);
cudaError_t launch_split_gemm_tc(const void* const a[3], const void* const b[3], int M, int N, int Mp, int Np, int Kp,
                                 bool sym, float* C, int ldc, uint32_t* check, cudaStream_t st);

// Exact tail: write one token's K and V [B, H_kv, d] into row t of [B, T_cap, H_kv, d]; merge two attention
// results over disjoint token sets through their log-sum-exp
cudaError_t launch_tail_append(int B, int T_cap, int H_kv, int d, int elem_bytes, int t, const void* k_new,
                               const void* v_new, void* tail_k, void* tail_v, cudaStream_t st);
cudaError_t launch_merge_attn(int B, int H_q, int d, const float* out_a, const float* lse_a, const float* out_b,
                              const float* lse_b, float* out, float* lse, cudaStream_t st);

}  // namespace lowram
