// tail.cu -- the exact tail of a decode cache: the tokens generated after the prompt was compressed are kept as
// explicit, already rotated keys and their values, and attended exactly next to the compressed body
// ("LowRAM Paper: Amortised Values and Low-Rank Keys for KV Compression", step-by-step: compression applies to
// the prompt's cache; decoding appends new tokens).  Two pieces live here:
//   append: one token's K and V [B, H_kv, d] copied into row t of the tail buffers [B, T_cap, H_kv, d];
//   merge:  two attention results of the same queries over disjoint token sets (body and tail) combined through
//           their log-sum-exp:  W = max(lse_a, lse_b), a = e^(lse_a - W), b = e^(lse_b - W),
//           out = (a out_a + b out_b) / (a + b),  lse = W + log(a + b); an empty set has lse = -inf.
// The tail's attention itself is the comparator kernel (dense.cu) reading the buffers in place.
#include "common.cuh"
#include "kernels.h"

namespace lowram {

namespace {

// 16 bytes per thread; each of K and V is B * H_kv * d * elem_bytes bytes, rows of H_kv * d elements
__global__ void tail_append_kernel(int B, int T_cap, int row_bytes, int t, const uint4* __restrict__ k_new,
                                   const uint4* __restrict__ v_new, uint4* __restrict__ tail_k,
                                   uint4* __restrict__ tail_v) {
    const int per_row = row_bytes / 16;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * per_row) return;
    const int64_t b = i / per_row, c = i - b * per_row;
    const int64_t dst = (b * T_cap + t) * per_row + c;
    tail_k[dst] = __ldg(k_new + i);
    tail_v[dst] = __ldg(v_new + i);
}

// one warp per (sequence, q-head): every lane reads both log-sum-exps before lane 0 writes the merged one, and
// each feature is read and written by the same lane, so out and lse may alias out_a / lse_a (or the b pair).
__global__ void merge_attn_kernel(int BH, int d, const float* out_a, const float* lse_a, const float* out_b,
                                  const float* lse_b, float* out, float* lse) {
    const int64_t bh = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (bh >= BH) return;
    const float la = lse_a[bh], lb = lse_b[bh];
    const float W = fmaxf(la, lb);
    const bool any = W != -INFINITY;
    const float a = any ? __expf(la - W) : 0.0f, b = any ? __expf(lb - W) : 0.0f;
    const float inv = any ? 1.0f / (a + b) : 0.0f;
    for (int i = lane; i < d; i += 32) {
        const int64_t e = bh * d + i;
        out[e] = any ? (a * out_a[e] + b * out_b[e]) * inv : 0.0f;
    }
    __syncwarp();
    if (lse && lane == 0) lse[bh] = any ? W + logf(a + b) : -INFINITY;
}

}  // namespace

cudaError_t launch_tail_append(int B, int T_cap, int H_kv, int d, int elem_bytes, int t, const void* k_new,
                               const void* v_new, void* tail_k, void* tail_v, cudaStream_t st) {
    const int row_bytes = H_kv * d * elem_bytes;   // a multiple of 16: d is 64 or 128, elements of 2 or 4 bytes
    const int64_t n = (int64_t)B * (row_bytes / 16);
    if (n == 0) return cudaSuccess;
    tail_append_kernel<<<(unsigned)cdiv(n, 256), 256, 0, st>>>(B, T_cap, row_bytes, t, (const uint4*)k_new,
                                                              (const uint4*)v_new, (uint4*)tail_k, (uint4*)tail_v);
    return cudaGetLastError();
}

cudaError_t launch_merge_attn(int B, int H_q, int d, const float* out_a, const float* lse_a, const float* out_b,
                              const float* lse_b, float* out, float* lse, cudaStream_t st) {
    const int64_t n = (int64_t)B * H_q * 32;   // a warp per (sequence, q-head)
    if (n == 0) return cudaSuccess;
    merge_attn_kernel<<<(unsigned)cdiv(n, 256), 256, 0, st>>>(B * H_q, d, out_a, lse_a, out_b, lse_b, out, lse);
    return cudaGetLastError();
}

}  // namespace lowram
