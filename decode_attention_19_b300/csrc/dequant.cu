// dequant.cu -- int4 latent caches on the tensor-core path: an exact two-term bf16 split of the dequantised
// coefficients, and the matching column duplication of the layer's basis.
//
// Composing the low-rank key cache with quantisation ("LowRAM Paper: Amortised Values and Low-Rank Keys for KV
// Compression", the quantisation / eviction composition) stores the latent coefficients as int4 codes with one
// fp16 scale per 32 entries; a coefficient is code * scale.  That product has at most 14 significant bits (an
// 11-bit fp16 significand times a code of at most 3 bits), so it is the exact sum of two bf16 numbers:
//   hi = bf16(code * scale),  lo = bf16(code * scale - hi)   (the remainder has at most 7 significant bits).
// With A' = [hi | lo] (rank 2r) and B' = [W | W] the tensor-core kernels' product A' B'^T = (hi + lo) W^T
// equals C W^T exactly up to the fp32 accumulation order, so the bf16 kernels serve int4 caches unchanged.
#include "common.cuh"
#include "kernels.h"

namespace lowram {

namespace {

// One thread per 8 consecutive coefficients (4 bytes of codes, one scale): writes 8 hi values at column k and
// 8 lo values at column r + k of the row, 16 bytes each.
__global__ void int4_split_kernel(const uint32_t* __restrict__ codes, const __half* __restrict__ scales,
                                  int64_t rows, int r, __nv_bfloat16* __restrict__ out) {
    const int per_row = r / 8;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * per_row) return;
    const int64_t row = i / per_row;
    const int k = (int)(i - row * per_row) * 8;
    const uint32_t w = __ldg(codes + i);                       // entries k .. k+7, even entry in the low nibble
    const float sc = __half2float(__ldg(scales + row * (r / 32) + (k >> 5)));
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float x[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int nib = (int)((w >> (8 * e + 4 * t)) & 0xFu);
            x[t] = (float)(nib >= 8 ? nib - 16 : nib) * sc;     // exact in fp32
        }
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(x[0], x[1]);
        const float2 hf = __bfloat1622float2(h2);
        const __nv_bfloat162 l2 = __floats2bfloat162_rn(x[0] - hf.x, x[1] - hf.y);   // exact remainders
        hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
        lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + row * (int64_t)(2 * r));
    dst[k / 8] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    dst[(r + k) / 8] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// out[n] = [W[n] | W[n]] for the n rows of the basis, 16 bytes per thread.
__global__ void dup_cols_kernel(const uint4* __restrict__ W, int64_t rows, int r, uint4* __restrict__ out) {
    const int per_row = r / 8;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * per_row) return;
    const int64_t row = i / per_row;
    const int k = (int)(i - row * per_row);
    const uint4 v = __ldg(W + i);
    out[row * 2 * per_row + k] = v;
    out[row * 2 * per_row + per_row + k] = v;
}

}  // namespace

cudaError_t launch_int4_split(const void* codes, const void* scales, int64_t rows, int r, void* out,
                              cudaStream_t st) {
    const int64_t n = rows * (r / 8);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    int4_split_kernel<<<(unsigned)cdiv(n, threads), threads, 0, st>>>(
        (const uint32_t*)codes, (const __half*)scales, rows, r, (__nv_bfloat16*)out);
    return cudaGetLastError();
}

cudaError_t launch_dup_cols(const void* W, int64_t rows, int r, void* out, cudaStream_t st) {
    const int64_t n = rows * (r / 8);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    dup_cols_kernel<<<(unsigned)cdiv(n, threads), threads, 0, st>>>((const uint4*)W, rows, r, (uint4*)out);
    return cudaGetLastError();
}

}  // namespace lowram
