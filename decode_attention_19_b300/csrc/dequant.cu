// dequant.cu -- int4 latent caches on the tensor-core path: by default an fp16 copy of the dequantised
// coefficients (and of the layer's basis), or with LOWRAM_FLAG_INT4_EXACT_SPLIT an exact two-term bf16 split of
// them and the matching column duplication of the basis.
//
// fp16 copy: code * scale rounded to fp16 (11-bit significand, 2^-12 relative); the basis, bf16, is exact in fp16
// down to magnitudes of 2^-14, and the tensor-core kernels' kind::f16 MMAs take fp16 A and B alike.
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

// out[n] = [W[n] | W[n]] for the rows of `batches` bases of `rows` rows each (basis c starts c * stride8 16-byte
// pieces into W; the outputs are packed), 16 bytes per thread.
__global__ void dup_cols_kernel(const uint4* __restrict__ W, int64_t rows, int batches, int64_t stride8, int r,
                                uint4* __restrict__ out) {
    const int per_row = r / 8;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * batches * per_row) return;
    const int64_t row = i / per_row;                 // packed row over all bases
    const int k = (int)(i - row * per_row);
    const int64_t c = row / rows, rl = row - c * rows;
    const uint4 v = __ldg(W + c * stride8 + rl * per_row + k);
    out[row * 2 * per_row + k] = v;
    out[row * 2 * per_row + per_row + k] = v;
}

// fp16(code * scale) of 8 coefficients packed in one 32-bit word (even entry in the low nibble).
__device__ __forceinline__ uint4 int4x8_to_f16(uint32_t w, float sc) {
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int n0 = (int)((w >> (8 * e)) & 0xFu), n1 = (int)((w >> (8 * e + 4)) & 0xFu);
        const __half2 h2 = __floats2half2_rn((float)(n0 >= 8 ? n0 - 16 : n0) * sc, (float)(n1 >= 8 ? n1 - 16 : n1) * sc);
        o[e] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Both fp16 copies of an int4 call in one launch: threads [0, rows r / 16) take 16 consecutive coefficients each
// (8 bytes of codes, the one scale of their group of 32, 32 bytes out); the threads after them copy the bases,
// 16 bytes each (every bf16 value whose magnitude is at least 2^-14 is exact in fp16).
__global__ void int4_f16_copies_kernel(const uint2* __restrict__ codes, const __half* __restrict__ scales, int64_t rows,
                                       int r, uint4* __restrict__ out, const uint4* __restrict__ W, int64_t wrows,
                                       int wbatches, int64_t wstride8, uint4* __restrict__ wout) {
    const int64_t n16 = rows * (r / 16);
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n16) {
        const int per_row = r / 16;
        const int64_t row = i / per_row;
        const int k = (int)(i - row * per_row) * 16;
        const uint2 w = __ldg(codes + i);
        const float sc = __half2float(__ldg(scales + row * (r / 32) + (k >> 5)));
        out[2 * i] = int4x8_to_f16(w.x, sc);
        out[2 * i + 1] = int4x8_to_f16(w.y, sc);
        return;
    }
    const int64_t j = i - n16;
    const int per_row = r / 8;
    if (j >= wrows * wbatches * per_row) return;
    const int64_t row = j / per_row;
    const int k = (int)(j - row * per_row);
    const int64_t c = row / wrows, rl = row - c * wrows;
    const uint4 v = __ldg(W + c * wstride8 + rl * per_row + k);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __half2 h2 = __floats2half2_rn(__uint_as_float(u[e] << 16), __uint_as_float(u[e] & 0xffff0000u));
        o[e] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    wout[j] = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

cudaError_t launch_int4_f16_copies(const void* codes, const void* scales, int64_t rows, int r, void* out,
                                   const void* W, int64_t wrows, int wbatches, int64_t wstride, void* wout,
                                   cudaStream_t st) {
    const int64_t n = rows * (r / 16) + wrows * wbatches * (r / 8);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    int4_f16_copies_kernel<<<(unsigned)cdiv(n, threads), threads, 0, st>>>(
        (const uint2*)codes, (const __half*)scales, rows, r, (uint4*)out, (const uint4*)W, wrows, wbatches,
        wstride / 8, (uint4*)wout);
    return cudaGetLastError();
}

cudaError_t launch_int4_split(const void* codes, const void* scales, int64_t rows, int r, void* out,
                              cudaStream_t st) {
    const int64_t n = rows * (r / 8);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    int4_split_kernel<<<(unsigned)cdiv(n, threads), threads, 0, st>>>(
        (const uint32_t*)codes, (const __half*)scales, rows, r, (__nv_bfloat16*)out);
    return cudaGetLastError();
}

cudaError_t launch_dup_cols(const void* W, int64_t rows, int r, void* out, cudaStream_t st, int batches,
                            int64_t batch_stride) {
    const int64_t n = rows * batches * (r / 8);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    dup_cols_kernel<<<(unsigned)cdiv(n, threads), threads, 0, st>>>((const uint4*)W, rows, batches, batch_stride / 8, r,
                                                                      (uint4*)out);
    return cudaGetLastError();
}

}  // namespace lowram
