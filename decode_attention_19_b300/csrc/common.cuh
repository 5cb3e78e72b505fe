// common.cuh -- small device helpers shared by the kernels of liblowram.so (sm_103a).
//
// Element access for the storage formats, the sticky device check word, warp reductions, and the
// order-preserving float -> uint32 map used by the exact top-S selection.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lowram.h"

namespace lowram {

constexpr int kWarp = 32;

// ------------------------------------------------------------------------------------------------
// scalar loads from the storage dtypes
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float ld(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }

// Coefficient rows: float, bf16 or int4 (two codes per byte, even entry low, fp16 scale per 32).
template <typename T>
struct CoefRows {
    const T* base;
    int r;
    __device__ __forceinline__ float get(int64_t row, int k) const { return ld(base, row * r + k); }
};

struct CoefRowsInt4 {
    const uint8_t* codes;
    const __half* scales;
    int r;
    __device__ __forceinline__ float get(int64_t row, int k) const {
        uint8_t byte = codes[row * (r / 2) + (k >> 1)];
        int nib = (k & 1) ? (byte >> 4) : (byte & 0xF);
        int code = nib >= 8 ? nib - 16 : nib;
        return (float)code * __half2float(scales[row * (r / 32) + (k >> 5)]);
    }
};

// Residual rows: float, bf16, or int8 with one fp16 scale per row.
template <typename T>
struct ResRows {
    const T* base;
    int d;
    __device__ __forceinline__ float get(int64_t row, int i) const { return ld(base, row * d + i); }
};

struct ResRowsInt8 {
    const int8_t* codes;
    const __half* scales;
    int d;
    __device__ __forceinline__ float get(int64_t row, int i) const {
        return (float)codes[row * d + i] * __half2float(scales[row]);
    }
};

// ------------------------------------------------------------------------------------------------
// device check word: sticky bits in the first word of the caller's workspace
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void flag(uint32_t* check, uint32_t bit) {
    if (check) atomicOr(check, bit);
}

// ------------------------------------------------------------------------------------------------
// reductions
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Order-preserving map: a < b (as floats, no NaN) <=> key(a) < key(b) (as unsigned).
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + __expf(-x)); }
// SiLU with the fast reciprocal-based division (a few ulp; the tensor-core path's operands are bf16).  For
// x < -88 the denominator is +inf and the result is -0.
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__host__ __device__ constexpr int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace lowram
