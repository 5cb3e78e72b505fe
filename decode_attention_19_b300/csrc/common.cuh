// common.cuh -- small device helpers shared by the kernels of liblowram.so (sm_103a).
//
// Element access for the storage formats, the sticky device check word, warp reductions, and the
// order-preserving float -> uint32 map used by the exact top-S selection.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

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

// ------------------------------------------------------------------------------------------------
// programmatic dependent launch: a kernel launched with launch_pdl may start while the previous kernel in
// the stream is finishing; it must call grid_dep_wait() before it reads anything that kernel wrote.  A
// kernel calls grid_dep_trigger() to let its dependent start being scheduled (its memory is still only
// visible to the dependent after the dependent's grid_dep_wait()).
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace lowram
