// predict.cuh -- rebuild pre-RoPE keys and run the per-head value predictor for 32 token rows on
// CUDA cores in fp32.
//
// Key rebuild ("Asymmetric key compression with xKV", LowRAM Paper: Amortised Values and Low-Rank
// Keys for KV Compression): k_pre[t, i] = sum_k coef[row_t, k] * basis[h*d + i, k].
// Predictor ("Value cache amortisation in plain language", same page; LowRAM abstract: a lightweight
// per-head predictor): v[t] = w2[h] . SiLU(w1[h] . k_pre[t] + b1[h]) + b2[h].
#pragma once

#include "simt_tile.cuh"

namespace lowram {

constexpr int kMaxD = 128;

// Residual rows of any stored dtype, decoded at run time (the residual add is a small part of the work).
struct ResView {
    int dtype;  // LOWRAM_F32, LOWRAM_BF16, LOWRAM_INT8_VEC
    const void* val;
    const __half* scale;
    int d;
    __device__ __forceinline__ float get(int64_t row, int i) const {
        if (dtype == LOWRAM_BF16) return __bfloat162float(((const __nv_bfloat16*)val)[row * d + i]);
        if (dtype == LOWRAM_INT8_VEC) return (float)((const int8_t*)val)[row * d + i] * __half2float(scale[row]);
        return ((const float*)val)[row * d + i];
    }
};

// Shared-memory floats used by predict_rows (staging + K, H, V tiles) for a hidden width m <= NJm*32.
__host__ __device__ constexpr int predict_smem_floats(int NJm) {
    return tile_smem_floats(NJm) + 32 * (kMaxD + 1) * 2 + 32 * (NJm * 32 + 1);
}

// rows[t]: global coefficient row (b*T + token) or -1 for padding; padded rows produce zeros in K.
template <typename TA, typename CoefV>
__device__ __forceinline__ void rebuild_rows(const int64_t* rows, CoefV coef, int r, const TA* basis_h, int d,
                                             float* As, float* Bs, float* Ks) {
    float acc[4][4];
    zero_acc<4>(acc);
    tile_product<4>([&](int t, int k) { int64_t row = rows[t]; return row >= 0 ? coef.get(row, k) : 0.0f; },
                    [&](int n, int k) { return ld(basis_h, (int64_t)n * r + k); }, r, 0, d, As, Bs, acc);
    store_tile<4, false, true>(acc, Ks, d + 1, 0, d, nullptr);
    __syncthreads();
}

// K (already in Ks) -> H = SiLU(K w1^T + b1) -> V = H w2^T + b2, all in shared memory.
template <typename TA, int NJm, bool Accurate>
__device__ __forceinline__ void predict_from_keys(const TA* w1h, const float* b1h, const TA* w2h, const float* b2h,
                                                  int d, int m, float* As, float* Bs, const float* Ks, float* Hs,
                                                  float* Vs) {
    {
        float acc[4][NJm];
        zero_acc<NJm>(acc);
        tile_product<NJm>([&](int t, int k) { return Ks[t * (d + 1) + k]; },
                          [&](int n, int k) { return ld(w1h, (int64_t)n * d + k); }, d, 0, m, As, Bs, acc);
        store_tile<NJm, true, Accurate>(acc, Hs, m + 1, 0, m, b1h);
    }
    __syncthreads();
    {
        float acc[4][4];
        zero_acc<4>(acc);
        tile_product<4>([&](int t, int k) { return Hs[t * (m + 1) + k]; },
                        [&](int n, int k) { return ld(w2h, (int64_t)n * m + k); }, m, 0, d, As, Bs, acc);
        store_tile<4, false, Accurate>(acc, Vs, d + 1, 0, d, b2h);
    }
    __syncthreads();
}

}  // namespace lowram
