// compress.cu -- the write side of one layer group, on CUDA cores in fp32.
//
// Method passages (web pages about arXiv:2611.07025):
//   "LowRAM Paper: Amortised Values and Low-Rank Keys for KV Compression", "Step-by-step mental model
//     for one decoding session", step 1: at prefill RoPE is inverted, per-head MLPs map keys to
//     values, sparse residuals are stored for bad fits, and keys are compressed with low-rank bases
//     shared across the layer group; "Value cache amortisation in plain language": the per-token
//     reconstruction error decides which tokens keep a residual.
//   "LowRAM: Low-Rank Keys and Amortised Values for Composable KV Cache Compression at Test-Time",
//     Abstract: residuals only for the tokens the predictor reconstructs worst; composes with
//     quantisation.
// The error ranking decides which tokens are stored exactly, so the predictor runs in fp32 here
// (accurate expf) rather than on bf16 tensor-core operands.
#include "kernels.h"
#include "predict.cuh"

namespace lowram {

// ------------------------------------------------------------------------------------------------
// project: coef[row, n] = sum_k proj[n, k] * k_pre_cat[row, k], rows = B*T tokens, n < r.
// grid (rows/32, r/256).  Keys given after RoPE are rotated back on load.
// ------------------------------------------------------------------------------------------------
template <typename TA>
struct KeyLoader {
    const TA* keys;  // [B*T, N]
    const int32_t* pos;
    const float* rcos;
    const float* rsin;
    int64_t row0;
    int T, N, d, max_pos;
    bool post_rope;
    const int* Ps;   // positions of the tile's rows (shared memory)
    __device__ __forceinline__ float operator()(int t, int k) const {
        const int64_t row = row0 + t;
        const TA* kr = keys + row * N;
        if (!post_rope) return ld(kr, k);
        const int half = d / 2, i = k % d;
        const int p = Ps[t];
        if (i < half) {
            const float c = rcos[(int64_t)i * max_pos + p], s = rsin[(int64_t)i * max_pos + p];
            return ld(kr, k) * c + ld(kr, k + half) * s;   // rotate by -angle: x cos + y sin
        }
        const int i0 = i - half;
        const float c = rcos[(int64_t)i0 * max_pos + p], s = rsin[(int64_t)i0 * max_pos + p];
        return ld(kr, k) * c - ld(kr, k - half) * s;       // y cos - x sin
    }
};

template <typename TA>
__global__ void __launch_bounds__(kTileThreads) project_kernel(CompressArgs a, int64_t rows_total) {
    extern __shared__ float sm[];
    const auto& s = a.s;
    const int N = s.G * s.H_kv * s.d, r = s.r;
    const int64_t row0 = (int64_t)blockIdx.x * kTileRows;
    const int n0 = blockIdx.y * 256;
    float* As = sm;
    float* Bs = As + kTileRows * kStride;
    int* Ps = (int*)(Bs + 8 * 32 * kStride);
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
    if (tid < kTileRows) {
        int64_t row = row0 + tid;
        int p = 0;
        if (row < rows_total) {
            p = a.pos ? a.pos[row] : (int)(row % s.T);
            if (s.keys_post_rope && (p < 0 || p >= s.max_pos)) {
                flag(a.check, LOWRAM_CHECK_POS_RANGE);
                p = p < 0 ? 0 : s.max_pos - 1;
            }
        }
        Ps[tid] = p;
    }
    __syncthreads();
    // rows beyond the end read row 0 of the tile's clamp (their output is not written)
    const int64_t last = rows_total - 1;
    KeyLoader<TA> kl{(const TA*)a.keys, a.pos, a.rope_cos, a.rope_sin, row0, s.T, N, s.d, s.max_pos,
                     s.keys_post_rope != 0, Ps};
    float acc[4][8];
    zero_acc<8>(acc);
    tile_product<8>([&](int t, int k) { return row0 + t <= last ? kl(t, k) : 0.0f; },
                    [&](int n, int k) { return a.proj[(int64_t)n * N + k]; }, N, n0, r, As, Bs, acc);

    // store: f32 / bf16 round to nearest even / int4 with fp16 scale per 32 columns (one warp = one group)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t row = row0 + ty * 4 + u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int n = n0 + tx + 32 * j;
            const int n_base = n0 + 32 * j;          // warp-uniform
            if (n_base >= r) continue;
            const float x = acc[u][j];
            if (s.coef_dtype == LOWRAM_INT4_G32) {
                float amax = warp_max(fabsf(x));
                __half sh = __float2half_rn(amax / 7.0f);
                float sc = __half2float(sh);
                int code = 0;
                if (sc > 0.0f) code = max(-7, min(7, __float2int_rn(x / sc)));
                int other = __shfl_down_sync(0xffffffffu, code, 1);
                if (row < rows_total) {
                    if ((tx & 1) == 0)
                        ((uint8_t*)a.coef_out)[row * (r / 2) + n / 2] = (uint8_t)((code & 0xF) | ((other & 0xF) << 4));
                    if (tx == 0) ((__half*)a.coef_scale_out)[row * (r / 32) + n / 32] = sh;
                }
            } else if (row < rows_total && n < r) {
                if (s.coef_dtype == LOWRAM_BF16) ((__nv_bfloat16*)a.coef_out)[row * r + n] = __float2bfloat16_rn(x);
                else ((float*)a.coef_out)[row * r + n] = x;
            }
        }
    }
}

// ------------------------------------------------------------------------------------------------
// predict + error: err[b, h, t] = || v[b, t, h, :] - MLP(k_pre from the stored coefficients) ||_2
// grid (T/32, H_kv, B)
// ------------------------------------------------------------------------------------------------
template <typename TA, typename CoefV, int NJm>
__global__ void __launch_bounds__(kTileThreads) predict_err_kernel(CompressArgs a, int layer, CoefV coef, float* err) {
    extern __shared__ float sm[];
    const auto& s = a.s;
    const int d = s.d, m = s.m, T = s.T;
    const int t0 = blockIdx.x * kTileRows, h = blockIdx.y, b = blockIdx.z;
    float* As = sm;
    float* Bs = As + kTileRows * kStride;
    float* Ks = Bs + NJm * 32 * kStride;
    float* Vs = Ks + kTileRows * (kMaxD + 1);
    float* Hs = Vs + kTileRows * (kMaxD + 1);
    int64_t* Rows = (int64_t*)(Hs + kTileRows * (NJm * 32 + 1));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < kTileRows) Rows[tid] = t0 + tid < T ? (int64_t)b * T + t0 + tid : -1;
    __syncthreads();
    rebuild_rows<TA>(Rows, coef, s.r, (const TA*)a.basis[layer] + (int64_t)h * d * s.r, d, As, Bs, Ks);
    predict_from_keys<TA, NJm, true>((const TA*)a.w1[layer] + (int64_t)h * m * d,
                                     a.b1[layer] ? a.b1[layer] + (int64_t)h * m : nullptr,
                                     (const TA*)a.w2[layer] + (int64_t)h * d * m,
                                     a.b2[layer] ? a.b2[layer] + (int64_t)h * d : nullptr, d, m, As, Bs, Ks, Hs, Vs);
    const TA* V = (const TA*)a.values[layer];
    for (int u = 0; u < 4; ++u) {
        const int t = warp * 4 + u;
        if (t0 + t >= T) continue;
        const TA* vt = V + (((int64_t)b * T + t0 + t) * s.H_kv + h) * d;
        float ss = 0.0f;
        for (int i = lane; i < d; i += 32) {
            float df = ld(vt, i) - Vs[t * (d + 1) + i];
            ss = fmaf(df, df, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) err[((int64_t)b * s.H_kv + h) * T + t0 + t] = sqrtf(ss);
    }
}

// ------------------------------------------------------------------------------------------------
// residual rows: for the kept tokens, R = v - MLP(k_pre), stored f32 / bf16 / int8 + fp16 scale.
// grid (n_res/32, H_kv, B)
// ------------------------------------------------------------------------------------------------
template <typename TA, typename CoefV, int NJm>
__global__ void __launch_bounds__(kTileThreads) residual_rows_kernel(CompressArgs a, int layer, CoefV coef) {
    extern __shared__ float sm[];
    const auto& s = a.s;
    const int d = s.d, m = s.m, T = s.T, n_res = s.n_res;
    const int j0 = blockIdx.x * kTileRows, h = blockIdx.y, b = blockIdx.z;
    float* As = sm;
    float* Bs = As + kTileRows * kStride;
    float* Ks = Bs + NJm * 32 * kStride;
    float* Vs = Ks + kTileRows * (kMaxD + 1);
    float* Hs = Vs + kTileRows * (kMaxD + 1);
    int64_t* Rows = (int64_t*)(Hs + kTileRows * (NJm * 32 + 1));
    int* Tok = (int*)(Rows + kTileRows);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t bh = (int64_t)b * s.H_kv + h;
    const int32_t* ridx = a.res_idx_out[layer] + bh * n_res;
    if (tid < kTileRows) {
        int j = j0 + tid;
        int t = j < n_res ? ridx[j] : -1;
        Tok[tid] = t;
        Rows[tid] = t >= 0 ? (int64_t)b * T + t : -1;
    }
    __syncthreads();
    rebuild_rows<TA>(Rows, coef, s.r, (const TA*)a.basis[layer] + (int64_t)h * d * s.r, d, As, Bs, Ks);
    predict_from_keys<TA, NJm, true>((const TA*)a.w1[layer] + (int64_t)h * m * d,
                                     a.b1[layer] ? a.b1[layer] + (int64_t)h * m : nullptr,
                                     (const TA*)a.w2[layer] + (int64_t)h * d * m,
                                     a.b2[layer] ? a.b2[layer] + (int64_t)h * d : nullptr, d, m, As, Bs, Ks, Hs, Vs);
    const TA* V = (const TA*)a.values[layer];
    for (int u = 0; u < 4; ++u) {
        const int t = warp * 4 + u;
        const int tok = Tok[t];
        if (tok < 0) continue;
        const TA* vt = V + (((int64_t)b * T + tok) * s.H_kv + h) * d;
        const int64_t orow = bh * n_res + j0 + t;
        float x[kMaxD / 32];
        float amax = 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxD / 32; ++q) {
            int i = lane + 32 * q;
            x[q] = i < d ? ld(vt, i) - Vs[t * (d + 1) + i] : 0.0f;
            amax = fmaxf(amax, fabsf(x[q]));
        }
        if (s.res_dtype == LOWRAM_INT8_VEC) {
            amax = warp_max(amax);
            __half sh = __float2half_rn(amax / 127.0f);
            float sc = __half2float(sh);
#pragma unroll
            for (int q = 0; q < kMaxD / 32; ++q) {
                int i = lane + 32 * q;
                if (i < d) {
                    int code = sc > 0.0f ? max(-127, min(127, __float2int_rn(x[q] / sc))) : 0;
                    ((int8_t*)a.res_val_out[layer])[orow * d + i] = (int8_t)code;
                }
            }
            if (lane == 0) ((__half*)a.res_scale_out[layer])[orow] = sh;
        } else {
#pragma unroll
            for (int q = 0; q < kMaxD / 32; ++q) {
                int i = lane + 32 * q;
                if (i >= d) continue;
                if (s.res_dtype == LOWRAM_BF16) ((__nv_bfloat16*)a.res_val_out[layer])[orow * d + i] = __float2bfloat16_rn(x[q]);
                else ((float*)a.res_val_out[layer])[orow * d + i] = x[q];
            }
        }
    }
}

// ------------------------------------------------------------------------------------------------
// launchers
// ------------------------------------------------------------------------------------------------
template <int NJm>
static size_t predict_kernel_smem() {
    return sizeof(float) * predict_smem_floats(NJm) + sizeof(int64_t) * kTileRows + sizeof(int) * kTileRows + 64;
}

cudaError_t launch_project(const CompressArgs& a, cudaStream_t st) {
    const auto& s = a.s;
    const int64_t rows = (int64_t)s.B * s.T;
    if (rows == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * (kTileRows * kStride + 8 * 32 * kStride) + sizeof(int) * kTileRows + 64;
    dim3 grid((unsigned)cdiv(rows, kTileRows), (unsigned)cdiv(s.r, 256));
    cudaError_t e;
    if (s.act_dtype == LOWRAM_BF16) {
        auto k = project_kernel<__nv_bfloat16>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess) return e;
        k<<<grid, kTileThreads, smem, st>>>(a, rows);
    } else {
        auto k = project_kernel<float>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess) return e;
        k<<<grid, kTileThreads, smem, st>>>(a, rows);
    }
    return cudaGetLastError();
}

template <typename TA, typename CoefV, int NJm>
static cudaError_t pe_go(const CompressArgs& a, int layer, CoefV coef, float* err, cudaStream_t st) {
    const size_t smem = predict_kernel_smem<NJm>();
    auto k = predict_err_kernel<TA, CoefV, NJm>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)cdiv(a.s.T, kTileRows), (unsigned)a.s.H_kv, (unsigned)a.s.B);
    k<<<grid, kTileThreads, smem, st>>>(a, layer, coef, err);
    return cudaGetLastError();
}

template <typename TA, typename CoefV, int NJm>
static cudaError_t rr_go(const CompressArgs& a, int layer, CoefV coef, cudaStream_t st) {
    const size_t smem = predict_kernel_smem<NJm>();
    auto k = residual_rows_kernel<TA, CoefV, NJm>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)cdiv(a.s.n_res, kTileRows), (unsigned)a.s.H_kv, (unsigned)a.s.B);
    k<<<grid, kTileThreads, smem, st>>>(a, layer, coef);
    return cudaGetLastError();
}

// The error ranking reads the STORED coefficients, exactly what the decode path will read.
cudaError_t launch_predict_err(const CompressArgs& a, int layer, float* err, cudaStream_t st) {
    const auto& s = a.s;
    if ((int64_t)s.B * s.T == 0) return cudaSuccess;
    const bool big = s.m > 128;
    if (s.coef_dtype == LOWRAM_INT4_G32) {
        CoefRowsInt4 c{(const uint8_t*)a.coef_out, (const __half*)a.coef_scale_out, s.r};
        if (s.act_dtype == LOWRAM_BF16)
            return big ? pe_go<__nv_bfloat16, CoefRowsInt4, 8>(a, layer, c, err, st) : pe_go<__nv_bfloat16, CoefRowsInt4, 4>(a, layer, c, err, st);
        return big ? pe_go<float, CoefRowsInt4, 8>(a, layer, c, err, st) : pe_go<float, CoefRowsInt4, 4>(a, layer, c, err, st);
    }
    if (s.coef_dtype == LOWRAM_BF16) {
        CoefRows<__nv_bfloat16> c{(const __nv_bfloat16*)a.coef_out, s.r};
        if (s.act_dtype == LOWRAM_BF16)
            return big ? pe_go<__nv_bfloat16, decltype(c), 8>(a, layer, c, err, st) : pe_go<__nv_bfloat16, decltype(c), 4>(a, layer, c, err, st);
        return big ? pe_go<float, decltype(c), 8>(a, layer, c, err, st) : pe_go<float, decltype(c), 4>(a, layer, c, err, st);
    }
    CoefRows<float> c{(const float*)a.coef_out, s.r};
    if (s.act_dtype == LOWRAM_BF16)
        return big ? pe_go<__nv_bfloat16, decltype(c), 8>(a, layer, c, err, st) : pe_go<__nv_bfloat16, decltype(c), 4>(a, layer, c, err, st);
    return big ? pe_go<float, decltype(c), 8>(a, layer, c, err, st) : pe_go<float, decltype(c), 4>(a, layer, c, err, st);
}

cudaError_t launch_residual_rows(const CompressArgs& a, int layer, cudaStream_t st) {
    const auto& s = a.s;
    if ((int64_t)s.B * s.n_res == 0) return cudaSuccess;
    const bool big = s.m > 128;
    if (s.coef_dtype == LOWRAM_INT4_G32) {
        CoefRowsInt4 c{(const uint8_t*)a.coef_out, (const __half*)a.coef_scale_out, s.r};
        if (s.act_dtype == LOWRAM_BF16)
            return big ? rr_go<__nv_bfloat16, CoefRowsInt4, 8>(a, layer, c, st) : rr_go<__nv_bfloat16, CoefRowsInt4, 4>(a, layer, c, st);
        return big ? rr_go<float, CoefRowsInt4, 8>(a, layer, c, st) : rr_go<float, CoefRowsInt4, 4>(a, layer, c, st);
    }
    if (s.coef_dtype == LOWRAM_BF16) {
        CoefRows<__nv_bfloat16> c{(const __nv_bfloat16*)a.coef_out, s.r};
        if (s.act_dtype == LOWRAM_BF16)
            return big ? rr_go<__nv_bfloat16, decltype(c), 8>(a, layer, c, st) : rr_go<__nv_bfloat16, decltype(c), 4>(a, layer, c, st);
        return big ? rr_go<float, decltype(c), 8>(a, layer, c, st) : rr_go<float, decltype(c), 4>(a, layer, c, st);
    }
    CoefRows<float> c{(const float*)a.coef_out, s.r};
    if (s.act_dtype == LOWRAM_BF16)
        return big ? rr_go<__nv_bfloat16, decltype(c), 8>(a, layer, c, st) : rr_go<__nv_bfloat16, decltype(c), 4>(a, layer, c, st);
    return big ? rr_go<float, decltype(c), 8>(a, layer, c, st) : rr_go<float, decltype(c), 4>(a, layer, c, st);
}

}  // namespace lowram
