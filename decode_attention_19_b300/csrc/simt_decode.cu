// simt_decode.cu -- decode-path kernels on CUDA cores: RoPE tables, selection keys (K1), value
// regeneration with softmax partials (K3), and the split-softmax merge (K4).
//
// Method passages (web pages about arXiv:2611.07025):
//   "LowRAM: Low-Rank Keys and Amortised Values for Composable KV Cache Compression at Test-Time",
//     Abstract: reconstruct only a selected subset of KV pairs at each decoding step.
//   "LowRAM Paper: Amortised Values and Low-Rank Keys for KV Compression", "Asymmetric key compression
//     with xKV" (low-rank keys, RoPE re-applied during attention) and "Value cache amortisation in
//     plain language" (values regenerated from keys plus residuals for the worst tokens).
// The float32 cache uses these kernels for the whole path; bf16 / int4 caches use the tensor-core
// kernels of tc_decode.cu for K1 and K3 and share K2 and K4.
#include "kernels.h"
#include "predict.cuh"

namespace lowram {

// ------------------------------------------------------------------------------------------------
// RoPE tables: cos/sin(p * theta^(-2i/d)) formed and evaluated in fp64, stored [d/2][max_pos] fp32.
// ------------------------------------------------------------------------------------------------
__global__ void rope_table_kernel(int d, double theta, int max_pos, float* cos_out, float* sin_out) {
    const int i = blockIdx.y;
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= max_pos) return;
    const double w = pow(theta, -2.0 * (double)i / (double)d);
    double s, c;
    sincos((double)p * w, &s, &c);
    cos_out[(int64_t)i * max_pos + p] = (float)c;
    sin_out[(int64_t)i * max_pos + p] = (float)s;
}

cudaError_t launch_rope_table(int d, double theta, int max_pos, float* cos_out, float* sin_out, cudaStream_t st) {
    dim3 grid((unsigned)cdiv(max_pos, 256), (unsigned)(d / 2));
    rope_table_kernel<<<grid, 256, 0, st>>>(d, theta, max_pos, cos_out, sin_out);
    return cudaGetLastError();
}

// Positions of 32 token rows, range-checked against the tables (clamped, flagged).
__device__ __forceinline__ int checked_pos(const int32_t* pos, int64_t row, int t, int max_pos, uint32_t* check) {
    int p = pos ? pos[row] : t;
    if (p < 0 || p >= max_pos) {
        flag(check, LOWRAM_CHECK_POS_RANGE);
        p = p < 0 ? 0 : max_pos - 1;
    }
    return p;
}

// Rotated dot product q . RoPE(k_pre) for one token row held in shared memory, lanes split the pairs.
__device__ __forceinline__ float rotated_dot(const float* qv, const float* krow, int d, int p, int max_pos,
                                             const float* rcos, const float* rsin, int lane) {
    const int h = d / 2;
    float acc = 0.0f;
    for (int i = lane; i < h; i += 32) {
        float c = rcos[(int64_t)i * max_pos + p], s = rsin[(int64_t)i * max_pos + p];
        float x = krow[i], y = krow[i + h];
        acc = fmaf(qv[i], x * c - y * s, acc);
        acc = fmaf(qv[i + h], y * c + x * s, acc);
    }
    return warp_sum(acc);
}

// ------------------------------------------------------------------------------------------------
// K1 (CUDA cores): selection key of every token.  grid (T/32, H_kv, B), 256 threads.
// ------------------------------------------------------------------------------------------------
template <typename TA, typename CoefV>
__global__ void __launch_bounds__(kTileThreads) score_simt_kernel(DecodeArgs a, CoefV coef) {
    extern __shared__ float sm[];
    const auto& s = a.s;
    const int d = s.d, r = s.r, T = s.T, g = a.g;
    const int t0 = blockIdx.x * kTileRows, h = blockIdx.y, b = blockIdx.z;
    float* As = sm;
    float* Bs = As + kTileRows * kStride;
    float* Ks = Bs + 4 * 32 * kStride;
    float* Qs = Ks + kTileRows * (kMaxD + 1);
    int* Ps = (int*)(Qs + 8 * kMaxD);
    int64_t* Rows = (int64_t*)(Ps + kTileRows);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid < kTileRows) {
        int t = t0 + tid;
        Rows[tid] = t < T ? (int64_t)b * T + t : -1;
        Ps[tid] = t < T ? checked_pos(a.pos, (int64_t)b * T + t, t, s.max_pos, a.check) : 0;
    }
    for (int e = tid; e < g * d; e += kTileThreads) Qs[e] = ld((const TA*)a.q, ((int64_t)b * s.H_q + h * g) * d + e);
    __syncthreads();
    rebuild_rows<TA>(Rows, coef, r, (const TA*)a.basis + b * s.basis_batch_stride + (int64_t)h * d * r, d, As, Bs, Ks);

    for (int u = 0; u < 4; ++u) {
        const int t = warp * 4 + u;
        float best = -INFINITY;
        for (int jq = 0; jq < g; ++jq)
            best = fmaxf(best, a.scale * rotated_dot(Qs + jq * d, Ks + t * (d + 1), d, Ps[t], s.max_pos, a.rope_cos,
                                                     a.rope_sin, lane));
        if (lane == 0 && t0 + t < T) a.key[((int64_t)b * s.H_kv + h) * T + t0 + t] = best;
    }
}

// ------------------------------------------------------------------------------------------------
// K3 (CUDA cores): values of 32 selected tokens + softmax partial per q-head.  grid (chunks, H_kv, B).
// partial layout [B, H_q, n_chunks, d + 2]: acc[0..d), running max, running sum.
// ------------------------------------------------------------------------------------------------
template <typename TA, typename CoefV, int NJm>
__global__ void __launch_bounds__(kTileThreads) vregen_simt_kernel(DecodeArgs a, CoefV coef, ResView res) {
    extern __shared__ float sm[];
    const auto& s = a.s;
    const int d = s.d, r = s.r, m = s.m, T = s.T, g = a.g, n_res = s.n_res, S_eff = a.S_eff;
    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    float* As = sm;
    float* Bs = As + kTileRows * kStride;
    float* Ks = Bs + NJm * 32 * kStride;
    float* Vs = Ks + kTileRows * (kMaxD + 1);
    float* Hs = Vs + kTileRows * (kMaxD + 1);
    float* Qs = Hs + kTileRows * (NJm * 32 + 1);
    float* Ss = Qs + 8 * kMaxD;                 // [g][32] scaled logits
    int* Ps = (int*)(Ss + 8 * kTileRows);
    int* Tok = Ps + kTileRows;                  // token index or -1
    int64_t* Rows = (int64_t*)(Tok + kTileRows);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t bh = (int64_t)b * s.H_kv + h;
    const int32_t* ridx = a.res_idx + bh * n_res;

    if (tid < kTileRows) {
        int j = chunk * kTileRows + tid;
        int t = j < S_eff ? a.sel[bh * S_eff + j] : -1;
        if (t >= T) t = T - 1;  // selection output is always in range; keep the invariant explicit
        Tok[tid] = t;
        Rows[tid] = t >= 0 ? (int64_t)b * T + t : -1;
        Ps[tid] = t >= 0 ? checked_pos(a.pos, (int64_t)b * T + t, t, s.max_pos, nullptr) : 0;
    }
    for (int e = tid; e < g * d; e += kTileThreads) Qs[e] = ld((const TA*)a.q, ((int64_t)b * s.H_q + h * g) * d + e);
    // one CTA per (b, h) validates the residual list: in range and strictly ascending
    if (chunk == 0)
        for (int j = tid; j < n_res; j += kTileThreads)
            if (ridx[j] < 0 || ridx[j] >= T || (j > 0 && ridx[j] <= ridx[j - 1])) flag(a.check, LOWRAM_CHECK_RES_INDEX);
    __syncthreads();

    rebuild_rows<TA>(Rows, coef, r, (const TA*)a.basis + b * s.basis_batch_stride + (int64_t)h * d * r, d, As, Bs, Ks);
    // scaled logits of the selected tokens (RoPE re-applied on the fly)
    for (int u = 0; u < 4; ++u) {
        const int t = warp * 4 + u;
        for (int jq = 0; jq < g; ++jq) {
            float v = a.scale * rotated_dot(Qs + jq * d, Ks + t * (d + 1), d, Ps[t], s.max_pos, a.rope_cos, a.rope_sin,
                                            lane);
            if (lane == 0) Ss[jq * kTileRows + t] = Tok[t] >= 0 ? v : -INFINITY;
        }
    }
    // a predictor per sequence: sequence b's weights mlp_batch_stride elements on, its biases [B, H_kv, .]
    const int64_t mo = b * s.mlp_batch_stride, bias_bh = s.mlp_batch_stride ? bh : h;
    predict_from_keys<TA, NJm, false>((const TA*)a.w1 + mo + (int64_t)h * m * d, a.b1 ? a.b1 + bias_bh * m : nullptr,
                                      (const TA*)a.w2 + mo + (int64_t)h * d * m, a.b2 ? a.b2 + bias_bh * d : nullptr, d, m,
                                      As, Bs, Ks, Hs, Vs);
    // residual add: binary search of each selected token in the ascending residual list
    for (int u = 0; u < 4; ++u) {
        const int t = warp * 4 + u;
        const int tok = Tok[t];
        if (tok < 0 || n_res == 0) continue;
        int lo = 0, hi = n_res - 1, hit = -1;
        while (lo <= hi) {
            int mid = (lo + hi) >> 1;
            int v = ridx[mid];
            if (v == tok) { hit = mid; break; }
            if (v < tok) lo = mid + 1; else hi = mid - 1;
        }
        if (hit >= 0)
            for (int i = lane; i < d; i += 32) Vs[t * (d + 1) + i] += res.get(bh * n_res + hit, i);
    }
    __syncthreads();
    // softmax partial: warp jq handles q-head jq
    if (warp < g) {
        const int jq = warp;
        float sv = Ss[jq * kTileRows + lane];
        float mx = warp_max(sv);
        float p = (sv == -INFINITY) ? 0.0f : __expf(sv - mx);
        float l = warp_sum(p);
        float* dst = a.partial + (((int64_t)b * s.H_q + h * g + jq) * a.n_chunks + chunk) * (d + 2);
        for (int i = lane; i < d; i += 32) {
            float acc = 0.0f;
            for (int t = 0; t < kTileRows; ++t) acc = fmaf(__shfl_sync(0xffffffffu, p, t), Vs[t * (d + 1) + i], acc);
            dst[i] = acc;
        }
        if (lane == 0) {
            dst[d] = mx;
            dst[d + 1] = l;
        }
    }
}

// ------------------------------------------------------------------------------------------------
// K4: merge split-softmax partials.  One CTA of 256 threads per (b, q-head):
//   W = max_c m_c, w_c = exp(m_c - W), L = sum_c w_c l_c, out = sum_c w_c acc_c / L, lse = W + log L.
// The per-chunk weights go to shared memory; each output feature is summed by two threads, each taking
// alternate groups of 16 chunks as one batch of independent loads, and the two halves add in shared memory.
// ------------------------------------------------------------------------------------------------
constexpr int kMergeThreads = 256;
constexpr int kMergeBatch = 16;

__device__ __forceinline__ float merge_reduce(float v, float* red, bool is_max) {
    v = is_max ? warp_max(v) : warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < kMergeThreads / 32; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(int n_chunks, int d, const float* __restrict__ partial,
                                                              float* __restrict__ out, float* __restrict__ lse) {
    extern __shared__ float wts[];   // [n_chunks]
    __shared__ float red[kMergeThreads / 32];
    __shared__ float half_sum[kMaxD];
    const int w = blockIdx.x, tid = threadIdx.x;
    const int64_t rw = d + 2;
    const float* P = partial + (int64_t)w * n_chunks * rw;
    grid_dep_wait();   // the records come from the kernel before
    float M = -INFINITY;
    for (int c = tid; c < n_chunks; c += kMergeThreads) M = fmaxf(M, P[c * rw + d]);
    M = merge_reduce(M, red, true);
    float L = 0.0f;
    for (int c = tid; c < n_chunks; c += kMergeThreads) {
        const float mc = P[c * rw + d];
        const float wc = (mc == -INFINITY) ? 0.0f : __expf(mc - M);
        wts[c] = wc;
        L = fmaf(wc, P[c * rw + d + 1], L);
    }
    L = merge_reduce(L, red, false);   // also orders the wts[] writes before their reads
    const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
    const int f = tid & (kMaxD - 1), half = tid / kMaxD;
    float acc = 0.0f;
    if (f < d) {
        for (int c0 = half * kMergeBatch; c0 < n_chunks; c0 += 2 * kMergeBatch) {
            float v[kMergeBatch];
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) v[u] = (c0 + u < n_chunks) ? P[(c0 + u) * rw + f] : 0.0f;
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u)
                if (c0 + u < n_chunks) acc = fmaf(wts[c0 + u], v[u], acc);
        }
        if (half == 1) half_sum[f] = acc;
    }
    __syncthreads();
    if (half == 0 && f < d) out[(int64_t)w * d + f] = (acc + half_sum[f]) * inv;
    if (lse && tid == 0) lse[w] = (L > 0.0f) ? M + logf(L) : -INFINITY;
}

// The same merge for d = 128 with one warp per (b, q-head) and no block barrier: chunks in batches of eight, every
// load of a batch (each chunk's maximum and weight sum, broadcast, and the lane's four output features) issued
// before any is used, and the batches folded into a running maximum with the usual rescale.  Eight rows per CTA of
// 256 threads.
__global__ void __launch_bounds__(256) merge_warp_kernel(int BH, int n_chunks, const float* __restrict__ partial,
                                                         float* __restrict__ out, float* __restrict__ lse) {
    grid_dep_wait();   // the records come from the kernel before
    const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (w >= BH) return;
    constexpr int64_t rw = 128 + 2;
    const float* P = partial + (int64_t)w * n_chunks * rw;
    float M = -INFINITY, L = 0.0f;
    float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int c0 = 0; c0 < n_chunks; c0 += 8) {
        float mc[8], lc[8];
        float2 v0[8], v1[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const bool in = c0 + u < n_chunks;
            const float* pc = P + (in ? c0 + u : 0) * rw;
            mc[u] = in ? pc[128] : -INFINITY;
            lc[u] = in ? pc[129] : 0.0f;
            v0[u] = *reinterpret_cast<const float2*>(pc + 4 * lane);   // rw even: 8-byte aligned
            v1[u] = *reinterpret_cast<const float2*>(pc + 4 * lane + 2);
        }
        float Mb = M;
#pragma unroll
        for (int u = 0; u < 8; ++u) Mb = fmaxf(Mb, mc[u]);
        if (Mb == -INFINITY) continue;   // nothing weighted yet
        const float r = M == -INFINITY ? 0.0f : __expf(M - Mb);   // rescale what the batches before summed
        L *= r;
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] *= r;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float wc = mc[u] == -INFINITY ? 0.0f : __expf(mc[u] - Mb);
            L = fmaf(wc, lc[u], L);
            a[0] = fmaf(wc, v0[u].x, a[0]);
            a[1] = fmaf(wc, v0[u].y, a[1]);
            a[2] = fmaf(wc, v1[u].x, a[2]);
            a[3] = fmaf(wc, v1[u].y, a[3]);
        }
        M = Mb;
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    *reinterpret_cast<float4*>(out + (int64_t)w * 128 + 4 * lane) =
        make_float4(a[0] * inv, a[1] * inv, a[2] * inv, a[3] * inv);
    if (lse && lane == 0) lse[w] = L > 0.0f ? M + logf(L) : -INFINITY;
}

cudaError_t launch_merge(int B, int H_q, int n_chunks, int d, const float* partial, float* out, float* lse,
                         cudaStream_t st) {
    const int BH = B * H_q;
    if (BH == 0) return cudaSuccess;
    if (d == 128 && n_chunks > 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0)
        return launch_pdl(merge_warp_kernel, dim3((unsigned)cdiv(BH, 8)), dim3(256), 0, st, BH, n_chunks, partial, out,
                          lse);
    const size_t smem = sizeof(float) * (size_t)(n_chunks > 0 ? n_chunks : 1);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(merge_kernel, dim3((unsigned)BH), dim3(kMergeThreads), smem, st, n_chunks, d, partial, out, lse);
}

// ------------------------------------------------------------------------------------------------
// launchers
// ------------------------------------------------------------------------------------------------
static size_t score_smem() {
    return sizeof(float) * (kTileRows * kStride + 4 * 32 * kStride + kTileRows * (kMaxD + 1) + 8 * kMaxD) +
           sizeof(int) * kTileRows + sizeof(int64_t) * kTileRows + 64;
}

template <int NJm>
static size_t vregen_smem() {
    return sizeof(float) * (kTileRows * kStride + NJm * 32 * kStride + 2 * kTileRows * (kMaxD + 1) +
                            kTileRows * (NJm * 32 + 1) + 8 * kMaxD + 8 * kTileRows) +
           sizeof(int) * 2 * kTileRows + sizeof(int64_t) * kTileRows + 64;
}

template <typename TA, typename CoefV>
static cudaError_t score_go(const DecodeArgs& a, CoefV coef, cudaStream_t st) {
    const size_t smem = score_smem();
    auto k = score_simt_kernel<TA, CoefV>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)cdiv(a.s.T, kTileRows), (unsigned)a.s.H_kv, (unsigned)a.s.B);
    k<<<grid, kTileThreads, smem, st>>>(a, coef);
    return cudaGetLastError();
}

cudaError_t launch_score_simt(const DecodeArgs& a, cudaStream_t st) {
    if ((int64_t)a.s.B * a.s.T == 0) return cudaSuccess;
    const auto& s = a.s;
    if (s.coef_dtype == LOWRAM_INT4_G32) {
        CoefRowsInt4 c{(const uint8_t*)a.coef, (const __half*)a.coef_scale, s.r};
        return s.act_dtype == LOWRAM_BF16 ? score_go<__nv_bfloat16>(a, c, st) : score_go<float>(a, c, st);
    }
    if (s.act_dtype == LOWRAM_BF16) return score_go<__nv_bfloat16>(a, CoefRows<__nv_bfloat16>{(const __nv_bfloat16*)a.coef, s.r}, st);
    return score_go<float>(a, CoefRows<float>{(const float*)a.coef, s.r}, st);
}

template <typename TA, typename CoefV, int NJm>
static cudaError_t vregen_go(const DecodeArgs& a, CoefV coef, ResView res, cudaStream_t st) {
    const size_t smem = vregen_smem<NJm>();
    auto k = vregen_simt_kernel<TA, CoefV, NJm>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.n_chunks, (unsigned)a.s.H_kv, (unsigned)a.s.B);
    k<<<grid, kTileThreads, smem, st>>>(a, coef, res);
    return cudaGetLastError();
}

template <typename TA, typename CoefV>
static cudaError_t vregen_m(const DecodeArgs& a, CoefV coef, ResView res, cudaStream_t st) {
    if (a.s.m <= 128) return vregen_go<TA, CoefV, 4>(a, coef, res, st);
    return vregen_go<TA, CoefV, 8>(a, coef, res, st);
}

cudaError_t launch_vregen_simt(const DecodeArgs& a, cudaStream_t st) {
    if ((int64_t)a.s.B * a.n_chunks == 0) return cudaSuccess;
    const auto& s = a.s;
    ResView res{s.res_dtype, a.res_val, (const __half*)a.res_scale, s.d};
    if (s.coef_dtype == LOWRAM_INT4_G32) {
        CoefRowsInt4 c{(const uint8_t*)a.coef, (const __half*)a.coef_scale, s.r};
        return s.act_dtype == LOWRAM_BF16 ? vregen_m<__nv_bfloat16>(a, c, res, st) : vregen_m<float>(a, c, res, st);
    }
    if (s.act_dtype == LOWRAM_BF16)
        return vregen_m<__nv_bfloat16>(a, CoefRows<__nv_bfloat16>{(const __nv_bfloat16*)a.coef, s.r}, res, st);
    return vregen_m<float>(a, CoefRows<float>{(const float*)a.coef, s.r}, res, st);
}

}  // namespace lowram
