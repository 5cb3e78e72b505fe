// predict_fit.cu -- test-time fit of the per-head value predictor on the prompt: full-batch Adam on the mean
// squared error of v_hat = w2 silu(w1 k + b1) + b2 against the prompt's values (LowRAM abstract: the predictor is
// fitted at test time; "Value cache amortisation in plain language": values are predicted from pre-RoPE keys).
//
// Gradient (one kv-head, N tokens, E = v_hat - v, c = 2 / (N d)):
//   g_w2 = c E^T H,  g_b2 = c sum_t E_t,  dZ = (E w2) * silu'(Z),  g_w1 = c dZ^T K,  g_b1 = c sum_t dZ_t,
//   with Z = K w1^T + b1, H = silu(Z), silu'(z) = s + z s (1 - s), s = 1 / (1 + e^-z); loss = sum E^2 / (N d).
// predictor_grad_kernel: CTAs over (token range, kv-head, half of the hidden units).  A CTA walks its tokens
// in tiles of 32: the forward pass over all m hidden units (the output needs all of them), then the backward
// pass for its 128 hidden units; each thread keeps an 8-column block of g_w2 and of g_w1 in registers across
// the tiles and adds them to the global gradient once, with atomics.  fp32 CUDA cores throughout: the fit
// compares with an fp64 reference step by step.
// adam_kernel: one Adam step with bias correction on a flat parameter array.
#include "common.cuh"
#include "kernels.h"
#include "predict_fit.h"
#include "simt_tile.cuh"

namespace lowram {

namespace {

constexpr int kPfThreads = 256;
constexpr int kPfTok = 32;          // tokens per tile (the tile product's row count)

struct PfLayout {                   // shared-memory carve-up, floats
    int d, m, ld_d, ld_m, ld_h;
    __host__ __device__ int ks() const { return 0; }
    __host__ __device__ int vs() const { return ks() + kPfTok * ld_d; }
    __host__ __device__ int zs() const { return vs() + kPfTok * ld_d; }
    __host__ __device__ int hs() const { return zs() + kPfTok * ld_m; }
    __host__ __device__ int es() const { return hs() + kPfTok * ld_m; }
    __host__ __device__ int dzs() const { return es() + kPfTok * ld_d; }
    __host__ __device__ int stage() const { return dzs() + kPfTok * ld_h; }
    __host__ __device__ int total(int nj) const { return stage() + tile_smem_floats(nj); }
};

__host__ __device__ inline PfLayout pf_layout(int d, int m) { return PfLayout{d, m, d + 1, m + 1, 129}; }

template <typename TA, int NJM, int NJD, int RB>
__global__ void __launch_bounds__(kPfThreads, 1)
    predictor_grad_kernel(int64_t N, int H_kv, int d, int m, const TA* __restrict__ keys,
                          const TA* __restrict__ values, const float* __restrict__ w1, const float* __restrict__ b1,
                          const float* __restrict__ w2, const float* __restrict__ b2, int n_blk, float* loss,
                          float* g_w1, float* g_b1, float* g_w2, float* g_b2) {
    extern __shared__ float sm[];
    const PfLayout L = pf_layout(d, m);
    float* Ks = sm + L.ks();
    float* Vs = sm + L.vs();
    float* Zs = sm + L.zs();
    float* Hs = sm + L.hs();
    float* Es = sm + L.es();
    float* dZs = sm + L.dzs();
    float* As = sm + L.stage();
    float* Bs = As + kTileRows * kStride;
    const int blk = blockIdx.x, h = blockIdx.y, half = blockIdx.z;
    const int jb = half * 128, mh = min(128, m - jb);      // this CTA's hidden units [jb, jb + mh)
    const int tid = threadIdx.x;
    const float* W1 = w1 + (int64_t)h * m * d;
    const float* W2 = w2 + (int64_t)h * d * m;
    const float* B1 = b1 + (int64_t)h * m;
    const float* B2 = b2 + (int64_t)h * d;
    const int64_t per = (N + n_blk - 1) / n_blk;
    const int64_t n_begin = blk * per, n_end = min(N, n_begin + per);
    // register-held gradient blocks: g_w2[i][jb + j], i = (tid / 16) * RB + a, j = (tid % 16) * 8 + c;
    // g_w1[jb + j][k], j = (tid / 16) * 8 + a, k = (tid % 16) * RB + c
    const int r16 = tid >> 4, c16 = tid & 15;
    float gw2[RB][8], gw1[8][RB];
#pragma unroll
    for (int a = 0; a < RB; ++a)
#pragma unroll
        for (int c = 0; c < 8; ++c) gw2[a][c] = gw1[c][a] = 0.0f;
    float gb1 = 0.0f, gb2 = 0.0f, lsum = 0.0f;   // thread tid < mh: g_b1[jb + tid]; tid < d (half 0): g_b2[tid]
    for (int64_t t0 = n_begin; t0 < n_end; t0 += kPfTok) {
        const int nt = (int)min((int64_t)kPfTok, n_end - t0);
        // tokens of the tile: keys and values of head h, float32; rows past the range are zero
        for (int e = tid; e < kPfTok * d; e += kPfThreads) {
            const int t = e / d, k = e - t * d;
            const int64_t off = ((t0 + t) * H_kv + h) * d + k;
            Ks[t * L.ld_d + k] = t < nt ? ld(keys, off) : 0.0f;
            Vs[t * L.ld_d + k] = t < nt ? ld(values, off) : 0.0f;
        }
        __syncthreads();
        // forward: Z = K w1^T + b1, H = silu(Z) (all m hidden units)
        {
            float acc[4][NJM];
            zero_acc<NJM>(acc);
            tile_product<NJM>([&](int t, int k) { return Ks[t * L.ld_d + k]; },
                              [&](int j, int k) { return W1[(int64_t)j * d + k]; }, d, 0, m, As, Bs, acc);
            const int tx = tid & 31, ty = tid >> 5;
#pragma unroll
            for (int jj = 0; jj < NJM; ++jj) {
                const int j = tx + 32 * jj;
                if (j >= m) continue;
                const float bj = B1[j];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float z = acc[u][jj] + bj;
                    Zs[(ty * 4 + u) * L.ld_m + j] = z;
                    Hs[(ty * 4 + u) * L.ld_m + j] = z / (1.0f + expf(-z));
                }
            }
        }
        __syncthreads();
        // output and error: E = H w2^T + b2 - V (rows past the range: zero)
        {
            float acc[4][NJD];
            zero_acc<NJD>(acc);
            tile_product<NJD>([&](int t, int k) { return Hs[t * L.ld_m + k]; },
                              [&](int i, int k) { return W2[(int64_t)i * m + k]; }, m, 0, d, As, Bs, acc);
            const int tx = tid & 31, ty = tid >> 5;
#pragma unroll
            for (int ii = 0; ii < NJD; ++ii) {
                const int i = tx + 32 * ii;
                if (i >= d) continue;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int t = ty * 4 + u;
                    const float e = t < nt ? acc[u][ii] + B2[i] - Vs[t * L.ld_d + i] : 0.0f;
                    Es[t * L.ld_d + i] = e;
                    lsum = fmaf(e, e, lsum);
                }
            }
        }
        __syncthreads();
        // backward for this CTA's hidden units: dZ = (E w2[:, jb:]) * silu'(Z)
        {
            float acc[4][4];
            zero_acc<4>(acc);
            tile_product<4>([&](int t, int k) { return Es[t * L.ld_d + k]; },
                            [&](int j, int k) { return W2[(int64_t)k * m + jb + j]; }, d, 0, mh, As, Bs, acc);
            const int tx = tid & 31, ty = tid >> 5;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int j = tx + 32 * jj;
                if (j >= mh) continue;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int t = ty * 4 + u;
                    const float z = Zs[t * L.ld_m + jb + j];
                    const float s = 1.0f / (1.0f + expf(-z));
                    dZs[t * L.ld_h + j] = acc[u][jj] * (s + z * s * (1.0f - s));
                }
            }
        }
        __syncthreads();
        // gradient blocks over the tile's tokens
        for (int t = 0; t < kPfTok; ++t) {
            float ev[RB], kv[RB], hv[8], dz[8];
#pragma unroll
            for (int a = 0; a < RB; ++a) {
                ev[a] = Es[t * L.ld_d + r16 * RB + a];
                kv[a] = Ks[t * L.ld_d + c16 * RB + a];
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int jh = c16 * 8 + c, jz = r16 * 8 + c;
                hv[c] = jh < mh ? Hs[t * L.ld_m + jb + jh] : 0.0f;
                dz[c] = jz < mh ? dZs[t * L.ld_h + jz] : 0.0f;
            }
#pragma unroll
            for (int a = 0; a < RB; ++a)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    gw2[a][c] = fmaf(ev[a], hv[c], gw2[a][c]);
                    gw1[c][a] = fmaf(dz[c], kv[a], gw1[c][a]);
                }
            if (tid < mh) gb1 += dZs[t * L.ld_h + tid];
            if (half == 0 && tid < d) gb2 += Es[t * L.ld_d + tid];
        }
        __syncthreads();
    }
    const float cscale = 2.0f / ((float)N * (float)d);
#pragma unroll
    for (int a = 0; a < RB; ++a)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int i = r16 * RB + a, j = c16 * 8 + c;
            if (i < d && j < mh) atomicAdd(&g_w2[((int64_t)h * d + i) * m + jb + j], gw2[a][c] * cscale);
            const int jz = r16 * 8 + c, k = c16 * RB + a;
            if (jz < mh && k < d) atomicAdd(&g_w1[((int64_t)h * m + jb + jz) * d + k], gw1[c][a] * cscale);
        }
    if (tid < mh) atomicAdd(&g_b1[(int64_t)h * m + jb + tid], gb1 * cscale);
    if (half == 0 && tid < d) atomicAdd(&g_b2[(int64_t)h * d + tid], gb2 * cscale);
    if (half == 0) {
        // loss: the sum of squared errors of this CTA's tokens, over (N d)
        lsum = warp_sum(lsum);
        if ((tid & 31) == 0) atomicAdd(&loss[h], lsum / ((float)N * (float)d));
    }
}

__global__ void adam_kernel(float* p, const float* g, float* mom, float* vel, int64_t n, float lr, float beta1,
                            float beta2, float eps, float bc1, float bc2) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float gi = g[i];
    const float mi = beta1 * mom[i] + (1.0f - beta1) * gi;
    const float vi = beta2 * vel[i] + (1.0f - beta2) * gi * gi;
    mom[i] = mi;
    vel[i] = vi;
    p[i] -= lr * (mi / bc1) / (sqrtf(vi / bc2) + eps);
}

template <typename TA, int NJM, int NJD, int RB>
cudaError_t grad_go(const PredictorFitArgs& a, cudaStream_t st) {
    const int64_t N = (int64_t)a.B * a.T;
    const int n_half = (a.m + 127) / 128;
    const PfLayout L = pf_layout(a.d, a.m);
    const size_t smem = sizeof(float) * (size_t)L.total(NJM > NJD ? NJM : NJD);
    auto k = predictor_grad_kernel<TA, NJM, NJD, RB>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t tiles = (N + kPfTok - 1) / kPfTok;
    const int n_blk = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (2 * sms) / (a.H_kv * n_half) + 1));
    k<<<dim3((unsigned)n_blk, (unsigned)a.H_kv, (unsigned)n_half), kPfThreads, smem, st>>>(
        N, a.H_kv, a.d, a.m, (const TA*)a.keys, (const TA*)a.values, a.w1, a.b1, a.w2, a.b2, n_blk, a.loss, a.g_w1,
        a.g_b1, a.g_w2, a.g_b2);
    return cudaGetLastError();
}

template <typename TA>
cudaError_t grad_dispatch(const PredictorFitArgs& a, cudaStream_t st) {
    // NJM: hidden-unit column groups of the forward product (m <= NJM*32); NJD: output groups (d = NJD*32);
    // RB: rows of a thread's gradient block (d / 16)
    if (a.d == 128) {
        if (a.m <= 128) return grad_go<TA, 4, 4, 8>(a, st);
        return grad_go<TA, 8, 4, 8>(a, st);
    }
    if (a.m <= 128) return grad_go<TA, 4, 2, 4>(a, st);
    return grad_go<TA, 8, 2, 4>(a, st);
}

}  // namespace

cudaError_t launch_predictor_grad(const PredictorFitArgs& a, cudaStream_t st) {
    const size_t n1 = (size_t)a.H_kv * a.m * a.d, nb1 = (size_t)a.H_kv * a.m, nb2 = (size_t)a.H_kv * a.d;
    cudaError_t e;
    if ((e = cudaMemsetAsync(a.g_w1, 0, sizeof(float) * n1, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.g_w2, 0, sizeof(float) * n1, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.g_b1, 0, sizeof(float) * nb1, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.g_b2, 0, sizeof(float) * nb2, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.loss, 0, sizeof(float) * a.H_kv, st)) != cudaSuccess) return e;
    if ((int64_t)a.B * a.T == 0) return cudaSuccess;
    return a.bf16 ? grad_dispatch<__nv_bfloat16>(a, st) : grad_dispatch<float>(a, st);
}

cudaError_t launch_adam(float* p, const float* g, float* mom, float* vel, int64_t n, float lr, float beta1, float beta2,
                        float eps, int step, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const float bc1 = 1.0f - powf(beta1, (float)step), bc2 = 1.0f - powf(beta2, (float)step);
    adam_kernel<<<(unsigned)cdiv(n, 256), 256, 0, st>>>(p, g, mom, vel, n, lr, beta1, beta2, eps, bc1, bc2);
    return cudaGetLastError();
}

}  // namespace lowram
