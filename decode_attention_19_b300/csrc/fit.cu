// fit.cu -- the group's shared low-rank key basis from the prompt's keys: the cross-layer SVD of the
// RoPE-inverted keys ("LowRAM Paper: Amortised Values and Low-Rank Keys for KV Compression", "Asymmetric key
// compression with xKV": the G layers' keys are stacked and factored together after RoPE is inverted).
//
// With X = k_cat [N = B*T tokens, D = G*H_kv*d] in float32 (rotated back by each token's position when the
// keys are given rotated), the rank-r subspace of X's largest singular values is spanned by the top-r
// eigenvectors of the Gram matrix X^T X [D, D].  They are found by subspace iteration:
//   Q_0 seeded Gaussian [D, r];  repeat `iters` times:  Z = (X^T X) Q,  Q = Z R^-1  with  Z^T Z = R^T R,
// i.e. Cholesky QR (Z^T Z and its Cholesky factor in fp64), and one more Cholesky QR of the last Q so that
// Q^T Q = I to float32 accuracy.  Any orthonormal basis of the subspace serves the method (the rebuilt keys
// X Q Q^T do not depend on the rotation within it), so no Rayleigh-Ritz ordering step is taken.
// Outputs: proj = Q^T [r, D] float32 (a left inverse of the stacked bases) and the G layer blocks of Q as the
// bases [H_kv*d, r] in the activation dtype: the inputs lowram_compress takes.
//
// Kernels: a key prep pass (dtype, inverse RoPE), a Gram kernel (64 x 64 output tiles of the upper triangle,
// mirrored, split over tokens with atomics when the tiles alone do not fill the GPU), a row-major SGEMM, a
// single-CTA fp64 Cholesky, a row-parallel triangular solve, and the output pass.  All CUDA cores: the fit runs once
// per prompt and the Gram product needs fp32 accumulation of fp32 keys.
#include "common.cuh"
#include "kernels.h"

namespace lowram {

namespace {

constexpr int kFT = 64;        // output tile edge
constexpr int kFK = 16;        // reduction chunk
constexpr int kFThreads = 256; // 16 x 16 threads, 4 x 4 outputs each

// X[n, k] (float32) of token n = b*T + t: dtype conversion, and the inverse rotation when the keys are rotated
template <typename TA>
__global__ void prep_keys_kernel(const TA* __restrict__ keys, int64_t N, int T, int D, int d, const int32_t* pos,
                                 const float* rcos, const float* rsin, int max_pos, int post_rope,
                                 uint32_t* check, float* __restrict__ X) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N * D) return;
    const int64_t n = i / D;
    const int k = (int)(i - n * D);
    const TA* row = keys + n * D;
    if (!post_rope) {
        X[i] = ld(row, k);
        return;
    }
    int p = pos ? pos[n] : (int)(n % T);
    if (p < 0 || p >= max_pos) {
        if ((k % d) == 0) flag(check, LOWRAM_CHECK_POS_RANGE);
        p = p < 0 ? 0 : max_pos - 1;
    }
    const int half = d / 2, j = k % d;
    const int f = j < half ? j : j - half;
    const float c = rcos[(int64_t)f * max_pos + p], s = rsin[(int64_t)f * max_pos + p];
    // rotate by -angle: (x, y) -> (x cos + y sin, y cos - x sin)
    X[i] = j < half ? ld(row, k) * c + ld(row, k + half) * s : ld(row, k) * c - ld(row, k - half) * s;
}

// C[D, D] (+)= X^T X over rows [n_begin, n_end) of X [N, D] (row-major); upper-triangle tiles only, each written
// with its mirror.  Split over rows (blockIdx.z) when `atomic`.
template <typename TAcc>
__global__ void __launch_bounds__(kFThreads) gram_kernel(const float* __restrict__ X, int64_t N, int D, int n_split,
                                                         bool atomic, TAcc* __restrict__ C) {
    // upper-triangle tile (bi <= bj) from the linear block index
    const int nt = (D + kFT - 1) / kFT;
    int lin = blockIdx.x, bi = 0;
    while (lin >= nt - bi) {
        lin -= nt - bi;
        ++bi;
    }
    const int bj = bi + lin;
    const int i0 = bi * kFT, j0 = bj * kFT;
    const int64_t per = (N + n_split - 1) / n_split;
    const int64_t n_begin = blockIdx.z * per, n_end = min(N, n_begin + per);
    __shared__ float As[kFK][kFT + 4], Bs[kFK][kFT + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    TAcc acc[4][4] = {};
    for (int64_t n0 = n_begin; n0 < n_end; n0 += kFK) {
        for (int e = tid; e < kFK * kFT; e += kFThreads) {
            const int r = e / kFT, c = e % kFT;
            const int64_t n = n0 + r;
            As[r][c] = (n < n_end && i0 + c < D) ? X[n * D + i0 + c] : 0.0f;
            Bs[r][c] = (n < n_end && j0 + c < D) ? X[n * D + j0 + c] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kFK; ++k) {
            float a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a[u] = As[k][ty * 4 + u];
                b[u] = Bs[k][tx * 4 + u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] += (TAcc)a[u] * (TAcc)b[v];
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int i = i0 + ty * 4 + u, j = j0 + tx * 4 + v;
            if (i >= D || j >= D) continue;
            if (atomic) {
                atomicAdd(&C[(int64_t)i * D + j], acc[u][v]);
                if (bi != bj) atomicAdd(&C[(int64_t)j * D + i], acc[u][v]);
            } else {
                C[(int64_t)i * D + j] = acc[u][v];
                if (bi != bj) C[(int64_t)j * D + i] = acc[u][v];
            }
        }
}

// C[M, Nc] = A[M, K] B[K, Nc], row-major float32
__global__ void __launch_bounds__(kFThreads) sgemm_kernel(const float* __restrict__ A, const float* __restrict__ B,
                                                          int M, int K, int Nc, float* __restrict__ C) {
    const int m0 = blockIdx.y * kFT, c0 = blockIdx.x * kFT;
    __shared__ float As[kFK][kFT + 4], Bs[kFK][kFT + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += kFK) {
        for (int e = tid; e < kFK * kFT; e += kFThreads) {
            const int r = e % kFK, m = e / kFK;      // A tile: consecutive threads along k within a row
            As[r][m] = (m0 + m < M && k0 + r < K) ? A[(int64_t)(m0 + m) * K + k0 + r] : 0.0f;
            const int kr = e / kFT, c = e % kFT;     // B tile: consecutive threads along the row
            Bs[kr][c] = (k0 + kr < K && c0 + c < Nc) ? B[(int64_t)(k0 + kr) * Nc + c0 + c] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kFK; ++k) {
            float a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a[u] = As[k][ty * 4 + u];
                b[u] = Bs[k][tx * 4 + u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int m = m0 + ty * 4 + u, c = c0 + tx * 4 + v;
            if (m < M && c < Nc) C[(int64_t)m * Nc + c] = acc[u][v];
        }
}

// Seeded standard normal start: splitmix64 of (seed, element) gives two uniforms, Box-Muller one normal.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

__global__ void init_normal_kernel(float* Q, int64_t n, uint64_t seed) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint64_t h = splitmix64(seed ^ splitmix64((uint64_t)i));
    const float u1 = ((float)(h >> 40) + 1.0f) * (1.0f / 16777217.0f);     // (0, 1]
    const float u2 = (float)((h >> 16) & 0xFFFFFFu) * (1.0f / 16777216.0f);
    Q[i] = sqrtf(-2.0f * logf(u1)) * cospif(2.0f * u2);
}

// One CTA: S [r, r] fp64 is overwritten with its Cholesky factor (S = L L^T, L lower), which is also written
// as float32 to Lf [r, r] (lower triangle; the strict upper triangle is not read).  A pivot at or below 1e-10 of
// the largest diagonal entry (rounding noise of float32 iterates: the keys have rank below r) sets
// LOWRAM_CHECK_NOT_PD and stops; Lf is then incomplete and the fit's result is void.
__global__ void __launch_bounds__(1024) chol_kernel(double* S, int r, float* Lf, uint32_t* check) {
    __shared__ int bad;
    __shared__ double floor_pivot;
    const int tid = threadIdx.x, nt = blockDim.x;
    if (tid == 0) {
        bad = 0;
        double mx = 0.0;
        for (int k = 0; k < r; ++k) mx = fmax(mx, S[(int64_t)k * r + k]);
        // pivot k ~ (lambda_k / lambda_1)^2 of the largest: below 1e-10 (an eigenvalue under 1e-5 of the largest,
        // the level of float32 rounding in the Gram matrix) the iterate has lost rank
        floor_pivot = 1e-10 * mx;
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31, nwarps = nt >> 5;
    for (int k = 0; k < r; ++k) {
        if (tid == 0) {
            const double p = S[(int64_t)k * r + k];
            if (!(p > floor_pivot)) bad = 1;
            else S[(int64_t)k * r + k] = sqrt(p);
        }
        __syncthreads();
        if (bad) break;
        const double lkk = S[(int64_t)k * r + k];
        for (int i = k + 1 + tid; i < r; i += nt) S[(int64_t)i * r + k] /= lkk;
        __syncthreads();
        // trailing update of the lower triangle: S[i][j] -= L[i][k] L[j][k], k < j <= i; a warp per row i, its
        // lanes along j
        for (int i = k + 1 + warp; i < r; i += nwarps) {
            const double lik = S[(int64_t)i * r + k];
            for (int j = k + 1 + lane; j <= i; j += 32) S[(int64_t)i * r + j] -= lik * S[(int64_t)j * r + k];
        }
        __syncthreads();
    }
    if (bad) {
        if (tid == 0) flag(check, LOWRAM_CHECK_NOT_PD);
        return;
    }
    for (int64_t e = tid; e < (int64_t)r * r; e += nt) {
        const int i = (int)(e / r), j = (int)(e - (int64_t)i * r);
        Lf[e] = j <= i ? (float)S[e] : 0.0f;
    }
}

// Q = Z R^-1 with R = L^T: each row q of Q solves q L^T = z, i.e. q_j = (z_j - sum_{k<j} q_k L[j][k]) / L[j][j]
// (forward substitution; L's row j is contiguous).  A warp per row; the row's solution so far in shared memory.
constexpr int kTrsmWarps = 8;
__global__ void __launch_bounds__(kTrsmWarps * 32) trsm_rows_kernel(const float* __restrict__ Z,
                                                                    const float* __restrict__ Lf, int D, int r,
                                                                    float* __restrict__ Q) {
    extern __shared__ float xs[];   // [kTrsmWarps][r]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kTrsmWarps + warp;
    if (row >= D) return;
    float* x = xs + warp * r;
    const float* z = Z + (int64_t)row * r;
    for (int j = 0; j < r; ++j) {
        const float* lj = Lf + (int64_t)j * r;
        float acc = 0.0f;
        for (int k = lane; k < j; k += 32) acc = fmaf(x[k], lj[k], acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        const float v = (z[j] - acc) / lj[j];
        if (lane == 0) x[j] = v;
        __syncwarp();
    }
    for (int j = lane; j < r; j += 32) Q[(int64_t)row * r + j] = x[j];
}

// The G output bases, passed by value.
struct BasisPtrs {
    void* p[16];
};

// proj[j][k] = Q[k][j];  basis_l[row][j] = Q[l * H_kv * d + row][j] in the activation dtype
template <typename TA>
__global__ void fit_out_kernel(const float* __restrict__ Q, int D, int r, int rows_per_layer, float* proj,
                               BasisPtrs bases) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)D * r) return;
    const int k = (int)(i / r), j = (int)(i - (int64_t)k * r);
    const float v = Q[i];
    proj[(int64_t)j * D + k] = v;
    const int l = k / rows_per_layer, row = k - l * rows_per_layer;
    TA* bl = (TA*)bases.p[l];
    if constexpr (sizeof(TA) == 2) bl[(int64_t)row * r + j] = __float2bfloat16_rn(v);
    else bl[(int64_t)row * r + j] = v;
}

template <typename TAcc>
cudaError_t gram(const float* X, int64_t N, int D, TAcc* C, int sms, cudaStream_t st) {
    const int nt = (D + kFT - 1) / kFT;
    const int tiles = nt * (nt + 1) / 2;
    int n_split = 1;
    while ((int64_t)tiles * n_split < 4LL * sms && n_split * 2 * kFK * 8 <= N) n_split *= 2;
    if (n_split > 1) {
        cudaError_t e = cudaMemsetAsync(C, 0, sizeof(TAcc) * (size_t)D * D, st);
        if (e != cudaSuccess) return e;
    }
    gram_kernel<TAcc><<<dim3((unsigned)tiles, 1, (unsigned)n_split), kFThreads, 0, st>>>(X, N, D, n_split, n_split > 1, C);
    return cudaGetLastError();
}

cudaError_t sgemm(const float* A, const float* B, int M, int K, int Nc, float* C, cudaStream_t st) {
    const dim3 grid((unsigned)cdiv(Nc, kFT), (unsigned)cdiv(M, kFT));
    sgemm_kernel<<<grid, kFThreads, 0, st>>>(A, B, M, K, Nc, C);
    return cudaGetLastError();
}

}  // namespace

size_t fit_workspace_bytes(int64_t N, int D, int r) {
    auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
    return a(sizeof(float) * (size_t)N * D) + a(sizeof(float) * (size_t)D * D) + 2 * a(sizeof(float) * (size_t)D * r) +
           a(sizeof(double) * (size_t)r * r) + a(sizeof(float) * (size_t)r * r);
}

cudaError_t launch_fit_basis(const FitArgs& f, cudaStream_t st) {
    auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const int64_t N = (int64_t)f.B * f.T;
    const int D = f.G * f.H_kv * f.d, r = f.r;
    char* w = (char*)f.scratch;
    float* X = (float*)w;
    w += a(sizeof(float) * (size_t)N * D);
    float* Gm = (float*)w;
    w += a(sizeof(float) * (size_t)D * D);
    float* Q = (float*)w;
    w += a(sizeof(float) * (size_t)D * r);
    float* Z = (float*)w;
    w += a(sizeof(float) * (size_t)D * r);
    double* S = (double*)w;
    w += a(sizeof(double) * (size_t)r * r);
    float* Lf = (float*)w;

    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t e;
    const int64_t nx = N * D;
    if (f.bf16)
        prep_keys_kernel<__nv_bfloat16><<<(unsigned)cdiv(nx, 256), 256, 0, st>>>(
            (const __nv_bfloat16*)f.keys, N, f.T, D, f.d, f.pos, f.rope_cos, f.rope_sin, f.max_pos, f.post_rope,
            f.check, X);
    else
        prep_keys_kernel<float><<<(unsigned)cdiv(nx, 256), 256, 0, st>>>((const float*)f.keys, N, f.T, D, f.d, f.pos,
                                                                        f.rope_cos, f.rope_sin, f.max_pos,
                                                                        f.post_rope, f.check, X);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = gram<float>(X, N, D, Gm, sms, st)) != cudaSuccess) return e;
    init_normal_kernel<<<(unsigned)cdiv((int64_t)D * r, 256), 256, 0, st>>>(Q, (int64_t)D * r, f.seed);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // Cholesky QR of Z into Q: Z^T Z = L L^T (fp64), Q = Z L^-T by row-wise forward substitution
    const size_t trsm_smem = sizeof(float) * (size_t)kTrsmWarps * r;
    if ((e = cudaFuncSetAttribute(trsm_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)trsm_smem)) !=
        cudaSuccess)
        return e;
    auto chol_qr = [&](const float* Zin, float* Qout) -> cudaError_t {
        cudaError_t e2 = gram<double>(Zin, D, r, S, sms, st);
        if (e2 != cudaSuccess) return e2;
        chol_kernel<<<1, 1024, 0, st>>>(S, r, Lf, f.check);
        if ((e2 = cudaGetLastError()) != cudaSuccess) return e2;
        trsm_rows_kernel<<<(unsigned)cdiv(D, kTrsmWarps), kTrsmWarps * 32, trsm_smem, st>>>(Zin, Lf, D, r, Qout);
        return cudaGetLastError();
    };
    for (int it = 0; it < f.iters; ++it) {
        if ((e = sgemm(Gm, Q, D, D, r, Z, st)) != cudaSuccess) return e;
        if ((e = chol_qr(Z, Q)) != cudaSuccess) return e;
    }
    if ((e = cudaMemcpyAsync(Z, Q, sizeof(float) * (size_t)D * r, cudaMemcpyDeviceToDevice, st)) != cudaSuccess) return e;
    if ((e = chol_qr(Z, Q)) != cudaSuccess) return e;   // second pass: Q^T Q = I to float32 accuracy
    BasisPtrs bp{};
    for (int l = 0; l < f.G; ++l) bp.p[l] = f.basis_out[l];
    const int64_t no = (int64_t)D * r;
    if (f.bf16)
        fit_out_kernel<__nv_bfloat16><<<(unsigned)cdiv(no, 256), 256, 0, st>>>(Q, D, r, f.H_kv * f.d, f.proj_out, bp);
    else
        fit_out_kernel<float><<<(unsigned)cdiv(no, 256), 256, 0, st>>>(Q, D, r, f.H_kv * f.d, f.proj_out, bp);
    return cudaGetLastError();
}

}  // namespace lowram
