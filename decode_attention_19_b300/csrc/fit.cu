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
// Kernels: a key prep pass (dtype, inverse RoPE); the Gram matrix and each step's product Z = (X^T X) Q on the
// tensor cores in float32 accuracy (tc_fit.cu: an exact three-term bf16 split of the float32 operands, six bf16
// products accumulated in float32); Z^T Z in fp64 on the CUDA cores (64 x 64 upper-triangle tiles, mirrored, split
// over rows with atomics when the tiles alone do not fill the GPU); a blocked multi-CTA fp64 Cholesky; a
// row-parallel triangular solve; and the output pass.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

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
    // operands converted once, on their way into shared memory (an fp64 conversion costs as much as an fp64 FMA)
    __shared__ TAcc As[kFK][kFT + 4], Bs[kFK][kFT + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    TAcc acc[4][4] = {};
    for (int64_t n0 = n_begin; n0 < n_end; n0 += kFK) {
        for (int e = tid; e < kFK * kFT; e += kFThreads) {
            const int r = e / kFT, c = e % kFT;
            const int64_t n = n0 + r;
            As[r][c] = (TAcc)((n < n_end && i0 + c < D) ? X[n * D + i0 + c] : 0.0f);
            Bs[r][c] = (TAcc)((n < n_end && j0 + c < D) ? X[n * D + j0 + c] : 0.0f);
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kFK; ++k) {
            TAcc a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a[u] = As[k][ty * 4 + u];
                b[u] = Bs[k][tx * 4 + u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] += a[u] * b[v];
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

// Blocked Cholesky of S [r, r] fp64 (S = L L^T, L lower, written over S's lower triangle), panel by panel
// (kCb columns) over many CTAs: the panel's diagonal block is factored by one CTA, the rows below it are solved
// against it (L21 = S21 L11^-T) a warp per row, and the trailing lower triangle takes the panel's product
// (S22 -= L21 L21^T) in 16 x 16 tiles.  A pivot at or below 1e-10 of the largest diagonal entry of S (rounding
// noise of float32 iterates: the keys have rank below r) sets LOWRAM_CHECK_NOT_PD; every later kernel of the
// factorization then returns at once and the fit's result is void.  The float32 copy Lf [r, r] (lower
// triangle; zeros above) is what the triangular solve reads.
constexpr int kCb = 32;
constexpr int kCT = 16;      // trailing-update tile edge

__device__ __forceinline__ bool not_pd(const uint32_t* check) {
    return check && (*(volatile const uint32_t*)check & LOWRAM_CHECK_NOT_PD);
}

// pivot floor: 1e-10 of the largest diagonal entry of S (the pivots are ~ (lambda_k / lambda_1)^2 of it: below
// 1e-10, an eigenvalue under 1e-5 of the largest, the level of float32 rounding in the Gram matrix, the iterate
// has lost rank)
__global__ void __launch_bounds__(256) chol_floor_kernel(const double* __restrict__ S, int r, double* floor_out) {
    __shared__ double wm[8];
    double mx = 0.0;
    for (int k = threadIdx.x; k < r; k += 256) mx = fmax(mx, S[(int64_t)k * r + k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < 8; ++w) mx = fmax(mx, wm[w]);
        *floor_out = 1e-10 * fmax(mx, wm[0]);
    }
}

// the diagonal block of panel k0 (kb x kb): thread (i, j) = (warp, lane) holds element (i, j) of the lower
// triangle in a register; per pivot k the pivot thread takes one reciprocal square root, the column threads scale
// and publish column k, and every thread below and right of the pivot takes its one product
__global__ void __launch_bounds__(kCb * kCb) chol_diag_kernel(double* S, int r, int k0, const double* floor_p,
                                                              uint32_t* check) {
    if (not_pd(check)) return;
    __shared__ double col[kCb];
    __shared__ double s_rl;
    __shared__ int s_bad;
    const int kb = min(kCb, r - k0), i = threadIdx.x >> 5, j = threadIdx.x & 31;
    const bool in = i < kb && j <= i;
    double a = in ? S[(int64_t)(k0 + i) * r + k0 + j] : 0.0;
    const double fl = *floor_p;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int k = 0; k < kb; ++k) {
        if (i == k && j == k) {
            if (!(a > fl)) {
                s_bad = 1;
            } else {
                const double rl = rsqrt(a);   // 1 / l_kk
                s_rl = rl;
                a *= rl;                      // l_kk
            }
        }
        __syncthreads();
        if (s_bad) break;                     // the same answer in every thread
        if (j == k && i > k && i < kb) {
            a *= s_rl;                        // l_ik
            col[i] = a;
        }
        __syncthreads();
        if (in && j > k) a -= col[i] * col[j];   // i >= j > k
    }
    if (s_bad) {
        if (threadIdx.x == 0) flag(check, LOWRAM_CHECK_NOT_PD);
        return;
    }
    if (in) S[(int64_t)(k0 + i) * r + k0 + j] = a;
}

// rows i >= k0 + kb of panel k0, a warp per row, lane t holding s_it: right-looking, so step j needs no reduction:
// l_ij = s_ij / l_jj is final on lane j, and every lane t > j takes s_it -= l_ij l_tj
constexpr int kCRowWarps = 4;
__global__ void __launch_bounds__(kCRowWarps * 32) chol_rows_kernel(double* S, int r, int k0, const uint32_t* check) {
    if (not_pd(check)) return;
    __shared__ double Lb[kCb][kCb + 1], rinv[kCb];
    const int kb = min(kCb, r - k0), k1 = k0 + kb, tid = threadIdx.x;
    for (int e = tid; e < kb * kb; e += kCRowWarps * 32) {
        const int i = e / kb, j = e - (e / kb) * kb;
        Lb[i][j] = j <= i ? S[(int64_t)(k0 + i) * r + k0 + j] : 0.0;
    }
    if (tid < kb) rinv[tid] = 1.0 / S[(int64_t)(k0 + tid) * r + k0 + tid];   // one division per lane, in parallel
    __syncthreads();
    const int lane = tid & 31, i = k1 + blockIdx.x * kCRowWarps + (tid >> 5);
    if (i >= r) return;
    double* row = S + (int64_t)i * r + k0;
    double v = lane < kb ? row[lane] : 0.0;
    for (int j = 0; j < kb; ++j) {
        const double lj = __shfl_sync(0xffffffffu, v * rinv[j], j);
        if (lane == j) v = lj;
        else if (lane > j && lane < kb) v -= lj * Lb[lane][j];
    }
    if (lane < kb) row[lane] = v;
}

// S[i][j] -= sum_{t < kb} L[i][k0 + t] L[j][k0 + t] for k0 + kb <= j <= i < r, a 16 x 16 tile per CTA
__global__ void __launch_bounds__(kCT * kCT) chol_update_kernel(double* S, int r, int k0, const uint32_t* check) {
    if (not_pd(check)) return;
    __shared__ double Li[kCT][kCb + 1], Lj[kCT][kCb + 1];
    const int kb = min(kCb, r - k0), k1 = k0 + kb;
    const int nt = (int)cdiv(r - k1, kCT);
    int lin = blockIdx.x, bi = 0;                    // lower-triangle tile (bj <= bi) from the linear index
    while (lin > bi) {
        lin -= bi + 1;
        ++bi;
    }
    const int bj = lin;
    if (bi >= nt) return;
    const int i0 = k1 + bi * kCT, j0 = k1 + bj * kCT, tid = threadIdx.x;
    for (int e = tid; e < kCT * kb; e += kCT * kCT) {
        const int a = e / kb, q = e - (e / kb) * kb;
        Li[a][q] = i0 + a < r ? S[(int64_t)(i0 + a) * r + k0 + q] : 0.0;
        Lj[a][q] = j0 + a < r ? S[(int64_t)(j0 + a) * r + k0 + q] : 0.0;
    }
    __syncthreads();
    const int a = tid / kCT, c = tid % kCT, i = i0 + a, j = j0 + c;
    if (i >= r || j > i) return;
    double acc = 0.0;
    for (int q = 0; q < kb; ++q) acc += Li[a][q] * Lj[c][q];
    S[(int64_t)i * r + j] -= acc;
}

__global__ void chol_out_kernel(const double* __restrict__ S, int r, float* __restrict__ Lf, const uint32_t* check) {
    if (not_pd(check)) return;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= (int64_t)r * r) return;
    const int i = (int)(e / r), j = (int)(e - (e / r) * r);
    Lf[e] = j <= i ? (float)S[e] : 0.0f;
}

cudaError_t cholesky(double* S, int r, float* Lf, double* floor_p, uint32_t* check, cudaStream_t st) {
    chol_floor_kernel<<<1, 256, 0, st>>>(S, r, floor_p);
    cudaError_t e = cudaGetLastError();
    for (int k0 = 0; k0 < r && e == cudaSuccess; k0 += kCb) {
        const int kb = std::min(kCb, r - k0), n = r - k0 - kb;
        chol_diag_kernel<<<1, kCb * kCb, 0, st>>>(S, r, k0, floor_p, check);
        if (n > 0) {
            chol_rows_kernel<<<(unsigned)cdiv(n, kCRowWarps), kCRowWarps * 32, 0, st>>>(S, r, k0, check);
            const int nt = (int)cdiv(n, kCT);
            chol_update_kernel<<<(unsigned)(nt * (nt + 1) / 2), kCT * kCT, 0, st>>>(S, r, k0, check);
        }
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    chol_out_kernel<<<(unsigned)cdiv((int64_t)r * r, 256), 256, 0, st>>>(S, r, Lf, check);
    return cudaGetLastError();
}

// Q = Z R^-1 with R = L^T: each row q of Q solves q L^T = z, i.e. q_j = (z_j - sum_{k<j} q_k L[j][k]) / L[j][j]
// (forward substitution; L's row j is contiguous, and zero above the diagonal).  A warp solves ROWS rows together,
// so each row of L it reads from L2 serves all of them; the rows' solutions so far live in shared memory.  The
// first 512 columns of L's next row are loaded into registers while the current row is applied (16 a lane), so
// the steps do not wait on L2 one after another; columns past 512 (r > 512) are loaded in batches of 512.
constexpr int kTrsmWarps = 8;
constexpr int kTrsmPre = 16;   // L values a lane holds per batch: 512 columns a warp
template <int ROWS>
__global__ void __launch_bounds__(kTrsmWarps * 32) trsm_rows_kernel(const float* __restrict__ Z,
                                                                    const float* __restrict__ Lf, int D, int r,
                                                                    float* __restrict__ Q) {
    extern __shared__ float xs[];   // [kTrsmWarps][ROWS][r]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * kTrsmWarps + warp) * ROWS;
    if (row0 >= D) return;
    float* x = xs + (size_t)warp * ROWS * r;
    for (int e = lane; e < ROWS * r; e += 32) x[e] = 0.0f;   // rows past D stay zero
    __syncwarp();
    auto load_batch = [&](const float* lrow, int kb, float (&v)[kTrsmPre]) {
#pragma unroll
        for (int u = 0; u < kTrsmPre; ++u) {
            const int k = kb + u * 32 + lane;
            v[u] = k < r ? lrow[k] : 0.0f;
        }
    };
    float nxt[kTrsmPre];
    load_batch(Lf, 0, nxt);
    for (int j = 0; j < r; ++j) {
        const float* lj = Lf + (int64_t)j * r;
        float cur[kTrsmPre];
#pragma unroll
        for (int u = 0; u < kTrsmPre; ++u) cur[u] = nxt[u];
        if (j + 1 < r) load_batch(lj + r, 0, nxt);            // row j+1, in flight during this step
        const float ljj = lj[j];
        const float zq = lane < ROWS && row0 + lane < D ? Z[(int64_t)(row0 + lane) * r + j] : 0.0f;
        float acc[ROWS];
#pragma unroll
        for (int q = 0; q < ROWS; ++q) acc[q] = 0.0f;
#pragma unroll
        for (int u = 0; u < kTrsmPre; ++u) {
            if (u * 32 >= j) break;                            // uniform over the warp
            const int k = u * 32 + lane;
            if (k < j)
#pragma unroll
                for (int q = 0; q < ROWS; ++q) acc[q] = fmaf(x[q * r + k], cur[u], acc[q]);
        }
        for (int kb = kTrsmPre * 32; kb < j; kb += kTrsmPre * 32) {
            float v[kTrsmPre];
            load_batch(lj, kb, v);
#pragma unroll
            for (int u = 0; u < kTrsmPre; ++u) {
                const int k = kb + u * 32 + lane;
                if (k < j)
#pragma unroll
                    for (int q = 0; q < ROWS; ++q) acc[q] = fmaf(x[q * r + k], v[u], acc[q]);
            }
        }
#pragma unroll
        for (int q = 0; q < ROWS; ++q)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
        float mine = acc[0];                       // lane q finishes row q
#pragma unroll
        for (int q = 1; q < ROWS; ++q)
            if (lane == q) mine = acc[q];
        if (lane < ROWS && row0 + lane < D) x[lane * r + j] = (zq - mine) / ljj;
        __syncwarp();
    }
    for (int q = 0; q < ROWS && row0 + q < D; ++q)
        for (int j = lane; j < r; j += 32) Q[(int64_t)(row0 + q) * r + j] = x[q * r + j];
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

}  // namespace

// Workspace: X [N, D] float32; the three bf16 terms of X^T [Dp, Np], of the Gram matrix [Dp, Dp] and of Q^T
// [Rp, Dp] (Np = N rounded up to 64, Dp = D to 256, Rp = r to 256: the tensor-core tiles); the Gram matrix [D, D],
// Q and Z [D, r] float32; S [r, r] fp64, Lf [r, r] float32 and the pivot floor.
namespace {
struct FitLayout {
    int64_t Np, Dp, Rp;
    size_t x, xt, gm, gt, qt, q, z, s, lf, fl, total;
};
FitLayout fit_layout(int64_t N, int D, int r) {
    auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
    FitLayout L;
    L.Np = cdiv(N, 64) * 64;
    L.Dp = cdiv(D, 256) * 256;
    L.Rp = cdiv(r, 256) * 256;
    size_t o = 0;
    L.x = o;
    o += a(sizeof(float) * (size_t)N * D);
    L.xt = o;
    o += 3 * a(2 * (size_t)L.Dp * L.Np);
    L.gm = o;
    o += a(sizeof(float) * (size_t)D * D);
    L.gt = o;
    o += 3 * a(2 * (size_t)L.Dp * L.Dp);
    L.qt = o;
    o += 3 * a(2 * (size_t)L.Rp * L.Dp);
    L.q = o;
    o += a(sizeof(float) * (size_t)D * r);
    L.z = o;
    o += a(sizeof(float) * (size_t)D * r);
    L.s = o;
    o += a(sizeof(double) * (size_t)r * r);
    L.lf = o;
    o += a(sizeof(float) * (size_t)r * r);
    L.fl = o;
    o += a(sizeof(double));
    L.total = o;
    return L;
}
}  // namespace

size_t fit_workspace_bytes(int64_t N, int D, int r) { return fit_layout(N, D, r).total; }

cudaError_t launch_fit_basis(const FitArgs& f, cudaStream_t st) {
    const int64_t N = (int64_t)f.B * f.T;
    const int D = f.G * f.H_kv * f.d, r = f.r;
    const FitLayout L = fit_layout(N, D, r);
    char* w = (char*)f.scratch;
    float* X = (float*)(w + L.x);
    auto terms = [&](size_t off, int64_t rows, int64_t cols, void* (&t)[3]) {
        const size_t step = ((2 * (size_t)rows * cols) + 255) & ~(size_t)255;
        for (int i = 0; i < 3; ++i) t[i] = w + off + i * step;
    };
    void *Xt[3], *Gt[3], *Qt[3];
    terms(L.xt, L.Dp, L.Np, Xt);
    terms(L.gt, L.Dp, L.Dp, Gt);
    terms(L.qt, L.Rp, L.Dp, Qt);
    float* Gm = (float*)(w + L.gm);
    float* Q = (float*)(w + L.q);
    float* Z = (float*)(w + L.z);
    double* S = (double*)(w + L.s);
    float* Lf = (float*)(w + L.lf);
    double* floor_p = (double*)(w + L.fl);

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
    // Gram matrix X^T X on the tensor cores: the terms of X^T [Dp, Np] (reduction over tokens along the rows)
    if ((e = launch_split3(X, false, (int)N, D, D, true, (int)L.Dp, (int)L.Np, Xt, st)) != cudaSuccess) return e;
    if ((e = launch_split_gemm_tc(Xt, Xt, D, D, (int)L.Dp, (int)L.Dp, (int)L.Np, true, Gm, D, f.check, st)) !=
        cudaSuccess)
        return e;
    if ((e = launch_split3(Gm, false, D, D, D, false, (int)L.Dp, (int)L.Dp, Gt, st)) != cudaSuccess) return e;
    init_normal_kernel<<<(unsigned)cdiv((int64_t)D * r, 256), 256, 0, st>>>(Q, (int64_t)D * r, f.seed);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // Cholesky QR of Z into Q: Z^T Z = L L^T (fp64), Q = Z L^-T by row-wise forward substitution
    // four rows per warp while their solutions fit in shared memory, else one
    const bool four = sizeof(float) * (size_t)kTrsmWarps * 4 * r <= 200 * 1024;
    const int trsm_rows = four ? 4 : 1;
    const size_t trsm_smem = sizeof(float) * (size_t)kTrsmWarps * trsm_rows * r;
    if ((e = cudaFuncSetAttribute(four ? trsm_rows_kernel<4> : trsm_rows_kernel<1>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)trsm_smem)) != cudaSuccess)
        return e;
    auto chol_qr = [&](const float* Zin, float* Qout) -> cudaError_t {
        cudaError_t e2 = gram<double>(Zin, D, r, S, sms, st);
        if (e2 != cudaSuccess) return e2;
        if ((e2 = cholesky(S, r, Lf, floor_p, f.check, st)) != cudaSuccess) return e2;
        const unsigned grid = (unsigned)cdiv(D, kTrsmWarps * trsm_rows);
        if (four) trsm_rows_kernel<4><<<grid, kTrsmWarps * 32, trsm_smem, st>>>(Zin, Lf, D, r, Qout);
        else trsm_rows_kernel<1><<<grid, kTrsmWarps * 32, trsm_smem, st>>>(Zin, Lf, D, r, Qout);
        return cudaGetLastError();
    };
    for (int it = 0; it < f.iters; ++it) {
        // Z = G Q on the tensor cores: the terms of Q^T [Rp, Dp]
        if ((e = launch_split3(Q, false, D, r, r, true, (int)L.Rp, (int)L.Dp, Qt, st)) != cudaSuccess) return e;
        if ((e = launch_split_gemm_tc(Gt, Qt, D, r, (int)L.Dp, (int)L.Rp, (int)L.Dp, false, Z, r, f.check, st)) !=
            cudaSuccess)
            return e;
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
