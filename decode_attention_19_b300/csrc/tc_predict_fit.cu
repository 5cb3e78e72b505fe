// tc_predict_fit.cu -- the test-time fit of the value predictor with its products on the tensor cores: each Adam
// step's forward and backward products are float32-accurate tcgen05 GEMMs (tc_fit.cu: every float32 operand split
// exactly into three bf16 terms, six bf16 products accumulated in float32), with the elementwise steps between
// them ("LowRAM Paper: Amortised Values and Low-Rank Keys for KV Compression", Abstract: the predictor is fitted at
// test time; "Value cache amortisation in plain language": values are predicted from pre-RoPE keys).
//
// Per kv-head h, with K [N, d] its keys, V [N, d] its values and c = 2 / (N d):
//   Z  = K w1^T                 GEMM (A = K's terms, B = w1's)        H  = silu(Z + b1)
//   Vh = H w2^T                 GEMM (A = H's terms, B = w2's)        E  = Vh + b2 - V,  loss = sum E^2 / (N d),
//                                                                     g_b2 = c sum_t E_t
//   dH = E w2                   GEMM (A = E's terms, B = w2^T's)      dZ = dH * silu'(Z + b1),  g_b1 = c sum_t dZ_t
//   g_w2 = c E^T H              GEMM over the tokens (A = E^T's terms, B = H^T's)
//   g_w1 = c dZ^T K             GEMM over the tokens (A = dZ^T's terms, B = K^T's)
// with silu(z) = z s, silu'(z) = s + z s (1 - s), s = 1 / (1 + e^-z).  The keys' terms (token-major and
// transposed, every head) are written once per fit; the rest once per step and head, in scratch the heads reuse.
// The bias sums and the loss reduce over a CTA's rows in shared memory first, then add once per CTA.
#include "common.cuh"
#include "kernels.h"
#include "predict_fit.h"

namespace lowram {

namespace {

int64_t r128(int64_t x) { return (x + 127) / 128 * 128; }
int64_t r64(int64_t x) { return (x + 63) / 64 * 64; }
size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

struct PfTcLayout {
    int64_t N, Np, dp, mB, m64;
    size_t kn, kt, w1t, w2t, w2tt, z, hb, eb, dz, hn, ht, en, et, dzt, total;
    size_t term(int64_t rows, int64_t cols) const { return a256(2 * (size_t)rows * cols); }
};

// Np: tokens to 128 (rows of A tiles; K of the token reductions); dp, mB: d and m as tile rows (128); m64: m as K
PfTcLayout pf_tc_layout(int64_t N, int H_kv, int d, int m) {
    PfTcLayout L;
    L.N = N;
    L.Np = r128(N);
    L.dp = r128(d);
    L.mB = r128(m);
    L.m64 = r64(m);
    size_t o = 0;
    auto take = [&](size_t& at, size_t bytes) {
        at = o;
        o += bytes;
    };
    take(L.kn, 3 * (size_t)H_kv * L.term(L.Np, d));      // K's terms [H_kv][Np, d]
    take(L.kt, 3 * (size_t)H_kv * L.term(L.dp, L.Np));   // K^T's terms [H_kv][dp, Np]
    take(L.w1t, 3 * L.term(L.mB, d));                    // w1_h [m, d]
    take(L.w2t, 3 * L.term(L.dp, L.m64));                // w2_h [d, m]
    take(L.w2tt, 3 * L.term(L.mB, d));                   // w2_h^T [m, d]
    take(L.z, a256(sizeof(float) * (size_t)N * m));      // Z
    take(L.hb, a256(sizeof(float) * (size_t)N * m));     // H
    take(L.eb, a256(sizeof(float) * (size_t)N * d));     // Vh, then E
    take(L.dz, a256(sizeof(float) * (size_t)N * m));     // dH, then dZ
    take(L.hn, 3 * L.term(L.Np, L.m64));                 // H's terms
    take(L.ht, 3 * L.term(L.mB, L.Np));                  // H^T's
    take(L.en, 3 * L.term(L.Np, d));                     // E's
    take(L.et, 3 * L.term(L.dp, L.Np));                  // E^T's
    take(L.dzt, 3 * L.term(L.mB, L.Np));                 // dZ^T's
    L.total = o;
    return L;
}

void terms_at(char* base, size_t off, size_t step, void* (&t)[3]) {
    for (int i = 0; i < 3; ++i) t[i] = base + off + i * step;
}

__device__ __forceinline__ float sigmoid(float z) { return 1.0f / (1.0f + expf(-z)); }

// H = silu(Z + b1) over [N, m]
__global__ void pf_act_kernel(const float* __restrict__ Z, const float* __restrict__ b1, int64_t n, int m,
                              float* __restrict__ H) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float z = Z[i] + b1[i % m];
    H[i] = z * sigmoid(z);
}

// Column reductions over a CTA's rows: thread (tx, ty) of 32 x 8 takes column blockIdx.x*32 + tx and rows
// blockIdx.y*kPfRows + ty, + 8, ...; the CTA adds its column sums (and its sum of squares) once.
constexpr int kPfRows = 256;

// E = Vh + b2 - V (in place), loss[h] += sum E^2 / (N d), g_b2 += c sum_t E_t
template <typename TA>
__global__ void __launch_bounds__(256) pf_err_kernel(float* __restrict__ E, const float* __restrict__ b2,
                                                     const TA* __restrict__ V, int64_t N, int H_kv, int h, int d,
                                                     float c, float* __restrict__ g_b2, float* __restrict__ loss) {
    __shared__ float cs[8][33], sq[8];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5, j = blockIdx.x * 32 + tx;
    float col = 0.0f, ss = 0.0f;
    if (j < d) {
        const float bj = b2[j];
        const int64_t t1 = min(N, (int64_t)(blockIdx.y + 1) * kPfRows);
        for (int64_t t = (int64_t)blockIdx.y * kPfRows + ty; t < t1; t += 8) {
            const float e = E[t * d + j] + bj - ld(V, (t * H_kv + h) * d + j);
            E[t * d + j] = e;
            col += e;
            ss += e * e;
        }
    }
    cs[ty][tx] = col;
    ss = warp_sum(ss);
    if (tx == 0) sq[ty] = ss;
    __syncthreads();
    if (ty == 0) {
        float a = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) a += cs[k][tx];
        if (j < d) atomicAdd(&g_b2[j], c * a);
        if (tx == 0) {
            float q = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) q += sq[k];
            atomicAdd(loss, q / ((float)N * (float)d));
        }
    }
}

// dZ = dH * silu'(Z + b1) (in place over dH), g_b1 += c sum_t dZ_t
__global__ void __launch_bounds__(256) pf_dz_kernel(float* __restrict__ dZ, const float* __restrict__ Z,
                                                    const float* __restrict__ b1, int64_t N, int m, float c,
                                                    float* __restrict__ g_b1) {
    __shared__ float cs[8][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5, j = blockIdx.x * 32 + tx;
    float col = 0.0f;
    if (j < m) {
        const float bj = b1[j];
        const int64_t t1 = min(N, (int64_t)(blockIdx.y + 1) * kPfRows);
        for (int64_t t = (int64_t)blockIdx.y * kPfRows + ty; t < t1; t += 8) {
            const float z = Z[t * m + j] + bj, s = sigmoid(z);
            const float g = dZ[t * m + j] * (s + z * s * (1.0f - s));
            dZ[t * m + j] = g;
            col += g;
        }
    }
    cs[ty][tx] = col;
    __syncthreads();
    if (ty == 0 && j < m) {
        float a = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) a += cs[k][tx];
        atomicAdd(&g_b1[j], c * a);
    }
}

__global__ void pf_scale_kernel(float* __restrict__ g, int64_t n, float c) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) g[i] *= c;
}

}  // namespace

size_t predictor_tc_scratch_bytes(int64_t N, int H_kv, int d, int m) { return pf_tc_layout(N, H_kv, d, m).total; }

// The token-major split passes put 32 output rows (tokens) per grid row, and a grid has at most 65535 rows.
int64_t predictor_tc_max_tokens() { return 65535LL * 32; }

cudaError_t launch_predictor_prep_tc(const PredictorFitArgs& a, void* scratch, cudaStream_t st) {
    const int64_t N = (int64_t)a.B * a.T;
    if (N == 0) return cudaSuccess;
    const PfTcLayout L = pf_tc_layout(N, a.H_kv, a.d, a.m);
    char* w = (char*)scratch;
    const size_t kn1 = L.term(L.Np, a.d), kt1 = L.term(L.dp, L.Np);
    cudaError_t e = cudaSuccess;
    for (int h = 0; h < a.H_kv && e == cudaSuccess; ++h) {
        const size_t esz = a.bf16 ? 2 : 4;
        const void* src = (const char*)a.keys + (size_t)h * a.d * esz;
        void *kn[3], *kt[3];
        terms_at(w, L.kn + (size_t)h * 3 * kn1, kn1, kn);
        terms_at(w, L.kt + (size_t)h * 3 * kt1, kt1, kt);
        e = launch_split3(src, a.bf16, (int)N, a.d, (int64_t)a.H_kv * a.d, false, (int)L.Np, a.d, kn, st);
        if (e == cudaSuccess)
            e = launch_split3(src, a.bf16, (int)N, a.d, (int64_t)a.H_kv * a.d, true, (int)L.dp, (int)L.Np, kt, st);
    }
    return e;
}

cudaError_t launch_predictor_grad_tc(const PredictorFitArgs& a, void* scratch, uint32_t* check, cudaStream_t st) {
    const int64_t N = (int64_t)a.B * a.T;
    const int d = a.d, m = a.m, H_kv = a.H_kv;
    const size_t n1 = (size_t)H_kv * m * d;
    cudaError_t e;
    if ((e = cudaMemsetAsync(a.g_b1, 0, sizeof(float) * (size_t)H_kv * m, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.g_b2, 0, sizeof(float) * (size_t)H_kv * d, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.loss, 0, sizeof(float) * H_kv, st)) != cudaSuccess) return e;
    if (N == 0) {
        if ((e = cudaMemsetAsync(a.g_w1, 0, sizeof(float) * n1, st)) != cudaSuccess) return e;
        return cudaMemsetAsync(a.g_w2, 0, sizeof(float) * n1, st);
    }
    const PfTcLayout L = pf_tc_layout(N, H_kv, d, m);
    char* w = (char*)scratch;
    const float c = 2.0f / ((float)N * (float)d);
    const int Np = (int)L.Np, dp = (int)L.dp, mB = (int)L.mB, m64 = (int)L.m64;
    float* Z = (float*)(w + L.z);
    float* Hb = (float*)(w + L.hb);
    float* Eb = (float*)(w + L.eb);
    float* dZ = (float*)(w + L.dz);
    void *w1t[3], *w2t[3], *w2tt[3], *hn[3], *ht[3], *en[3], *et[3], *dzt[3];
    terms_at(w, L.w1t, L.term(L.mB, d), w1t);
    terms_at(w, L.w2t, L.term(L.dp, L.m64), w2t);
    terms_at(w, L.w2tt, L.term(L.mB, d), w2tt);
    terms_at(w, L.hn, L.term(L.Np, L.m64), hn);
    terms_at(w, L.ht, L.term(L.mB, L.Np), ht);
    terms_at(w, L.en, L.term(L.Np, d), en);
    terms_at(w, L.et, L.term(L.dp, L.Np), et);
    terms_at(w, L.dzt, L.term(L.mB, L.Np), dzt);
    const size_t kn1 = L.term(L.Np, d), kt1 = L.term(L.dp, L.Np);
    const dim3 red_d((unsigned)cdiv(d, 32), (unsigned)cdiv(N, kPfRows)), red_m((unsigned)cdiv(m, 32), (unsigned)cdiv(N, kPfRows));
    const unsigned ew = (unsigned)cdiv(N * m, 256);
    for (int h = 0; h < H_kv; ++h) {
        const float* w1h = a.w1 + (size_t)h * m * d;
        const float* w2h = a.w2 + (size_t)h * d * m;
        const float* b1h = a.b1 + (size_t)h * m;
        void *kn[3], *kt[3];
        terms_at(w, L.kn + (size_t)h * 3 * kn1, kn1, kn);
        terms_at(w, L.kt + (size_t)h * 3 * kt1, kt1, kt);
        // this head's weights as terms: w1 [m, d], w2 [d, m], w2^T [m, d]
        if ((e = launch_split3(w1h, false, m, d, d, false, mB, d, w1t, st)) != cudaSuccess) return e;
        if ((e = launch_split3(w2h, false, d, m, m, false, dp, m64, w2t, st)) != cudaSuccess) return e;
        if ((e = launch_split3(w2h, false, d, m, m, true, mB, d, w2tt, st)) != cudaSuccess) return e;
        // forward
        if ((e = launch_split_gemm_tc(kn, w1t, (int)N, m, Np, mB, d, false, Z, m, check, st)) != cudaSuccess) return e;
        pf_act_kernel<<<ew, 256, 0, st>>>(Z, b1h, N * m, m, Hb);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = launch_split3(Hb, false, (int)N, m, m, false, Np, m64, hn, st)) != cudaSuccess) return e;
        if ((e = launch_split3(Hb, false, (int)N, m, m, true, mB, Np, ht, st)) != cudaSuccess) return e;
        if ((e = launch_split_gemm_tc(hn, w2t, (int)N, d, Np, dp, m64, false, Eb, d, check, st)) != cudaSuccess)
            return e;
        if (a.bf16)
            pf_err_kernel<__nv_bfloat16><<<red_d, 256, 0, st>>>(Eb, a.b2 + (size_t)h * d,
                                                                (const __nv_bfloat16*)a.values, N, H_kv, h, d, c,
                                                                a.g_b2 + (size_t)h * d, a.loss + h);
        else
            pf_err_kernel<float><<<red_d, 256, 0, st>>>(Eb, a.b2 + (size_t)h * d, (const float*)a.values, N, H_kv, h,
                                                        d, c, a.g_b2 + (size_t)h * d, a.loss + h);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // backward
        if ((e = launch_split3(Eb, false, (int)N, d, d, false, Np, d, en, st)) != cudaSuccess) return e;
        if ((e = launch_split3(Eb, false, (int)N, d, d, true, dp, Np, et, st)) != cudaSuccess) return e;
        if ((e = launch_split_gemm_tc(en, w2tt, (int)N, m, Np, mB, d, false, dZ, m, check, st)) != cudaSuccess)
            return e;
        pf_dz_kernel<<<red_m, 256, 0, st>>>(dZ, Z, b1h, N, m, c, a.g_b1 + (size_t)h * m);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = launch_split3(dZ, false, (int)N, m, m, true, mB, Np, dzt, st)) != cudaSuccess) return e;
        if ((e = launch_split_gemm_tc(et, ht, d, m, dp, mB, Np, false, a.g_w2 + (size_t)h * d * m, m, check, st)) !=
            cudaSuccess)
            return e;
        if ((e = launch_split_gemm_tc(dzt, kt, m, d, mB, dp, Np, false, a.g_w1 + (size_t)h * m * d, d, check, st)) !=
            cudaSuccess)
            return e;
    }
    pf_scale_kernel<<<(unsigned)cdiv((int64_t)n1, 256), 256, 0, st>>>(a.g_w1, (int64_t)n1, c);
    pf_scale_kernel<<<(unsigned)cdiv((int64_t)n1, 256), 256, 0, st>>>(a.g_w2, (int64_t)n1, c);
    return cudaGetLastError();
}

}  // namespace lowram
