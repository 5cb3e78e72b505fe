// dense.cu -- comparator: split-T decode attention over an explicit, uncompressed, already rotated
// K/V cache [B, T, H_kv, d].  Same split-softmax partial layout and merge kernel as the compressed
// path.  This is the cache the compressed one replaces (LowRAM abstract: the KV cache's memory
// footprint caps batch size and throughput).
//
// HBM-bound: every K and V byte is read once with 16-byte loads.  A group of d/VEC lanes holds one
// token (VEC elements per lane); the lanes of a group reduce the q.k dot products with xor shuffles
// and keep an online softmax state per q-head; groups, then warps, merge their states at the end.
#include "common.cuh"
#include "kernels.h"

namespace lowram {

constexpr int kDenseThreads = 128;

template <typename TE>
struct Vec16;
template <>
struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void load(const __nv_bfloat16* p, float (&x)[8]) {
        uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
};
template <>
struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void load(const float* p, float (&x)[4]) {
        float4 u = __ldg(reinterpret_cast<const float4*>(p));
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    }
};

// merge (m2, l2, a2) into (m, l, a)
template <int V>
__device__ __forceinline__ void merge_state(float& m, float& l, float (&a)[V], float m2, float l2, const float (&a2)[V]) {
    const float M = fmaxf(m, m2);
    const float f1 = (m == -INFINITY) ? 0.0f : __expf(m - M);
    const float f2 = (m2 == -INFINITY) ? 0.0f : __expf(m2 - M);
    l = l * f1 + l2 * f2;
#pragma unroll
    for (int e = 0; e < V; ++e) a[e] = a[e] * f1 + a2[e] * f2;
    m = M;
}

template <typename TE, int D, int G>
__global__ void __launch_bounds__(kDenseThreads) dense_kernel(int T, int H_q, int H_kv, float scale,
                                                              const TE* __restrict__ q, const TE* __restrict__ K,
                                                              const TE* __restrict__ V, float* __restrict__ partial,
                                                              int n_split) {
    constexpr int VEC = Vec16<TE>::N;
    constexpr int LPT = D / VEC;          // lanes per token
    constexpr int TPW = 32 / LPT;         // tokens per warp step
    constexpr int NW = kDenseThreads / 32;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, grp = lane / LPT, sub = lane % LPT;
    const int per = (int)cdiv(T, n_split);
    const int t_begin = split * per, t_end = min(T, t_begin + per);

    float qv[G][VEC];
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
        for (int e = 0; e < VEC; ++e) qv[j][e] = ld(q, ((int64_t)b * H_q + h * G + j) * D + sub * VEC + e) * scale;

    float m[G], l[G], acc[G][VEC];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.0f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[j][e] = 0.0f;
    }
    for (int t0 = t_begin + warp * TPW; t0 < t_end; t0 += NW * TPW) {
        const int t = t0 + grp;
        const bool valid = t < t_end;
        float kx[VEC], vx[VEC];
        if (valid) {
            const int64_t off = (((int64_t)b * T + t) * H_kv + h) * D + sub * VEC;
            Vec16<TE>::load(K + off, kx);
            Vec16<TE>::load(V + off, vx);
        }
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float s = 0.0f;
            if (valid)
#pragma unroll
                for (int e = 0; e < VEC; ++e) s = fmaf(qv[j][e], kx[e], s);
#pragma unroll
            for (int o = LPT / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (valid) {
                const float mn = fmaxf(m[j], s);
                const float corr = (m[j] == -INFINITY) ? 0.0f : __expf(m[j] - mn);
                const float p = __expf(s - mn);
                l[j] = l[j] * corr + p;
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[j][e] = fmaf(p, vx[e], acc[j][e] * corr);
                m[j] = mn;
            }
        }
    }
    // merge the token groups of the warp (lanes with the same sub hold the same features)
#pragma unroll
    for (int o = LPT; o < 32; o <<= 1) {
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float m2 = __shfl_xor_sync(0xffffffffu, m[j], o), l2 = __shfl_xor_sync(0xffffffffu, l[j], o);
            float a2[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) a2[e] = __shfl_xor_sync(0xffffffffu, acc[j][e], o);
            merge_state<VEC>(m[j], l[j], acc[j], m2, l2, a2);
        }
    }
    // merge the warps through shared memory
    __shared__ float sm_m[NW][G], sm_l[NW][G], sm_a[NW][G][D];
    if (grp == 0) {
#pragma unroll
        for (int j = 0; j < G; ++j) {
            if (sub == 0) {
                sm_m[warp][j] = m[j];
                sm_l[warp][j] = l[j];
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) sm_a[warp][j][sub * VEC + e] = acc[j][e];
        }
    }
    __syncthreads();
    if (warp == 0 && grp == 0) {
#pragma unroll
        for (int w = 1; w < NW; ++w)
#pragma unroll
            for (int j = 0; j < G; ++j) {
                float a2[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) a2[e] = sm_a[w][j][sub * VEC + e];
                merge_state<VEC>(m[j], l[j], acc[j], sm_m[w][j], sm_l[w][j], a2);
            }
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float* dst = partial + (((int64_t)b * H_q + h * G + j) * n_split + split) * (D + 2);
#pragma unroll
            for (int e = 0; e < VEC; ++e) dst[sub * VEC + e] = acc[j][e];
            if (sub == 0) {
                dst[D] = m[j];
                dst[D + 1] = l[j];
            }
        }
    }
}

int dense_splits(int B, int T, int H_kv) {
    const int64_t units = (int64_t)B * H_kv;
    if (units == 0 || T == 0) return 1;
    int64_t s = cdiv(148 * 8, units);
    s = s < 1 ? 1 : s;
    const int64_t cap = cdiv(T, 128);
    return (int)(s > cap ? cap : s);
}

template <typename TE, int D>
static cudaError_t dense_g(int B, int T, int H_q, int H_kv, float scale, const void* q, const void* k, const void* v,
                           float* partial, int n_split, cudaStream_t st) {
    dim3 grid((unsigned)n_split, (unsigned)H_kv, (unsigned)B);
    const TE *Q = (const TE*)q, *K = (const TE*)k, *V = (const TE*)v;
    switch (H_q / H_kv) {
        case 1: dense_kernel<TE, D, 1><<<grid, kDenseThreads, 0, st>>>(T, H_q, H_kv, scale, Q, K, V, partial, n_split); break;
        case 2: dense_kernel<TE, D, 2><<<grid, kDenseThreads, 0, st>>>(T, H_q, H_kv, scale, Q, K, V, partial, n_split); break;
        case 4: dense_kernel<TE, D, 4><<<grid, kDenseThreads, 0, st>>>(T, H_q, H_kv, scale, Q, K, V, partial, n_split); break;
        case 7: dense_kernel<TE, D, 7><<<grid, kDenseThreads, 0, st>>>(T, H_q, H_kv, scale, Q, K, V, partial, n_split); break;
        case 8: dense_kernel<TE, D, 8><<<grid, kDenseThreads, 0, st>>>(T, H_q, H_kv, scale, Q, K, V, partial, n_split); break;
        default: return cudaErrorNotSupported;
    }
    return cudaGetLastError();
}

cudaError_t launch_dense(int B, int T, int H_q, int H_kv, int d, int dtype, float scale, const void* q, const void* k,
                         const void* v, float* partial, int n_split, cudaStream_t st) {
    if (B == 0) return cudaSuccess;
    if (dtype == LOWRAM_BF16) {
        if (d == 128) return dense_g<__nv_bfloat16, 128>(B, T, H_q, H_kv, scale, q, k, v, partial, n_split, st);
        if (d == 64) return dense_g<__nv_bfloat16, 64>(B, T, H_q, H_kv, scale, q, k, v, partial, n_split, st);
    } else {
        if (d == 128) return dense_g<float, 128>(B, T, H_q, H_kv, scale, q, k, v, partial, n_split, st);
        if (d == 64) return dense_g<float, 64>(B, T, H_q, H_kv, scale, q, k, v, partial, n_split, st);
    }
    return cudaErrorNotSupported;
}

}  // namespace lowram
