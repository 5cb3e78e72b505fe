// evict.cu -- heavy hitters from accumulated attention, for an evicted cache (the eviction half of composing the
// compressed cache with eviction: "LowRAM Paper: Amortised Values and Low-Rank Keys for KV Compression",
// benchmarks; "LowRAM: predict values from keys, store only the misses", Key points: sinks, recent tokens and heavy
// hitters are kept).
//
// Attention mass of an observation window: W rotated queries per sequence (the prompt's last ones) each attend all
// T prompt tokens; mass[b, t] = sum_i sum_hq softmax_t(scale * q[b, i, hq] . k[b, t, hq / g])[t].
//   1. the log-sum-exp of every (window query, q-head) by the comparator's kernels (dense.cu), the W queries of a
//      sequence read its keys in place (sequence row stride 0);
//   2. mass_kernel: CTAs of 32 tokens; per kv-head the logits of the tile's tokens against the head's W*g window
//      queries come from the register-blocked tile product, exp(logit - lse) is summed over the queries with warp
//      shuffles, and each token's mass is written once.
// Eviction plan: the first n_sink and last n_recent tokens are forced (score +inf), the rest ranked by mass; the
// exact top-T_keep selection (select.cu: ties to the lower index, output ascending) gives the kept tokens.
#include "common.cuh"
#include "kernels.h"
#include "evict.h"
#include "simt_tile.cuh"

namespace lowram {

namespace {

template <typename TA>
__global__ void __launch_bounds__(kTileThreads) mass_kernel(int T, int W, int H_q, int H_kv, int d, float scale,
                                                            const TA* __restrict__ q, const TA* __restrict__ k,
                                                            const float* __restrict__ lse, float* __restrict__ mass) {
    extern __shared__ float sm[];
    float* As = sm;
    float* Bs = As + kTileRows * kStride;
    const int b = blockIdx.y, t0 = blockIdx.x * kTileRows;
    const int g = H_q / H_kv, NQ = W * g;            // window query-heads per kv-head
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
    const TA* kb = k + (int64_t)b * T * H_kv * d;
    const TA* qb = q + (int64_t)b * W * H_q * d;
    const float* lb = lse + (int64_t)b * W * H_q;
    float row_mass[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int h = 0; h < H_kv; ++h) {
        for (int n0 = 0; n0 < NQ; n0 += 128) {
            float acc[4][4];
            zero_acc<4>(acc);
            // acc[u][j] = key(t0 + ty*4 + u) . query(n0 + tx + 32j), query n = (window i = n / g, head h*g + n % g)
            tile_product<4>(
                [&](int t, int kk) { return t0 + t < T ? ld(kb, ((int64_t)(t0 + t) * H_kv + h) * d + kk) : 0.0f; },
                [&](int n, int kk) {
                    const int i = n / g, hq = h * g + (n - i * g);
                    return ld(qb, ((int64_t)i * H_q + hq) * d + kk);
                },
                d, n0, NQ, As, Bs, acc);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float s = 0.0f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int n = n0 + tx + 32 * j;
                    if (n < NQ) {
                        const int i = n / g, hq = h * g + (n - i * g);
                        s += __expf(acc[u][j] * scale - lb[i * H_q + hq]);
                    }
                }
                row_mass[u] += warp_sum(s);
            }
        }
    }
    if (tx == 0)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int t = t0 + ty * 4 + u;
            if (t < T) mass[(int64_t)b * T + t] = row_mass[u];
        }
}

__global__ void evict_scores_kernel(const float* __restrict__ mass, int64_t n, int T, int n_sink, int n_recent,
                                    float* __restrict__ scores) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int t = (int)(i % T);
    scores[i] = (t < n_sink || t >= T - n_recent) ? INFINITY : mass[i];
}

}  // namespace

size_t mass_workspace_bytes(int B, int T, int W, int H_q, int H_kv, int d, int dtype) {
    auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const int ns = dense_records(W, T, H_kv, d, dtype);
    return a(sizeof(float) * (size_t)B * W * H_q) +                      // lse of every window query-head
           a(sizeof(float) * (size_t)W * H_q * ns * (d + 2)) +           // one sequence's split partials
           a(sizeof(float) * (size_t)W * H_q * d);                       // its (unused) attention outputs
}

cudaError_t launch_attention_mass(int B, int T, int W, int H_q, int H_kv, int d, int dtype, float scale,
                                  const void* q_win, const void* k, float* mass, void* scratch, cudaStream_t st) {
    auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
    if ((int64_t)B * T == 0) return cudaSuccess;
    const int ns = dense_splits(W, T, H_kv);
    char* w = (char*)scratch;
    float* lse = (float*)w;
    w += a(sizeof(float) * (size_t)B * W * H_q);
    float* partial = (float*)w;
    w += a(sizeof(float) * (size_t)W * H_q * dense_records(W, T, H_kv, d, dtype) * (d + 2));
    float* out_tmp = (float*)w;
    const size_t eb = dtype == LOWRAM_BF16 ? 2 : 4;
    cudaError_t e;
    for (int b = 0; b < B; ++b) {
        const char* qb = (const char*)q_win + (size_t)b * W * H_q * d * eb;
        const char* kb = (const char*)k + (size_t)b * T * H_kv * d * eb;
        // the W window queries of sequence b as W one-query "sequences" reading the same keys (row stride 0)
        if ((e = launch_dense(W, T, 0, H_q, H_kv, d, dtype, scale, qb, kb, kb, partial, ns, st)) != cudaSuccess)
            return e;
        if ((e = launch_merge(W, H_q, dense_records(W, T, H_kv, d, dtype), d, partial, out_tmp,
                              lse + (size_t)b * W * H_q, st)) != cudaSuccess)
            return e;
    }
    const size_t smem = sizeof(float) * tile_smem_floats(4);
    const dim3 grid((unsigned)cdiv(T, kTileRows), (unsigned)B);
    if (dtype == LOWRAM_BF16)
        mass_kernel<__nv_bfloat16><<<grid, kTileThreads, smem, st>>>(T, W, H_q, H_kv, d, scale,
                                                                     (const __nv_bfloat16*)q_win,
                                                                     (const __nv_bfloat16*)k, lse, mass);
    else
        mass_kernel<float><<<grid, kTileThreads, smem, st>>>(T, W, H_q, H_kv, d, scale, (const float*)q_win,
                                                             (const float*)k, lse, mass);
    return cudaGetLastError();
}

cudaError_t launch_evict_plan(int B, int T, int n_sink, int n_recent, int T_keep, const float* mass, float* scores,
                              int32_t* keep, uint32_t* check, cudaStream_t st) {
    const int64_t n = (int64_t)B * T;
    if (n == 0 || T_keep == 0) return cudaSuccess;
    evict_scores_kernel<<<(unsigned)cdiv(n, 256), 256, 0, st>>>(mass, n, T, n_sink, n_recent, scores);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_select_topn(B, T, T_keep, scores, keep, st, nullptr, nullptr, nullptr, 0, check);
}

}  // namespace lowram
