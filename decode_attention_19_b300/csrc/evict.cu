// evict.cu -- heavy hitters from accumulated attention, for an evicted cache (the eviction half of composing the
// compressed cache with eviction: "LowRAM Paper: Amortised Values and Low-Rank Keys for KV Compression",
// benchmarks; "LowRAM: predict values from keys, store only the misses", Key points: sinks, recent tokens and heavy
// hitters are kept).
//
// Attention mass of an observation window: W rotated queries per sequence (the prompt's last ones) each attend all
// T prompt tokens; mass[b, t] = sum_i sum_hq softmax_t(scale * q[b, i, hq] . k[b, t, hq / g])[t].  Two passes over
// the logits, the first for the log-sum-exp of every (window query, q-head), the second for the mass.  bf16 prompts
// run both on the tensor cores (tc_evict.cu); float32 prompts on CUDA cores here:
//   1. lse_partial_kernel: CTAs of a few 32-token tiles; per kv-head the logits of each tile's tokens against the
//      head's W*g window queries come from the register-blocked tile product (each key row is read once for all
//      of them), and every query's (max, sum of exp) over the CTA's tokens is written out; lse_reduce_kernel folds
//      the CTAs' pairs into the log-sum-exp of every (window query, q-head);
//   2. mass_kernel: CTAs of 32 tokens; the same logits again, exp(logit - lse) summed over the queries with warp
//      shuffles, and each token's mass written once.
// lse_reduce_kernel serves both paths (the chunks' pairs share one layout).
// Eviction plan: the first n_sink and last n_recent tokens are forced (score +inf), the rest ranked by mass; the
// exact top-T_keep selection (select.cu: ties to the lower index, output ascending) gives the kept tokens.
#include "common.cuh"
#include "kernels.h"
#include "evict.h"
#include "simt_tile.cuh"

#include <algorithm>

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

// Fold a (max, sum of exp(x - max)) pair into a running one; (-inf, 0) is the empty set.
__device__ __forceinline__ void lse_fold(float& m, float& s, float2 p) {
    const float M = fmaxf(m, p.x);
    if (M == -INFINITY) return;
    s = (m == -INFINITY ? 0.0f : s * __expf(m - M)) + (p.x == -INFINITY ? 0.0f : p.y * __expf(p.x - M));
    m = M;
}

// part[b][c][i*H_q + hq] = (max, sum of exp(logit - max)) of window query i, q-head hq over the tokens of tiles
// [c*chunk_tiles, (c+1)*chunk_tiles).  Per kv-head and group of 128 window query-heads, thread tid < 128 keeps
// the running pair of query n0 + tid; each tile is reduced over its 32 tokens (4 per thread, then the 8 warps
// through shared memory) before it is folded in.
template <typename TA>
__global__ void __launch_bounds__(kTileThreads) lse_partial_kernel(int T, int W, int H_q, int H_kv, int d,
                                                                   float scale, int chunk_tiles,
                                                                   const TA* __restrict__ q, const TA* __restrict__ k,
                                                                   float2* __restrict__ part) {
    extern __shared__ float sm[];
    float* As = sm;
    float* Bs = As + kTileRows * kStride;
    float2* red = reinterpret_cast<float2*>(Bs + 4 * 32 * kStride);      // [8 warps][128 queries]
    const int b = blockIdx.y, c = blockIdx.x;
    const int g = H_q / H_kv, NQ = W * g;
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
    const int tile_begin = c * chunk_tiles;
    const int tile_end = (int)min((int64_t)cdiv(T, kTileRows), (int64_t)tile_begin + chunk_tiles);
    const TA* kb = k + (int64_t)b * T * H_kv * d;
    const TA* qb = q + (int64_t)b * W * H_q * d;
    float2* pb = part + ((int64_t)b * gridDim.x + c) * ((int64_t)W * H_q);
    for (int h = 0; h < H_kv; ++h) {
        for (int n0 = 0; n0 < NQ; n0 += 128) {
            float run_m = -INFINITY, run_s = 0.0f;
            for (int tile = tile_begin; tile < tile_end; ++tile) {
                const int t0 = tile * kTileRows;
                float acc[4][4];
                zero_acc<4>(acc);
                tile_product<4>(
                    [&](int t, int kk) { return t0 + t < T ? ld(kb, ((int64_t)(t0 + t) * H_kv + h) * d + kk) : 0.0f; },
                    [&](int n, int kk) {
                        const int i = n / g, hq = h * g + (n - i * g);
                        return ld(qb, ((int64_t)i * H_q + hq) * d + kk);
                    },
                    d, n0, NQ, As, Bs, acc);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float m = -INFINITY, s = 0.0f;
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (t0 + ty * 4 + u < T) m = fmaxf(m, acc[u][j] * scale);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (t0 + ty * 4 + u < T) s += __expf(acc[u][j] * scale - m);
                    red[ty * 128 + tx + 32 * j] = make_float2(m, s);
                }
                __syncthreads();
                if (tid < 128)
#pragma unroll
                    for (int v = 0; v < 8; ++v) lse_fold(run_m, run_s, red[v * 128 + tid]);
                __syncthreads();
            }
            if (tid < 128 && n0 + tid < NQ) {
                const int n = n0 + tid, i = n / g, hq = h * g + (n - i * g);
                pb[i * H_q + hq] = make_float2(run_m, run_s);
            }
        }
    }
}

// lse[b][qi] for the NQall = W*H_q window query-heads of each sequence: a CTA of 8 warps per (b, 32 consecutive
// query-heads); warp w folds chunks w, w + 8, ..., then warp 0 folds the 8 pairs.  Every chunk holds at least one
// token, so the final maximum is finite and the sum at least 1.
__global__ void __launch_bounds__(256) lse_reduce_kernel(int n_chunks, int NQall, const float2* __restrict__ part,
                                                         float* __restrict__ lse) {
    __shared__ float2 red[8][32];
    const int b = blockIdx.y, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int qi = blockIdx.x * 32 + lane;
    float m = -INFINITY, s = 0.0f;
    if (qi < NQall) {
        const float2* pb = part + (int64_t)b * n_chunks * NQall + qi;
#pragma unroll 4
        for (int c = w; c < n_chunks; c += 8) lse_fold(m, s, pb[(int64_t)c * NQall]);
    }
    red[w][lane] = make_float2(m, s);
    __syncthreads();
    if (w == 0 && qi < NQall) {
#pragma unroll
        for (int v = 1; v < 8; ++v) lse_fold(m, s, red[v][lane]);
        lse[(int64_t)b * NQall + qi] = m + logf(s);
    }
}

// Tiles per lse_partial_kernel CTA: about 16 CTAs per SM over the whole grid, at least one tile each.
int lse_chunk_tiles(int B, int T) {
    const int64_t tiles = (int64_t)B * cdiv(T, kTileRows);
    return (int)std::max<int64_t>(1, tiles / (16 * 148));
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
    const size_t lse_bytes = a(sizeof(float) * (size_t)B * W * H_q);
    if (dtype == LOWRAM_BF16)
        return lse_bytes + a(sizeof(float2) * (size_t)B * window_tc_n_chunks(B, T) * W * H_q) +
               a((size_t)2 * B * H_kv * window_tc_qpad(W, H_q, H_kv) * d);    // the packed window queries
    const int ct = lse_chunk_tiles(B, T);
    const size_t n_chunks = T > 0 ? (size_t)cdiv(cdiv(T, kTileRows), ct) : 0;
    return lse_bytes + a(sizeof(float2) * (size_t)B * n_chunks * W * H_q);   // the chunks' (max, sum) pairs
}

cudaError_t launch_attention_mass(int B, int T, int W, int H_q, int H_kv, int d, int dtype, float scale,
                                  const void* q_win, const void* k, float* mass, void* scratch, uint32_t* check,
                                  cudaStream_t st) {
    auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
    if ((int64_t)B * T == 0) return cudaSuccess;
    float* lse = (float*)scratch;
    float2* part = (float2*)((char*)scratch + a(sizeof(float) * (size_t)B * W * H_q));
    const int NQall = W * H_q;
    const dim3 reduce_grid((unsigned)cdiv(NQall, 32), (unsigned)B);
    cudaError_t e;
    if (dtype == LOWRAM_BF16) {
        // tensor cores: pack the window queries, log-sum-exp pass, fold the chunks, mass pass
        const int n_chunks = window_tc_n_chunks(B, T);
        void* qp = (char*)part + a(sizeof(float2) * (size_t)B * n_chunks * NQall);
        if ((e = launch_pack_window(B, W, H_q, H_kv, d, q_win, qp, st)) != cudaSuccess) return e;
        if ((e = launch_window_tc(false, B, T, W, H_q, H_kv, d, scale, qp, k, part, nullptr, nullptr, check, st)) !=
            cudaSuccess)
            return e;
        lse_reduce_kernel<<<reduce_grid, 256, 0, st>>>(n_chunks, NQall, part, lse);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        return launch_window_tc(true, B, T, W, H_q, H_kv, d, scale, qp, k, nullptr, lse, mass, check, st);
    }
    // float32 prompts: the fp32 tile product on CUDA cores
    const int ct = lse_chunk_tiles(B, T);
    const int n_chunks = cdiv(cdiv(T, kTileRows), ct);
    const size_t lse_smem = sizeof(float) * (tile_smem_floats(4) + 2 * 8 * 128);
    lse_partial_kernel<float><<<dim3((unsigned)n_chunks, (unsigned)B), kTileThreads, lse_smem, st>>>(
        T, W, H_q, H_kv, d, scale, ct, (const float*)q_win, (const float*)k, part);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    lse_reduce_kernel<<<reduce_grid, 256, 0, st>>>(n_chunks, NQall, part, lse);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smem = sizeof(float) * tile_smem_floats(4);
    mass_kernel<float><<<dim3((unsigned)cdiv(T, kTileRows), (unsigned)B), kTileThreads, smem, st>>>(
        T, W, H_q, H_kv, d, scale, (const float*)q_win, (const float*)k, lse, mass);
    return cudaGetLastError();
}

cudaError_t launch_evict_plan(int B, int T, int n_sink, int n_recent, int T_keep, const float* mass, float* scores,
                              int32_t* keep, uint32_t* check, cudaStream_t st) {
    const int64_t n = (int64_t)B * T;
    if (n == 0 || T_keep == 0) return cudaSuccess;
    evict_scores_kernel<<<(unsigned)cdiv(n, 256), 256, 0, st>>>(mass, n, T, n_sink, n_recent, scores);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_select_topn(B, T, T_keep, scores, keep, st, nullptr, nullptr, 0, check);
}

}  // namespace lowram
