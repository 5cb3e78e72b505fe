// simt_tile.cuh -- a 32-row register-blocked fp32 tile product on CUDA cores.
//
//   acc[u][j] += sum_k A(row = ty*4 + u, k) * B(col = n0 + tx + 32*j, k)
//
// with 256 threads (ty = tid / 32, tx = tid % 32), 32 rows per tile and up to NJ*32 columns.  A and B
// are read through functors (global loads with dtype decoding, or shared memory), staged 32 k-values
// at a time in shared memory (row stride 33 floats, so column reads by the 32 lanes hit 32 banks).
// Used where fp32 accuracy is required (the write side's error ranking, float32 caches) and by the
// float32 decode path.  Columns >= N and k >= K read as zero.
#pragma once

#include "common.cuh"

namespace lowram {

constexpr int kTileRows = 32;
constexpr int kTileThreads = 256;
constexpr int kKC = 32;       // k-values staged per round
constexpr int kStride = kKC + 1;

// Shared-memory floats the staging buffers need for NJ column groups.
__host__ __device__ constexpr int tile_smem_floats(int NJ) { return kTileRows * kStride + NJ * 32 * kStride; }

template <int NJ, typename AF, typename BF>
__device__ __forceinline__ void tile_product(AF A, BF Bm, int K, int n0, int N, float* As, float* Bs,
                                             float (&acc)[4][NJ]) {
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
    for (int k0 = 0; k0 < K; k0 += kKC) {
        for (int e = tid; e < kTileRows * kKC; e += kTileThreads) {
            int t = e >> 5, k = e & 31;
            As[t * kStride + k] = (k0 + k < K) ? A(t, k0 + k) : 0.0f;
        }
        for (int e = tid; e < NJ * 32 * kKC; e += kTileThreads) {
            int n = e >> 5, k = e & 31;
            Bs[n * kStride + k] = (n0 + n < N && k0 + k < K) ? Bm(n0 + n, k0 + k) : 0.0f;
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < kKC; ++k) {
            float av[4], bv[NJ];
#pragma unroll
            for (int u = 0; u < 4; ++u) av[u] = As[(ty * 4 + u) * kStride + k];
#pragma unroll
            for (int j = 0; j < NJ; ++j) bv[j] = Bs[(tx + 32 * j) * kStride + k];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int j = 0; j < NJ; ++j) acc[u][j] = fmaf(av[u], bv[j], acc[u][j]);
        }
        __syncthreads();
    }
}

template <int NJ>
__device__ __forceinline__ void zero_acc(float (&acc)[4][NJ]) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < NJ; ++j) acc[u][j] = 0.0f;
}

// Write acc into a [32][ld] shared tile (columns n0 + tx + 32j < N), optionally adding a bias and
// applying SiLU (accurate expf when Accurate, else the fast exponential).
template <int NJ, bool Silu, bool Accurate>
__device__ __forceinline__ void store_tile(const float (&acc)[4][NJ], float* dst, int ld, int n0, int N,
                                           const float* bias) {
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        int n = n0 + tx + 32 * j;
        if (n >= N) continue;
        float bb = bias ? bias[n] : 0.0f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float x = acc[u][j] + bb;
            if (Silu) x = Accurate ? x / (1.0f + expf(-x)) : x / (1.0f + __expf(-x));
            dst[(ty * 4 + u) * ld + n] = x;
        }
    }
}

}  // namespace lowram
