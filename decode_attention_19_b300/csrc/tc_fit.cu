// tc_fit.cu -- the two dense products of the basis fit on the tensor cores (tcgen05), in float32 accuracy: the
// Gram matrix of the stacked RoPE-inverted keys and its product with the subspace iterate ("LowRAM Paper:
// Amortised Values and Low-Rank Keys for KV Compression", "Asymmetric key compression with xKV": the G layers'
// keys are stacked and factored together).
//
// A float32 value splits exactly into three bf16 terms, x = h + m + l with h = bf16(x), m = bf16(x - h) and
// l = bf16(x - h - m): each difference is exact in float32 and three 8-bit significands cover float32's 24.  Then
//   x y = h h' + (h m' + m h') + (h l' + m m' + l h') + (m l' + l m' + l l'),
// and the last group is below about 2^-23 |x y|, the size of one float32 rounding; the first six products are
// bf16 MMAs with float32 accumulation.  So C = A B^T over float32 A [M, K] and B [N, K] is one tcgen05
// accumulation chain over six (A term, B term) pairs times K / 64 reduction chunks.
//
// Operands are K-major bf16 terms, zero-padded (rows of A and of B to a multiple of 128, K to 64): the split
// kernel writes them, transposing when the float32 matrix holds the reduction along its rows (the keys
// [tokens, D] for the Gram matrix, the iterate Q [D, r]).  One CTA of 128 threads per 128 x BN output tile (BN = 256,
// or 128 when B's padded rows are not a multiple of 256): thread 0 TMA-loads a 16 KB A chunk and a BN x 128 B
// B chunk per stage into a 4-stage 128-byte-swizzled ring, thread 32 issues four M=128, N=BN, K=16 MMAs per chunk
// into a BN-column TMEM accumulator, and the four warps then read their 32 TMEM lanes and store the tile into C; when
// the tiles alone do not fill the GPU a tile's reduction is split over several CTAs (gridDim.z), which add their
// parts into C (zeroed first) with float32 reductions.  For a symmetric
// product (the Gram matrix, A = B) tiles wholly below the diagonal are skipped and every other tile adds its
// entries on or above the diagonal and their mirrors.  Every wait is bounded: on a timeout the CTA sets
// LOWRAM_CHECK_TIMEOUT, waits for the copies and MMAs it issued, frees TMEM and returns.
#include "kernels.h"
#include "tc_common.cuh"

namespace lowram {

namespace {

constexpr int kGM = 128;                  // output rows per tile (TMEM lanes)
constexpr int kGK = 64;                   // reduction elements per chunk: one 128-byte swizzled row
constexpr int kGStages = 4;
constexpr int kGThreads = 128;
constexpr int kGPairs = 6;
constexpr uint32_t kGABytes = kGM * kGK * 2;    // 16 KB
// BN = output columns per tile (TMEM columns): 256, or 128 when B's rows are not a multiple of 256
__host__ __device__ constexpr uint32_t g_bbytes(int BN) { return (uint32_t)BN * kGK * 2; }
__host__ __device__ constexpr int g_smem(int BN) { return 1024 /* alignment */ + kGStages * (int)(kGABytes + g_bbytes(BN)) + 256; }
// the six products, largest first: pair p multiplies A term (kPairA >> 4p) & 15 by B term (kPairB >> 4p) & 15
// (0 = h, 1 = m, 2 = l): hh, hm, mh, hl, lh, mm
constexpr uint32_t kPairA = 0x120100u, kPairB = 0x102010u;

struct SplitMaps {
    CUtensorMap a[3];   // A's terms [Mp, Kp], box 64 x 128
    CUtensorMap b[3];   // B's terms [Np, Kp], box 64 x BN
};

struct SplitGemmParams {
    int M, N;           // entries of C written: rows < M, columns < N
    int KC;             // reduction chunks of 64 per product
    int ldc;
    int sym;
    int n_split;        // reduction ranges per tile (gridDim.z): 1 stores the tile, more add it with reductions
    int vec4;           // ldc and C allow float4 accesses
    float* C;
    uint32_t* check;
};

template <int BN>
__global__ void __launch_bounds__(kGThreads, 1)
    split_gemm_tc_kernel(const __grid_constant__ SplitMaps maps, SplitGemmParams p) {
    using namespace tc;
    constexpr uint32_t kGBBytes = g_bbytes(BN);
    const int row0 = blockIdx.y * kGM, col0 = blockIdx.x * BN;
    if (p.sym && col0 + BN <= row0) return;           // below the diagonal: the mirror of a computed tile
    const int total = kGPairs * p.KC;
    const int per = (total + p.n_split - 1) / p.n_split;
    const int c_begin = blockIdx.z * per, n_chunks = min(total, c_begin + per) - c_begin;
    if (n_chunks <= 0) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* As = smem;                                // [stage][128 rows x 128 B]
    uint8_t* Bs = As + kGStages * kGABytes;            // [stage][BN rows x 128 B]
    uint64_t* full = (uint64_t*)(Bs + kGStages * kGBBytes);
    uint64_t* empty = full + kGStages;
    uint64_t* done = empty + kGStages;
    uint32_t* tmem_slot = (uint32_t*)(done + 1);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
    int* issued_s = (int*)(abort_flag + 1);            // chunks whose loads thread 0 issued
    int* consumed_s = issued_s + 1;                    // chunks whose loads thread 32 waited for
    if (layout_overflows(smem_raw, (const void*)(consumed_s + 1), p.check)) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        *issued_s = 0;
        *consumed_s = 0;
        fence_barrier_init();
        for (int i = 0; i < 3; ++i) {
            prefetch_tmap(&maps.a[i]);
            prefetch_tmap(&maps.b[i]);
        }
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, BN);
        tmem_relinquish();
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    bool ok = true;
    if (tid == 0) {
        // loads: chunk i of this CTA's range goes to stage i % kGStages once the MMAs of chunk i - kGStages,
        // its previous occupant, have completed
        int i = 0;
        for (; i < n_chunks; ++i) {
            const int s = i % kGStages;
            if (i >= kGStages && !mbar_wait(&empty[s], (uint32_t)((i / kGStages) - 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            const int c = c_begin + i, pr = c / p.KC, kc = c - pr * p.KC;
            const int ia = (int)((kPairA >> (4 * pr)) & 15u), ib = (int)((kPairB >> (4 * pr)) & 15u);
            mbar_expect_tx(&full[s], kGABytes + kGBBytes);
            tma_load_2d(As + s * kGABytes, &maps.a[ia], &full[s], kc * kGK, row0);
            tma_load_2d(Bs + s * kGBBytes, &maps.b[ib], &full[s], kc * kGK, col0);
        }
        *issued_s = i;
    } else if (tid == 32) {
        // MMAs: D [128 x BN] (+)= A chunk [128 x 64] B chunk [BN x 64]^T, four K=16 steps per chunk
        const uint32_t idesc = idesc_bf16(kGM, BN);
        int i = 0;
        for (; i < n_chunks; ++i) {
            const int s = i % kGStages;
            if (!mbar_wait(&full[s], (uint32_t)(i / kGStages) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            fence_after();
            const uint32_t a = smem_u32(As + s * kGABytes), b = smem_u32(Bs + s * kGBBytes);
#pragma unroll
            for (int k = 0; k < kGK / 16; ++k)
                mma_bf16(tmem, sdesc_sw128(a + k * 32), sdesc_sw128(b + k * 32), idesc, (i | k) != 0 ? 1u : 0u);
            mma_commit(&empty[s]);
        }
        *consumed_s = i;
        mma_commit(done);   // arrives once every MMA issued above has completed (at once if there were none)
    }
    const bool aborted = __syncthreads_or(!ok);
    bool acc_ok = false;
    if (!aborted) acc_ok = mbar_wait(done, 0u, abort_flag);
    if (!__syncthreads_and(acc_ok)) {
        if (tid == 0) {
            // loads still in flight land before the shared memory is released; then the MMAs
            for (int i = *consumed_s; i < *issued_s; ++i)
                mbar_wait_drain(&full[i % kGStages], (uint32_t)(i / kGStages) & 1u);
            mbar_wait_drain(done, 0u);
            flag(p.check, LOWRAM_CHECK_TIMEOUT);
        }
    } else {
        fence_after();
        // thread = output row (TMEM lane warp*32 + lane), 64 columns per pass; a tile that owns its outputs
        // (n_split == 1) stores them, else it adds them (float4 where the row allows)
        const int i = row0 + warp * 32 + lane;
        const uint32_t tw = tmem + ((uint32_t)(warp * 32) << 16);
        float* Ci = p.C + (int64_t)i * p.ldc;
        const bool own = p.n_split == 1;
        for (int cb = 0; cb < BN && col0 + cb < p.N; cb += 64) {
            float x[32], y[32];
            tmem_ld_2x32(tw + (uint32_t)cb, tw + (uint32_t)cb + 32u, x, y);
            if (i < p.M) {
#pragma unroll
                for (int u = 0; u < 64; u += 4) {
                    const int j = col0 + cb + u;
                    float v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) v[q] = u + q < 32 ? x[u + q] : y[u + q - 32];
                    if (!p.sym && p.vec4 && j + 3 < p.N) {
                        const float4 v4 = make_float4(v[0], v[1], v[2], v[3]);
                        if (own) *reinterpret_cast<float4*>(Ci + j) = v4;
                        else atomicAdd(reinterpret_cast<float4*>(Ci + j), v4);
                        continue;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int jq = j + q;
                        if (jq < p.N && (!p.sym || jq >= i)) {
                            float* mirror = p.C + (int64_t)jq * p.ldc + i;
                            if (own) {
                                Ci[jq] = v[q];
                                if (p.sym && jq > i) *mirror = v[q];
                            } else {
                                atomicAdd(Ci + jq, v[q]);
                                if (p.sym && jq > i) atomicAdd(mirror, v[q]);
                            }
                        }
                    }
                }
            }
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, BN);
    }
}

__device__ __forceinline__ void split3(float x, __nv_bfloat16& h, __nv_bfloat16& m, __nv_bfloat16& l) {
    h = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(h);          // exact
    m = __float2bfloat16_rn(r1);
    l = __float2bfloat16_rn(r1 - __bfloat162float(m)); // exact, and exactly representable
}

// out_t[orow][ocol] for t = h, m, l (each [out_rows, out_cols] bf16): the terms of src[orow][ocol], or of
// src[ocol][orow] when transposing; zero outside src [R, Cc] (row stride lds).  A CTA of 32 x 8 threads takes a
// 32 x 64 output tile through shared memory (held as t[column][row], so both layouts read the source along its
// rows), and each thread writes two adjacent columns as bf16 pairs.
template <typename TS>
__global__ void __launch_bounds__(256) split3_kernel(const TS* __restrict__ src, int R, int Cc, int64_t lds,
                                                     int transpose, int out_rows, int out_cols,
                                                     __nv_bfloat16* __restrict__ oh, __nv_bfloat16* __restrict__ om,
                                                     __nv_bfloat16* __restrict__ ol) {
    __shared__ float t[64][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    const int64_t ocol0 = (int64_t)blockIdx.x * 64, orow0 = (int64_t)blockIdx.y * 32;
    if (transpose) {
        // source rows ocol0 .. +63, columns orow0 .. +31
        for (int k = ty; k < 64; k += 8) {
            const int64_t sr = ocol0 + k, sc = orow0 + tx;
            t[k][tx] = (sr < R && sc < Cc) ? ld(src, sr * lds + sc) : 0.0f;
        }
    } else {
        // source rows orow0 .. +31, columns ocol0 .. +63
        for (int k = ty; k < 32; k += 8) {
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                const int c = tx + 32 * hlf;
                const int64_t sr = orow0 + k, sc = ocol0 + c;
                t[c][k] = (sr < R && sc < Cc) ? ld(src, sr * lds + sc) : 0.0f;
            }
        }
    }
    __syncthreads();
    const int c0 = 2 * tx;
    const int64_t ocol = ocol0 + c0;
    for (int k = ty; k < 32; k += 8) {
        const int64_t orow = orow0 + k;
        if (orow >= out_rows || ocol >= out_cols) continue;
        __nv_bfloat16 h0, m0, l0, h1, m1, l1;
        split3(t[c0][k], h0, m0, l0);
        const int64_t o = orow * out_cols + ocol;
        if (ocol + 1 < out_cols && (o & 1) == 0) {
            split3(t[c0 + 1][k], h1, m1, l1);
            *reinterpret_cast<__nv_bfloat162*>(oh + o) = __halves2bfloat162(h0, h1);
            *reinterpret_cast<__nv_bfloat162*>(om + o) = __halves2bfloat162(m0, m1);
            *reinterpret_cast<__nv_bfloat162*>(ol + o) = __halves2bfloat162(l0, l1);
        } else {
            oh[o] = h0;
            om[o] = m0;
            ol[o] = l0;
            if (ocol + 1 < out_cols) {
                split3(t[c0 + 1][k], h1, m1, l1);
                oh[o + 1] = h1;
                om[o + 1] = m1;
                ol[o + 1] = l1;
            }
        }
    }
}

}  // namespace

cudaError_t launch_split3(const void* src, bool src_bf16, int R, int Cc, int64_t lds, bool transpose, int out_rows,
                          int out_cols, void* const out[3], cudaStream_t st) {
    if ((int64_t)out_rows * out_cols == 0) return cudaSuccess;
    const dim3 grid((unsigned)cdiv(out_cols, 64), (unsigned)cdiv(out_rows, 32));
    __nv_bfloat16 *h = (__nv_bfloat16*)out[0], *m = (__nv_bfloat16*)out[1], *l = (__nv_bfloat16*)out[2];
    if (src_bf16)
        split3_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)src, R, Cc, lds, transpose ? 1 : 0,
                                                           out_rows, out_cols, h, m, l);
    else
        split3_kernel<float><<<grid, 256, 0, st>>>((const float*)src, R, Cc, lds, transpose ? 1 : 0, out_rows,
                                                   out_cols, h, m, l);
    return cudaGetLastError();
}

cudaError_t launch_split_gemm_tc(const void* const a[3], const void* const b[3], int M, int N, int Mp, int Np, int Kp,
                                 bool sym, float* C, int ldc, uint32_t* check, cudaStream_t st) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (Mp % kGM || Np % 128 || Kp % kGK || Mp < M || Np < N || Kp <= 0) return cudaErrorInvalidValue;
    const int BN = Np % 256 == 0 ? 256 : 128;
    cudaError_t e = cudaSuccess;
    SplitMaps maps;
    const uint64_t dA[2] = {(uint64_t)Kp, (uint64_t)Mp}, dB[2] = {(uint64_t)Kp, (uint64_t)Np};
    const uint32_t bA[2] = {(uint32_t)kGK, (uint32_t)kGM}, bB[2] = {(uint32_t)kGK, (uint32_t)BN};
    for (int t = 0; t < 3; ++t)
        if (!tc::make_map(&maps.a[t], a[t], 2, dA, bA) || !tc::make_map(&maps.b[t], b[t], 2, dB, bB))
            return cudaErrorInvalidValue;
    const int tm = Mp / kGM, tn = Np / BN;
    int tiles = 0;
    for (int bm = 0; bm < tm; ++bm)
        for (int bn = 0; bn < tn; ++bn) tiles += (!sym || bn * BN + BN > bm * kGM) ? 1 : 0;
    SplitGemmParams p;
    p.M = M;
    p.N = N;
    p.KC = Kp / kGK;
    p.ldc = ldc;
    p.sym = sym ? 1 : 0;
    p.C = C;
    p.check = check;
    // split the reduction while the tiles do not fill the GPU and each range keeps 4 chunks or more
    const int sms = tc::sm_count(), total = kGPairs * p.KC;
    int n_split = 1;
    while ((int64_t)tiles * n_split * 2 <= sms && total / (n_split * 2) >= 4) n_split *= 2;
    p.n_split = n_split;
    p.vec4 = (ldc % 4 == 0 && ((uintptr_t)C & 15u) == 0) ? 1 : 0;
    if (n_split > 1 && (e = cudaMemsetAsync(C, 0, sizeof(float) * (size_t)M * ldc, st)) != cudaSuccess) return e;
    const dim3 grid((unsigned)tn, (unsigned)tm, (unsigned)n_split);
    if (BN == 256) {
        e = cudaFuncSetAttribute(split_gemm_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, g_smem(256));
        if (e == cudaSuccess) split_gemm_tc_kernel<256><<<grid, kGThreads, g_smem(256), st>>>(maps, p);
    } else {
        e = cudaFuncSetAttribute(split_gemm_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, g_smem(128));
        if (e == cudaSuccess) split_gemm_tc_kernel<128><<<grid, kGThreads, g_smem(128), st>>>(maps, p);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace lowram
