// tc_decode.cu -- tensor-core (tcgen05) kernels of the decode path for bf16 caches.
//
// K1 score_tc: selection keys of every stored token.  Rebuilding the pre-RoPE keys from the low-rank
// factors ("Asymmetric key compression with xKV", LowRAM Paper: Amortised Values and Low-Rank Keys for
// KV Compression) is a dense [tokens x r] . [r x H_kv*d] product, the dominant cost of a decode call, so
// it runs on the tensor cores; RoPE ("re-applied during attention", same section), the q.k scores of the
// q-heads sharing each kv-head and their maximum (this library's exact-score selection key) are fused
// into the epilogue that reads the accumulators out of TMEM.
//
// Shape of the kernel (persistent, one CTA per SM, 320 threads):
//   warp 0      TMA producer: the 128-token latent tile [128 x r] (r/64 chunks of 16 KB, 128B swizzle,
//               resident for the whole tile) and a ring of basis chunks [256 features x 64] (32 KB each).
//   warp 1      TMEM owner (512 columns) and MMA issuer (one thread): per pair of kv-heads, M=128, N=256,
//               K=r in r/16 tcgen05.mma steps into one of two 256-column accumulators.
//   warps 2-9   epilogue: warp w reads TMEM lane quarter w%4 (32 tokens), head (w-2)/4 of the pair; one
//               thread holds one token's 128 features, applies RoPE from the cos/sin tables, forms the g
//               dot products with q and writes their maximum.  The accumulator is released as soon as it
//               has been read, so the next pair's MMAs overlap the arithmetic.
// Every wait is bounded (see tc_common.cuh); on a timeout the kernel flags LOWRAM_CHECK_TIMEOUT, drains
// the copies and MMAs it issued and returns.
#include <cudaTypedefs.h>

#include "kernels.h"
#include "tc_common.cuh"

namespace lowram {

namespace {

constexpr int kTokTile = 128;
constexpr int kChunkK = 64;                    // bf16 per 128-byte row
constexpr int kAChunkBytes = kTokTile * 128;   // 16 KB
constexpr int kPairN = 256;                    // basis rows per MMA (two heads of 128)
constexpr int kBStageBytes = kPairN * 128;     // 32 KB
constexpr int kScoreThreads = 320;
constexpr int kSmemLimit = 232448;

struct ScoreTcParams {
    int B, T, H_q, H_kv, r, max_pos, tiles_per_seq, n_tiles, KC, NP, NS;
    float scale;
    const __nv_bfloat16* q;
    const int32_t* pos;
    const float* rcos;
    const float* rsin;
    float* key;
    float* sall;        // [B, H_q, T] scaled logits of every q-head, or null
    uint32_t* check;
};

size_t score_smem_bytes(int KC, int NS) {
    return 1024 + (size_t)KC * kAChunkBytes + (size_t)NS * kBStageBytes + 8 * (2 * KC + 2 * NS + 5) + 16;
}

template <int G>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, ScoreTcParams p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* A = smem;
    uint8_t* Bst = A + p.KC * kAChunkBytes;
    uint64_t* a_full = (uint64_t*)(Bst + p.NS * kBStageBytes);
    uint64_t* a_empty = a_full + p.KC;
    uint64_t* b_full = a_empty + p.KC;
    uint64_t* b_empty = b_full + p.NS;
    uint64_t* t_full = b_empty + p.NS;
    uint64_t* t_empty = t_full + 2;
    uint64_t* m_drain = t_empty + 2;
    uint32_t* tmem_slot = (uint32_t*)(m_drain + 1);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.KC; ++i) {
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < p.NS; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&t_full[i], 1);
            mbar_init(&t_empty[i], 8 * 32);
        }
        mbar_init(m_drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t ib = 0;
            int it = 0, a_last = -1;     // iteration of the most recent latent-tile load
            for (int tile = blockIdx.x; tile < p.n_tiles && !*abort_flag; tile += gridDim.x, ++it) {
                const int b = tile / p.tiles_per_seq, t0 = (tile % p.tiles_per_seq) * kTokTile;
                for (int pp = 0; pp < p.NP; ++pp) {
                    for (int kc = 0; kc < p.KC; ++kc) {
                        if (pp == 0) {
                            if (!mbar_wait(&a_empty[kc], (it & 1) ^ 1, abort_flag)) goto produced;
                            mbar_expect_tx(&a_full[kc], kAChunkBytes);
                            tma_load_3d(A + kc * kAChunkBytes, &tmA, &a_full[kc], kc * kChunkK, t0, b);
                            a_last = it;
                        }
                        const uint32_t s = ib % p.NS, ph = (ib / p.NS) & 1;
                        if (!mbar_wait(&b_empty[s], ph ^ 1, abort_flag)) goto produced;
                        mbar_expect_tx(&b_full[s], kBStageBytes);
                        tma_load_2d(Bst + s * kBStageBytes, &tmB, &b_full[s], kc * kChunkK, pp * kPairN);
                        ++ib;
                    }
                }
            }
        produced:
            if (*abort_flag) {
                // drain: every copy issued lands before the CTA exits (chunks of the latest tile were loaded
                // in that tile's iteration, or not at all if the producer stopped before them)
                for (uint32_t k = (ib > (uint32_t)p.NS ? ib - p.NS : 0); k < ib; ++k)
                    mbar_wait_drain(&b_full[k % p.NS], (k / p.NS) & 1);
                if (a_last >= 0)
                    for (int kc = 0; kc < p.KC; ++kc) mbar_wait_drain(&a_full[kc], a_last & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kTokTile, kPairN);
            uint32_t ib = 0, j = 0;
            int it = 0;
            for (int tile = blockIdx.x; tile < p.n_tiles && !*abort_flag; tile += gridDim.x, ++it) {
                for (int pp = 0; pp < p.NP; ++pp, ++j) {
                    const uint32_t buf = j & 1;
                    if (!mbar_wait(&t_empty[buf], ((j >> 1) & 1) ^ 1, abort_flag)) goto issued;
                    fence_after();
                    const uint32_t d_tmem = tmem + buf * kPairN;
                    for (int kc = 0; kc < p.KC; ++kc) {
                        if (pp == 0 && !mbar_wait(&a_full[kc], it & 1, abort_flag)) goto issued;
                        const uint32_t s = ib % p.NS, ph = (ib / p.NS) & 1;
                        if (!mbar_wait(&b_full[s], ph, abort_flag)) goto issued;
                        fence_after();
                        const uint32_t a_addr = smem_u32(A + kc * kAChunkBytes);
                        const uint32_t b_addr = smem_u32(Bst + s * kBStageBytes);
#pragma unroll
                        for (int k = 0; k < kChunkK / 16; ++k)
                            mma_bf16(d_tmem, sdesc_sw128(a_addr + k * 32), sdesc_sw128(b_addr + k * 32), idesc,
                                     (kc | k) != 0);
                        mma_commit(&b_empty[s]);
                        if (pp == p.NP - 1) mma_commit(&a_empty[kc]);
                        ++ib;
                    }
                    mma_commit(&t_full[buf]);
                }
            }
        issued:
            // every MMA this thread issued completes before TMEM is released
            mma_commit(m_drain);
            mbar_wait_drain(m_drain, 0);
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        const int e = warp - 2;
        const int quarter = warp & 3;
        const int half = e >> 2;
        const int row = quarter * 32 + lane;
        uint32_t j = 0;
        for (int tile = blockIdx.x; tile < p.n_tiles && !*abort_flag; tile += gridDim.x) {
            const int b = tile / p.tiles_per_seq, t0 = (tile % p.tiles_per_seq) * kTokTile;
            const int t = t0 + row;
            int ps = 0;
            if (t < p.T) {
                ps = p.pos ? p.pos[(int64_t)b * p.T + t] : t;
                if (ps < 0 || ps >= p.max_pos) {
                    flag(p.check, LOWRAM_CHECK_POS_RANGE);
                    ps = ps < 0 ? 0 : p.max_pos - 1;
                }
            }
            for (int pp = 0; pp < p.NP; ++pp, ++j) {
                const uint32_t buf = j & 1;
                if (!mbar_wait(&t_full[buf], (j >> 1) & 1, abort_flag)) break;
                fence_after();
                const int h = pp * 2 + half;
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + buf * kPairN + half * 128;
                const __nv_bfloat16* qh = p.q + ((int64_t)b * p.H_q + h * G) * 128;   // same for all lanes
                float acc[G];
#pragma unroll
                for (int jq = 0; jq < G; ++jq) acc[jq] = 0.0f;
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    float x[32], y[32];
                    tmem_ld_2x32(taddr + c * 32, taddr + 64 + c * 32, x, y);
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const int i = c * 32 + jj;
                        const float cs = __ldg(p.rcos + (int64_t)i * p.max_pos + ps);
                        const float sn = __ldg(p.rsin + (int64_t)i * p.max_pos + ps);
                        const float kx = x[jj] * cs - y[jj] * sn;
                        const float ky = y[jj] * cs + x[jj] * sn;
#pragma unroll
                        for (int jq = 0; jq < G; ++jq) {
                            acc[jq] = fmaf(__bfloat162float(__ldg(qh + jq * 128 + i)), kx, acc[jq]);
                            acc[jq] = fmaf(__bfloat162float(__ldg(qh + jq * 128 + i + 64)), ky, acc[jq]);
                        }
                    }
                }
                fence_before();
                mbar_arrive(&t_empty[buf]);
                float best = -INFINITY;
#pragma unroll
                for (int jq = 0; jq < G; ++jq) best = fmaxf(best, acc[jq] * p.scale);
                if (t < p.T) {
                    p.key[((int64_t)b * p.H_kv + h) * p.T + t] = best;
                    if (p.sall)
#pragma unroll
                        for (int jq = 0; jq < G; ++jq)
                            p.sall[((int64_t)b * p.H_q + h * G + jq) * p.T + t] = acc[jq] * p.scale;
                }
            }
        }
    }

    // ---------------------------------------------------------------------- teardown
    fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) flag(p.check, LOWRAM_CHECK_TIMEOUT);
    if (warp == 1) {
        fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------------
using tc::encode_fn;
using tc::make_map;
using tc::sm_count;

int stages_for(int KC) {
    for (int ns = 4; ns >= 2; --ns)
        if (score_smem_bytes(KC, ns) <= (size_t)kSmemLimit) return ns;
    return 0;
}

bool g_ok(int g) { return g == 1 || g == 2 || g == 4 || g == 7 || g == 8; }

}  // namespace

bool tc_score_supported(const lowram_decode_shape& s) {
    const int g = s.H_q / s.H_kv;
    return s.act_dtype == LOWRAM_BF16 && s.coef_dtype == LOWRAM_BF16 && s.d == 128 && (s.H_kv * s.d) % kPairN == 0 &&
           s.r % kChunkK == 0 && s.r <= 640 && g_ok(g) && s.T > 0 && stages_for(s.r / kChunkK) >= 2 &&
           encode_fn() != nullptr;
}


cudaError_t launch_score_tc(const DecodeArgs& a, cudaStream_t st) {
    const auto& s = a.s;
    ScoreTcParams p{};
    p.B = s.B;
    p.T = s.T;
    p.H_q = s.H_q;
    p.H_kv = s.H_kv;
    p.r = s.r;
    p.max_pos = s.max_pos;
    p.tiles_per_seq = (int)cdiv(s.T, kTokTile);
    p.n_tiles = p.tiles_per_seq * s.B;
    p.KC = s.r / kChunkK;
    p.NP = s.H_kv * s.d / kPairN;
    p.NS = stages_for(p.KC);
    p.scale = a.scale;
    p.q = (const __nv_bfloat16*)a.q;
    p.pos = a.pos;
    p.rcos = a.rope_cos;
    p.rsin = a.rope_sin;
    p.key = a.key;
    p.sall = a.sall;
    p.check = a.check;
    if (p.n_tiles == 0) return cudaSuccess;
    CUtensorMap mA, mB;
    const uint64_t dA[3] = {(uint64_t)s.r, (uint64_t)s.T, (uint64_t)s.B};
    const uint32_t bA[3] = {kChunkK, kTokTile, 1};
    const uint64_t dB[2] = {(uint64_t)s.r, (uint64_t)s.H_kv * s.d};
    const uint32_t bB[2] = {kChunkK, kPairN};
    if (!make_map(&mA, a.coef, 3, dA, bA) || !make_map(&mB, a.basis, 2, dB, bB)) return cudaErrorInvalidValue;
    const size_t smem = score_smem_bytes(p.KC, p.NS);
    const int grid = std::min(p.n_tiles, sm_count());
    cudaError_t e = cudaSuccess;
    auto go = [&](auto kern) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) {
            kern<<<grid, kScoreThreads, smem, st>>>(mA, mB, p);
            e = cudaGetLastError();
        }
    };
    switch (s.H_q / s.H_kv) {
        case 1: go(score_tc_kernel<1>); break;
        case 2: go(score_tc_kernel<2>); break;
        case 4: go(score_tc_kernel<4>); break;
        case 7: go(score_tc_kernel<7>); break;
        case 8: go(score_tc_kernel<8>); break;
        default: return cudaErrorNotSupported;
    }
    return e;
}

}  // namespace lowram
