// tc_decode.cu -- tensor-core (tcgen05) key pass of the decode path for bf16 caches (K1).
//
// Selection keys of every stored token.  Rebuilding the pre-RoPE keys from the low-rank factors
// ("Asymmetric key compression with xKV", LowRAM Paper: Amortised Values and Low-Rank Keys for KV
// Compression) is a dense [tokens x r] . [r x H_kv*d] product, the dominant cost of a decode call, so it
// runs on the tensor cores; RoPE ("re-applied during attention", same section), the q.k scores of the
// q-heads sharing each kv-head and their maximum (this library's exact-score selection key) are fused into
// the epilogue that reads the accumulators out of TMEM.  Every q-head's scaled logit is stored too: the
// value pass takes the softmax of the selected tokens from exactly the scores the selection saw.
//
// Shape of the kernel: persistent CTA pairs (clusters of two, at most one CTA per SM), 320 threads per CTA.
// The work items are (tile pair, unit) in that order; a pair of CTAs walks a contiguous range of items, so the
// ranges differ by at most one unit (rather than by a whole tile pair of NU units), and CTA r of the pair takes
// tile 2*pair + r.  The key rebuild of a unit of UN/128 kv-heads is one pair MMA per k-step (tcgen05 cta_group::2, M=256, N=UN, K=16): each
// CTA supplies its tile's 128 token rows of A and half of the unit's basis rows of B, and each CTA's TMEM
// accumulates its own 128 tokens x UN features.  Compared with one CTA per tile, every SM reads only half
// of each basis chunk from shared memory.
//   warp 0      TMA producer (both CTAs): a ring of NS stages, each one 64-wide k-chunk of the CTA's
//               latent tile [128 x 64] and of its half of the unit's basis rows [UN/2 x 64].  The odd CTA's
//               copies complete on the even CTA's barrier, so one barrier covers the pair's stage.
//   warp 1      TMEM owner (both CTAs allocate the pair's 2*UN columns together) and, in the even CTA, the
//               MMA issuer; each stage's commit releases the stage in both CTAs.
//   warps 2-9   epilogue, all eight warps on every unit: warp w reads TMEM lane quarter w%4 and one half of
//               the 64 rotary frequencies in the 16x256b shape, so a thread holds four tokens and eight
//               frequencies.  It fetches their cos/sin once per tile into registers and per unit rotates the
//               unit's heads and accumulates the dot products with the queries (bf16 pairs in shared memory,
//               each loaded value serving the thread's four tokens; the softmax scale multiplies the finished
//               dot products) in packed fp32 pairs.  Shuffles sum over the four lanes that share a token; the
//               upper frequency half passes its partial sums to the lower half through shared memory.  Both
//               CTAs' epilogues release a TMEM buffer (double-buffered by unit) before the even CTA's MMAs
//               reuse it.
// Every wait is bounded (see tc_common.cuh); a failed wait stops both CTAs of the pair, which flag
// LOWRAM_CHECK_TIMEOUT, let what they issued complete and return.  The epilogue's named barriers are reached
// on every path, and the pair meets at a cluster barrier before either frees TMEM or exits.
#include <cudaTypedefs.h>

#include "kernels.h"
#include "tc_common.cuh"

namespace lowram {

namespace {

constexpr int kTokTile = 128;
constexpr int kChunkK = 64;                    // bf16 per 128-byte row
constexpr int kAChunkBytes = kTokTile * 128;   // 16 KB
constexpr int kScoreThreads = 320;
constexpr int kSmemLimit = 232448;

struct ScoreTcParams {
    int B, T, H_q, H_kv, r, max_pos, tiles_per_seq, n_tiles, KC, NU, NS;
    int pps;            // tile pairs per sequence when every sequence has its own basis (pairs stay within a
                        // sequence, whose basis both CTAs load), else 0 (pairs run over the whole batch)
    uint32_t idesc;     // MMA instruction descriptor: bf16 operands, or fp16 (an int4 cache's fp16 copy)
    float scale;
    const __nv_bfloat16* q;
    const int32_t* pos;
    const float* rcos;
    const float* rsin;
    float* key;
    float* sall;        // [B, T, H_q] scaled logits of every q-head (a token's q-heads contiguous), or null
    uint32_t* check;
};

// Stage s of the ring: one 64-wide k-chunk of the latent tile [128 x 64] and of the unit's basis rows
// [UN x 64], both 128B-swizzled as TMA writes them.
// Beside the ring: the queries of the current sequence (bf16 as given, grouped by frequency pair) and,
// double-buffered by unit, the exchange of partial dot products between the frequency halves [2][128][16] fp32.
size_t score_smem_bytes(int NS, int UN, int H_q) {
    return 1024 + (size_t)NS * (kAChunkBytes + (UN / 2) * 128) + (size_t)H_q * 128 * 2 + 2 * 128 * 16 * 4 +
           8 * (2 * NS + 5) + 16;
}

// Tile of CTA `rank` in tile pair `pr`: its sequence b, first token t0, and whether it is real (a tile past the end
// is computed on the last tile's data and not written).
__device__ __forceinline__ void pair_tile(const ScoreTcParams& p, int pr, int rank, int& b, int& t0, bool& real) {
    if (p.pps) {
        b = pr / p.pps;
        const int lt = 2 * (pr - b * p.pps) + rank;
        real = lt < p.tiles_per_seq;
        t0 = min(lt, p.tiles_per_seq - 1) * kTokTile;
    } else {
        const int tile = 2 * pr + rank;
        real = tile < p.n_tiles;
        const int lt = real ? tile : p.n_tiles - 1;
        b = lt / p.tiles_per_seq;
        t0 = (lt % p.tiles_per_seq) * kTokTile;
    }
}

template <int G, int HPU>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kScoreThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, ScoreTcParams p) {
    using namespace tc;
    constexpr int UN = HPU * 128;              // accumulator columns per unit = basis rows per pair MMA
    constexpr int kBHalf = (UN / 2) * 128;     // this CTA's half of a basis chunk [UN/2 x 64]
    constexpr int kStage = kAChunkBytes + kBHalf;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* St = smem;
    uint2* Qs = (uint2*)(St + p.NS * kStage);     // [H_q][32] query of the current sequence, bf16, by frequency pair
    float* Xs = (float*)(Qs + p.H_q * 32);         // [2][128 rows][16] partial dots of the upper frequencies
    uint64_t* b_full = (uint64_t*)(Xs + 2 * 128 * 16);   // (even CTA) both CTAs' copies of the stage landed
    uint64_t* b_empty = b_full + p.NS;                   // the pair's MMAs are done with the stage
    uint64_t* t_full = b_empty + p.NS;
    uint64_t* t_empty = t_full + 2;                      // (even CTA) both epilogues released the buffer
    uint64_t* m_drain = t_empty + 2;
    uint32_t* tmem_slot = (uint32_t*)(m_drain + 1);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
    if (layout_overflows(smem_raw, (const void*)(abort_flag + 1), p.check)) return;   // both CTAs of the pair alike

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();          // 0 issues the MMAs; 1 feeds its halves
    grid_dep_trigger();  // the selection kernel may be scheduled as SMs free up; it waits for this grid
    const uint32_t peer = rank ^ 1u;
    // the pair walks a contiguous range of (tile pair, unit) items; CTA `rank` takes tile 2*pair + rank (a tile
    // past the end is computed on the last tile's data and not written)
    const int n_pairs = p.pps ? p.B * p.pps : (p.n_tiles + 1) / 2;
    const int n_items = n_pairs * p.NU, cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    const int it_begin = (int)((int64_t)cl * n_items / ncl), it_end = (int)((int64_t)(cl + 1) * n_items / ncl);
    // work item -> (tile pair pr, unit u)
    auto item_up = [&](int it, int& u, int& pr) {
        pr = it / p.NU;
        u = it - pr * p.NU;
    };
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.NS; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&t_full[i], 1);
            mbar_init(&t_empty[i], 8 * 32 + 8);   // 256 local threads + one arrival per warp of the odd CTA
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
        tmem_alloc_pair(tmem_slot, 2 * UN);
        tmem_relinquish_pair();
    }
    fence_before();
    __syncthreads();
    cluster_sync();      // both CTAs' barriers exist and TMEM is allocated before any cross-CTA traffic
    fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t peer_abort = peer_smem((const void*)abort_flag, peer);
    // a failed wait stops both CTAs of the pair
    auto fail = [&]() {
        *abort_flag = 1;
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1) : "memory");
    };

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            uint32_t ib = 0;           // ring stages issued
            uint32_t s = 0, ph = 0;    // ring position of stage ib, kept incrementally (see the MMA issuer)
            for (int it = it_begin; it < it_end && !*abort_flag; ++it) {
                int u, pr;
                item_up(it, u, pr);
                int b, t0;
                bool real_t;
                pair_tile(p, pr, (int)rank, b, t0, real_t);
                (void)real_t;   // a tile past the end is loaded like the last one
                const int brow = u * UN + (int)rank * (UN / 2);
                {
                    for (int kc = 0; kc < p.KC; ++kc, ++ib) {
                        if (!mbar_wait_cluster(&b_empty[s], ph ^ 1, abort_flag)) {
                            fail();
                            goto produced;
                        }
                        uint8_t* dA = St + s * kStage;
                        uint8_t* dB = dA + kAChunkBytes;
                        if (rank == 0) {   // the even CTA's barrier counts both CTAs' bytes
                            mbar_expect_tx(&b_full[s], 2 * kStage);
                            tma_load_3d(dA, &tmA, &b_full[s], kc * kChunkK, t0, b);
                            if (p.pps) tma_load_3d(dB, &tmB, &b_full[s], kc * kChunkK, brow, b);
                            else tma_load_2d(dB, &tmB, &b_full[s], kc * kChunkK, brow);
                        } else {
                            const uint32_t bar = peer_smem(&b_full[s], 0);
                            tma_load_3d_pair(dA, &tmA, bar, kc * kChunkK, t0, b);
                            if (p.pps) tma_load_3d_pair(dB, &tmB, bar, kc * kChunkK, brow, b);
                            else tma_load_2d_pair(dB, &tmB, bar, kc * kChunkK, brow);
                        }
                        if (++s == (uint32_t)p.NS) {
                            s = 0;
                            ph ^= 1;
                        }
                    }
                }
            }
        produced:
            if (*abort_flag) {
                if (rank == 0) {   // stages older than the last NS were consumed by MMAs, so they have landed
                    for (uint32_t k = (ib > (uint32_t)p.NS ? ib - p.NS : 0); k < ib; ++k)
                        mbar_wait_drain(&b_full[k % p.NS], (k / p.NS) & 1);
                } else {           // this CTA's copies complete on the even CTA's barriers: give them time to land
                    const long long c0 = clock64();
                    while (clock64() - c0 < 4000000) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (rank == 0 && lane == 0) {
            // -------------------------------------------------------------- MMA issuer (even CTA)
            // One thread feeds the tensor pipe (a 256x256x16 pair MMA every 128 SM cycles at full rate), so the
            // loop keeps the ring position incrementally and rebuilds no descriptor: a stage adds its byte offset
            // >> 4 to the descriptor of stage 0, a 16-wide k-step 32 bytes (2 units).
            const uint32_t idesc = p.idesc;
            const uint64_t st_desc = sdesc_sw128(smem_u32(St));
            uint32_t s = 0, ph = 0, j = 0;
            for (int it = it_begin; it < it_end && !*abort_flag; ++it, ++j) {
                {
                    const uint32_t buf = j & 1;
                    if (!mbar_wait_cluster(&t_empty[buf], ((j >> 1) & 1) ^ 1, abort_flag)) {
                        fail();
                        goto issued;
                    }
                    fence_after();
                    const uint32_t d_tmem = tmem + buf * UN;
                    for (int kc = 0; kc < p.KC; ++kc) {
                        if (!mbar_wait(&b_full[s], ph, abort_flag)) {
                            fail();
                            goto issued;
                        }
                        fence_after();
                        const uint64_t ad = st_desc + s * (uint32_t)(kStage >> 4), bd = ad + (kAChunkBytes >> 4);
#pragma unroll
                        for (int k = 0; k < kChunkK / 16; ++k)
                            mma_bf16_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (kc | k) != 0);
                        mma_commit_pair(&b_empty[s], 0x3);
                        if (++s == (uint32_t)p.NS) {
                            s = 0;
                            ph ^= 1;
                        }
                    }
                    mma_commit_pair(&t_full[buf], 0x3);
                }
            }
        issued:
            // every MMA issued completes before TMEM is released
            mma_commit_pair(m_drain, 0x1);
            mbar_wait_drain(m_drain, 0);
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        // all eight warps work on every unit: warp w reads TMEM lane quarter w%4 and takes frequency half `fh`.
        // TMEM is read in the 16x256b shape, so a thread holds four tokens (rows quarter*32 + 16*lh + 8*i + r8,
        // lh, i in {0, 1}) and eight frequencies (fh*32 + 8c + 2*g4 + e, c in 0..3, e in {0, 1}); every query
        // value it loads from shared memory serves LHP*2 tokens.  The partial dot products are summed over the four
        // lanes that share a token (g4) with shuffles, and the two frequency halves meet through shared memory.
        constexpr int LHP = (G <= 4) ? 2 : 1;     // lane halves (token pairs) per pass over the accumulator
        constexpr int R = 2 * LHP;                // tokens per pass
        const int et = threadIdx.x - 64;
        const int fh = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int g4 = lane & 3, r8 = lane >> 2, b0 = lane & 1, b1 = (lane >> 1) & 1;
        const int64_t mp = p.max_pos;
        // the token this thread finishes (adds the other half's partial sums, takes the maximum and stores):
        // LHP == 2: the lower frequency half finishes all rows, one per lane;
        // LHP == 1: the frequency half fh finishes the rows of lane half lh == fh (lanes with b1 == 0)
        const int frow = (LHP == 2) ? quarter * 32 + 16 * b0 + 8 * b1 + r8 : quarter * 32 + 16 * fh + 8 * b0 + r8;
        const bool finisher = (LHP == 2) ? (fh == 0) : (b1 == 0);
        uint32_t j = 0;
        int cur_b = -1, cur_pr = -1;
        int b = 0, t0 = 0;
        bool real = false;
        // cos/sin of this thread's frequencies (f, f+1), f = fh*32 + 8c + 2*g4, at each of its four tokens'
        // positions ([2*lh + i][c]); fetched once per tile and kept in registers for every unit of the tile
        uint64_t c2[4][4], s2[4][4];
        // positions are the token indices (no position array): the tables are read at the thread's first token
        // only and its other three tokens, 8, 16 and 24 positions on, come from rotations by 8 positions
        // (the angle-addition formula with the tables at position 8; three fp32 steps, ~1e-7 relative)
        const bool rot = p.pos == nullptr && p.max_pos >= p.T && p.max_pos > 8;
        auto load_tables = [&](int bb, int tt0, bool rl) {
            if (rot) {
                const int t = tt0 + quarter * 32 + r8;
                const int ps = (rl && t < p.T) ? t : 0;
                const float* cb = p.rcos + (int64_t)(fh * 32 + 2 * g4) * mp;
                const float* sb = p.rsin + (int64_t)(fh * 32 + 2 * g4) * mp;
                uint64_t c8[4], s8[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    c2[0][c] = f2_pack(__ldg(cb + (8 * c) * mp + ps), __ldg(cb + (8 * c + 1) * mp + ps));
                    s2[0][c] = f2_pack(__ldg(sb + (8 * c) * mp + ps), __ldg(sb + (8 * c + 1) * mp + ps));
                    c8[c] = f2_pack(__ldg(cb + (8 * c) * mp + 8), __ldg(cb + (8 * c + 1) * mp + 8));
                    s8[c] = f2_pack(__ldg(sb + (8 * c) * mp + 8), __ldg(sb + (8 * c + 1) * mp + 8));
                }
#pragma unroll
                for (int k = 1; k < 4; ++k)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        c2[k][c] = f2_sub(f2_mul(c2[k - 1][c], c8[c]), f2_mul(s2[k - 1][c], s8[c]));
                        s2[k][c] = f2_fma(s2[k - 1][c], c8[c], f2_mul(c2[k - 1][c], s8[c]));
                    }
                return;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int t = tt0 + quarter * 32 + 16 * (k >> 1) + 8 * (k & 1) + r8;
                int ps = 0;
                if (rl && t < p.T) {
                    ps = p.pos ? p.pos[(int64_t)bb * p.T + t] : t;
                    if (ps < 0 || ps >= p.max_pos) {
                        flag(p.check, LOWRAM_CHECK_POS_RANGE);
                        ps = ps < 0 ? 0 : p.max_pos - 1;
                    }
                }
                const float* cb = p.rcos + (int64_t)(fh * 32 + 2 * g4) * mp + ps;
                const float* sb = p.rsin + (int64_t)(fh * 32 + 2 * g4) * mp + ps;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    c2[k][c] = f2_pack(__ldg(cb + (8 * c) * mp), __ldg(cb + (8 * c + 1) * mp));
                    s2[k][c] = f2_pack(__ldg(sb + (8 * c) * mp), __ldg(sb + (8 * c + 1) * mp));
                }
            }
        };
        // no abort test in the loop conditions: every epilogue thread walks the same items and reaches the
        // same named barriers; after an abort the waits fail at once and the work is skipped
        for (int it = it_begin; it < it_end; ++it, ++j) {
            int u, pr;
            item_up(it, u, pr);
            if (pr != cur_pr) {   // a new tile not fetched at the end of the item before
                cur_pr = pr;
                pair_tile(p, pr, (int)rank, b, t0, real);   // a tile past the end is computed but writes nothing
                if (b != cur_b) {
                    named_bar_sync(1, 256);      // every epilogue thread is done with the previous query
                    if (!*abort_flag) {
                        // Qs[q-head][frequency pair fp] = (q[2fp], q[2fp+1]), (q[64+2fp], q[64+2fp+1]) as bf16 pairs
                        // (the softmax scale is applied to the finished dot products);
                        // one item = a q-head's dims 8a..8a+7 and 64+8a..64+8a+7 (two 16-byte loads); H_q*8 items,
                        // one per thread for up to 32 q-heads
                        const uint4* qb = reinterpret_cast<const uint4*>(p.q + (int64_t)b * p.H_q * 128);
                        for (int e = et; e < p.H_q * 8; e += 256) {
                            const uint4 vx = qb[(e >> 3) * 16 + (e & 7)];
                            const uint4 vy = qb[(e >> 3) * 16 + 8 + (e & 7)];
                            uint2* dst = Qs + (e >> 3) * 32 + (e & 7) * 4;
                            dst[0] = make_uint2(vx.x, vy.x);
                            dst[1] = make_uint2(vx.y, vy.y);
                            dst[2] = make_uint2(vx.z, vy.z);
                            dst[3] = make_uint2(vx.w, vy.w);
                        }
                    }
                    named_bar_sync(1, 256);
                    cur_b = b;
                }
                load_tables(b, t0, real);
            }
            const uint32_t buf = j & 1;
            const bool ok = mbar_wait_cluster(&t_full[buf], (j >> 1) & 1, abort_flag);
            if (!ok) fail();
            float fin[HPU][G];     // this thread's sums for the token it finishes
#pragma unroll
            for (int hx = 0; hx < HPU; ++hx)
#pragma unroll
                for (int jq = 0; jq < G; ++jq) fin[hx][jq] = 0.0f;
            if (ok) {
                fence_after();
                const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
                for (int hx = 0; hx < HPU; ++hx) {
#pragma unroll
                    for (int pass = 0; pass < 2 / LHP; ++pass) {
                        uint64_t acc2[R][G];   // (even, odd) frequency partial sums per token and q-head
#pragma unroll
                        for (int k = 0; k < R; ++k)
#pragma unroll
                            for (int jq = 0; jq < G; ++jq) acc2[k][jq] = 0ull;
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {     // frequency blocks c = 2cc, 2cc+1
                            const uint32_t col = buf * UN + hx * 128 + fh * 32 + cc * 16;
                            float xv[LHP][8], yv[LHP][8];
                            if (LHP == 2)
                                tmem_ld_16x256b_4x2(lane_base + col, lane_base + (16u << 16) + col,
                                                    lane_base + col + 64, lane_base + (16u << 16) + col + 64,
                                                    xv[0], xv[LHP - 1], yv[0], yv[LHP - 1]);
                            else
                                tmem_ld_16x256b_2x2(lane_base + ((uint32_t)(16 * pass) << 16) + col,
                                                    lane_base + ((uint32_t)(16 * pass) << 16) + col + 64, xv[0],
                                                    yv[0]);
#pragma unroll
                            for (int cb = 0; cb < 2; ++cb) {
                                const int c = 2 * cc + cb;
                                uint64_t kx2[R], ky2[R];
#pragma unroll
                                for (int k = 0; k < R; ++k) {
                                    const int lhk = (LHP == 2) ? (k >> 1) : 0, ik = (LHP == 2) ? (k & 1) : k;
                                    const int kk = (LHP == 2) ? k : 2 * pass + k;   // index into c2/s2
                                    const uint64_t x2 = f2_pack(xv[lhk][cb * 4 + 2 * ik], xv[lhk][cb * 4 + 2 * ik + 1]);
                                    const uint64_t y2 = f2_pack(yv[lhk][cb * 4 + 2 * ik], yv[lhk][cb * 4 + 2 * ik + 1]);
                                    kx2[k] = f2_sub(f2_mul(x2, c2[kk][c]), f2_mul(y2, s2[kk][c]));   // x cos - y sin
                                    ky2[k] = f2_fma(y2, c2[kk][c], f2_mul(x2, s2[kk][c]));            // y cos + x sin
                                }
#pragma unroll
                                for (int jq = 0; jq < G; ++jq) {
                                    const uint2 qw = Qs[((u * HPU + hx) * G + jq) * 32 + fh * 16 + 4 * c + g4];
                                    // bf16 pair -> fp32 pair: the low half shifted up, the high half masked
                                    const uint64_t qx2 = f2_pack(__uint_as_float(qw.x << 16), __uint_as_float(qw.x & 0xffff0000u));
                                    const uint64_t qy2 = f2_pack(__uint_as_float(qw.y << 16), __uint_as_float(qw.y & 0xffff0000u));
#pragma unroll
                                    for (int k = 0; k < R; ++k) {
                                        acc2[k][jq] = f2_fma(qx2, kx2[k], acc2[k][jq]);
                                        acc2[k][jq] = f2_fma(qy2, ky2[k], acc2[k][jq]);
                                    }
                                }
                            }
                        }
                        // sum over the four lanes sharing a token (g4): reduce-scatter by lane bits
#pragma unroll
                        for (int jq = 0; jq < G; ++jq) {
                            float v[R];
#pragma unroll
                            for (int k = 0; k < R; ++k) {
                                const float2 h2 = f2_unpack(acc2[k][jq]);
                                v[k] = h2.x + h2.y;
                            }
                            if (LHP == 2) {
                                // keep lane half lh = b0, then token i = b1
                                float k0 = b0 ? v[R - 2] : v[0], k1 = b0 ? v[R - 1] : v[1];
                                const float s0 = b0 ? v[0] : v[R - 2], s1 = b0 ? v[1] : v[R - 1];
                                k0 += __shfl_xor_sync(0xffffffffu, s0, 1);
                                k1 += __shfl_xor_sync(0xffffffffu, s1, 1);
                                const float kk = b1 ? k1 : k0, ss = b1 ? k0 : k1;
                                fin[hx][jq] = kk + __shfl_xor_sync(0xffffffffu, ss, 2);
                            } else {
                                // keep token i = b0, then sum the b1 pair (both lanes hold the total)
                                float k0 = b0 ? v[R - 1] : v[0];
                                const float s0 = b0 ? v[0] : v[R - 1];
                                k0 += __shfl_xor_sync(0xffffffffu, s0, 1);
                                k0 += __shfl_xor_sync(0xffffffffu, k0, 2);
                                if (pass == fh) {
                                    fin[hx][jq] = k0;
                                } else if (b1 == 0) {   // the other half finishes this token
                                    const int orow = quarter * 32 + 16 * pass + 8 * b0 + r8;
                                    Xs[(buf * 128 + orow) * 16 + hx * G + jq] = k0;
                                }
                            }
                        }
                    }
                }
                fence_before();
                if (rank == 0) {
                    mbar_arrive_relaxed(&t_empty[buf]);
                } else {
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote_relaxed(peer_smem(&t_empty[buf], 0));
                }
            }
            // this item's tile, for the stores below; then, when the next item starts a new tile of the same
            // sequence, its tables are fetched now (this item's math is done with them), so that the loads run
            // during the exchange, the stores and the next accumulator wait
            const int sb = b, st0 = t0;
            const bool sreal = real;
            if (it + 1 < it_end) {
                int u2, pr2;
                item_up(it + 1, u2, pr2);
                if (pr2 != cur_pr) {
                    int b2, t02;
                    bool real2;
                    pair_tile(p, pr2, (int)rank, b2, t02, real2);
                    if (b2 == cur_b) {
                        cur_pr = pr2;
                        b = b2;
                        t0 = t02;
                        real = real2;
                        load_tables(b, t0, real);
                    }
                }
            }
            float* xs = Xs + (buf * 128 + frow) * 16;
            if (LHP == 2 && fh == 1)
#pragma unroll
                for (int hx = 0; hx < HPU; ++hx)
#pragma unroll
                    for (int jq = 0; jq < G; ++jq) xs[hx * G + jq] = fin[hx][jq];
            named_bar_sync(1, 256);      // (exchange buffers alternate by unit, so one barrier per unit)
            const int t = st0 + frow;
            if (finisher && ok && sreal && t < p.T) {
                // the unit's HPU * G q-heads of token t are contiguous in sall: vector stores where they align
                float sc[HPU * G];
#pragma unroll
                for (int hx = 0; hx < HPU; ++hx) {
                    const int h = u * HPU + hx;
                    float best = -INFINITY;
#pragma unroll
                    for (int jq = 0; jq < G; ++jq) {
                        sc[hx * G + jq] = (fin[hx][jq] + xs[hx * G + jq]) * p.scale;
                        best = fmaxf(best, sc[hx * G + jq]);
                    }
                    p.key[((int64_t)sb * p.H_kv + h) * p.T + t] = best;
                }
                if (p.sall) {
                    float* dst = p.sall + ((int64_t)sb * p.T + t) * p.H_q + u * HPU * G;
                    if constexpr ((HPU * G) % 4 == 0) {
#pragma unroll
                        for (int v = 0; v < HPU * G; v += 4)
                            *reinterpret_cast<float4*>(dst + v) = make_float4(sc[v], sc[v + 1], sc[v + 2], sc[v + 3]);
                    } else {
#pragma unroll
                        for (int v = 0; v < HPU * G; ++v) dst[v] = sc[v];
                    }
                }
            }
        }
    }

    // ---------------------------------------------------------------------- teardown
    fence_before();
    __syncthreads();
    cluster_sync();      // neither CTA leaves while the other may still touch its shared memory
    if (*abort_flag && threadIdx.x == 0) flag(p.check, LOWRAM_CHECK_TIMEOUT);
    if (warp == 1) {
        fence_after();
        tmem_dealloc_pair(tmem, 2 * UN);
    }
}

// ------------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------------
using tc::encode_fn;
using tc::make_map;
using tc::sm_count;

// Unit width (basis rows per MMA) and ring depth: two heads per unit when the kv-heads pair up, else one;
// as many stages as fit beside the queries.
struct ScoreConfig {
    int UN, NS;
};

ScoreConfig score_config(int H_q, int H_kv) {
    const int UN = (H_kv % 2 == 0 && H_q / H_kv != 8) ? 256 : 128;   // two heads of eight queries: registers
    for (int ns = 8; ns >= 2; --ns)
        if (score_smem_bytes(ns, UN, H_q) <= (size_t)kSmemLimit) return {UN, ns};
    return {0, 0};
}

bool g_ok(int g) { return g == 1 || g == 2 || g == 4 || g == 7 || g == 8; }

}  // namespace

bool tc_score_supported(const lowram_decode_shape& s) {
    const int g = s.H_q / s.H_kv;
    return s.act_dtype == LOWRAM_BF16 && (s.coef_dtype == LOWRAM_BF16 || s.coef_dtype == kCoefF16) && s.d == 128 &&
           s.r % kChunkK == 0 &&
           s.r <= 1024 && g_ok(g) && s.T > 0 && s.H_q <= 128 && score_config(s.H_q, s.H_kv).NS >= 2 &&
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
    p.pps = s.basis_batch_stride ? (p.tiles_per_seq + 1) / 2 : 0;
    const bool f16 = s.coef_dtype == kCoefF16;
    p.KC = s.r / kChunkK;
    const ScoreConfig cfg = score_config(s.H_q, s.H_kv);
    p.NU = s.H_kv * s.d / cfg.UN;
    p.idesc = s.coef_dtype == kCoefF16 ? tc::idesc_f16(2 * kTokTile, cfg.UN) : tc::idesc_bf16(2 * kTokTile, cfg.UN);
    p.NS = cfg.NS;
    p.scale = a.scale;
    p.q = (const __nv_bfloat16*)a.q;
    p.pos = a.pos;
    p.rcos = a.rope_cos;
    p.rsin = a.rope_sin;
    p.key = a.key;
    p.sall = a.sall;
    p.check = a.check;
    if (p.n_tiles == 0) return cudaSuccess;
    if (cfg.NS < 2) return cudaErrorNotSupported;
    CUtensorMap mA, mB;
    const uint64_t dA[3] = {(uint64_t)s.r, (uint64_t)s.T, (uint64_t)s.B};
    const uint32_t bA[3] = {kChunkK, kTokTile, 1};
    const uint64_t dB[3] = {(uint64_t)s.r, (uint64_t)s.H_kv * s.d, (uint64_t)s.B};
    const uint32_t bB[3] = {kChunkK, (uint32_t)cfg.UN / 2, 1};
    if (!make_map(&mA, a.coef, 3, dA, bA, 0, f16) ||
        !make_map(&mB, a.basis, p.pps ? 3 : 2, dB, bB, p.pps ? (uint64_t)s.basis_batch_stride : 0, f16))
        return cudaErrorInvalidValue;
    const size_t smem = score_smem_bytes(p.NS, cfg.UN, s.H_q);
    // CTA pairs (cluster of two), at most one CTA per SM
    const int n_pairs = p.pps ? s.B * p.pps : (p.n_tiles + 1) / 2;
    const int grid = 2 * std::min(n_pairs * p.NU, std::max(1, sm_count() / 2));
    cudaError_t e = cudaSuccess;
    auto go = [&](auto kern) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) {
            kern<<<grid, kScoreThreads, smem, st>>>(mA, mB, p);
            e = cudaGetLastError();
        }
    };
    const bool two = cfg.UN == 256;
#define LOWRAM_SCORE_GO(G_) (two ? go(score_tc_kernel<G_, 2>) : go(score_tc_kernel<G_, 1>))
    switch (s.H_q / s.H_kv) {
        case 1: LOWRAM_SCORE_GO(1); break;
        case 2: LOWRAM_SCORE_GO(2); break;
        case 4: LOWRAM_SCORE_GO(4); break;
        case 7: LOWRAM_SCORE_GO(7); break;
        case 8: LOWRAM_SCORE_GO(8); break;
        default: return cudaErrorNotSupported;
    }
#undef LOWRAM_SCORE_GO
    return e;
}

}  // namespace lowram
