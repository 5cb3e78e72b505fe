// tc_vregen.cu -- tensor-core (tcgen05) value regeneration for the selected tokens of bf16 caches (K3): one
// split-softmax record per 128-token chunk, merged by the merge kernel launched after it.
//
// The method: each decode step rebuilds only a selected subset of KV pairs (LowRAM abstract); a selected
// token's value is predicted from its pre-RoPE key by the head's MLP, plus the stored residual when the
// token is one of the worst-predicted ("Value cache amortisation in plain language", LowRAM Paper:
// Amortised Values and Low-Rank Keys for KV Compression; flowchart "Values are mostly a function of keys"
// of the wiki page).  The key itself comes from the low-rank factors ("Asymmetric key compression with
// xKV").
//
// Two reassociations, exact in real arithmetic, shape the kernel:
//   - the predictor's first layer acts on the rebuilt key, w1 (basis_h c) = (w1 basis_h) c, so the hidden
//     pre-activations of a selected token are one product of its latent row with F_h = w1[h] basis_h [m x r]
//     (folded once per call by spare CTAs of the selection kernel, stored bf16 -- fp16 for an int4 cache's fp16
//     copy -- in the workspace);
//   - the second layer is linear, so sum_t p_t (w2 s_t + b2 + r_t) = w2 (sum_t p_t s_t) + b2 sum_t p_t +
//     sum_t p_t r_t: a chunk applies w2 once per q-head to its softmax-weighted hidden sums, never forming the
//     tokens' values, and writes a plain flash-decoding record (weighted value sum, max logit, weight sum).
// The result equals regenerating the selected values and then attending, up to rounding order; F in bf16 rounds the
// folded weights where the unfolded chain would round the rebuilt keys.
//
// K3 is persistent: one CTA per SM walks a contiguous range of work items (kv-head h, sequence b, chunk of 128
// selected tokens), kv-head-major, so consecutive items share F_h, which stays resident in TMEM (m = 128,
// r <= 512) or in shared memory while it fits (else each ring stage carries its F chunk).  512 threads, launched at 128 registers each and re-split
// per warpgroup (setmaxnreg): 56 for warps 0-7, 200 for the epilogue warps 8-15:
//   warp 0      lane 0: TMA of F_h's k-chunks [m x 64] once per kv-head (into two staging buffers in TMEM
//               mode, into the resident copy otherwise) or per stage when streamed;
//   warp 1      TMEM owner (two accumulators of m columns) and MMA issuer (one thread):
//               D[m hidden x 128 tokens] = F_h . C_sel^T (M = 128 per 128 hidden units, N = 128, K = r), hidden
//               units on TMEM lanes, tokens on columns; item j accumulates into buffer j % 2.  In TMEM mode it
//               copies F_h's staged chunks into TMEM beside the accumulators (tcgen05.cp, once per kv-head) and
//               the MMAs read their A operand there: shared memory holds only 32 KB of staging and a deeper ring.
//   warps 2-3   idle (their warpgroup's registers go to the epilogue).
//   warps 4-7   gather: 16-byte cp.async of the selected tokens' latent rows into the 128B-swizzled ring, one
//               64-wide k-chunk per stage; the copies arrive on the stage's barrier when they land, so the warps
//               never wait for them and run ahead into the next items as far as the free slots allow.
//   warps 8-15  epilogue in two teams of four warps: team t takes the items j = t, t + 2, ... (TMEM buffer t),
//               each with its own scratch and named barrier, while the next items' rows land and multiply:
//               softmax weights of the chunk from the scaled logits the key pass stored (fetched a team item
//               ahead), the residual rows of the chunk's hits (loads issued before, used after, the accumulator
//               read); per thread one hidden unit and all 128 tokens: SiLU(D + b1) weighted by the softmax,
//               summed; the TMEM buffer is released; w2 (rows held in registers per kv-head) on the hidden sums;
//               the chunk's record.
// The records are merged by a separate kernel (a dependent launch): merging in the CTA that finished a
// (sequence, kv-head) last put a merge after the slowest CTA's last record and measured slower.
//
// Every pipeline wait is bounded by the call's wait limit (a parameter); on a timeout the kernel sets
// LOWRAM_CHECK_TIMEOUT, lets the copies and MMAs it issued complete, frees TMEM and returns.  Every named
// barrier is reached on every path.
#include "kernels.h"
#include "predict.cuh"
#include "tc_common.cuh"

namespace lowram {

namespace {

constexpr int kVThreads = 512;            // 16 warps launched at 128 registers a thread, then re-split:
constexpr int kProdRegs = 56;             //   warps 0-7 (TMA, MMA, gather) give registers back,
constexpr int kEpiRegs = 200;             //   warps 8-15 (epilogue) take them: 256 x 56 + 256 x 200 = 512 x 128
constexpr int kGat = 128;                 // gathering threads (warps 4-7)
constexpr int kTeam = 128;                // epilogue team: warps 8-11 and warps 12-15
constexpr int kRows = 128;               // selected tokens per item
constexpr int kCBytes = kRows * 128;     // latent chunk [128 tokens x 64] bf16, 128B-swizzled
constexpr int kGatRows = kRows / (kGat / 8);   // rows each gathering thread copies per stage
constexpr int kMaxStages = 12;
constexpr int kFStage = 2;               // TMEM mode: F_h staging buffers of 16 KB
constexpr size_t kSmemMax = 232448;

struct VregenTcParams {
    int B, T, H_q, H_kv, m, r, S_eff, n_chunks, n_res, KC, NS, n_items;
    int f_resident;           // F_h stays in shared memory for all of a kv-head's items
    int f_tmem;               // F_h stays in TMEM (M = 128, r <= 512), loaded once per kv-head through
                              // kFStage staging buffers; neither: F_h streamed with every ring stage
    int fold_per_seq;         // the folded weights hold one copy per sequence
    uint32_t idesc;           // MMA instruction descriptor: bf16 operands, or fp16 (an int4 cache's fp16 copy)
    long long mlp_stride;     // elements from sequence b's w2 to b+1's (0: shared); biases are then per sequence
    long long wait_cycles;
    const __nv_bfloat16* coef;   // [B, T, r] latent coefficients (2-byte elements; fp16 for an int4 cache's copy)
    const float* sall;        // [B, T, H_q] scaled logits written by the key pass
    const float* b1;          // [H_kv, m] ([B, H_kv, m] with a predictor per sequence) or null
    const float* b2;          // [H_kv, d] ([B, H_kv, d] likewise) or null
    const __nv_bfloat16* w2;  // [H_kv, d, m], sequence b's at b * mlp_stride
    const int32_t* sel;       // [B, H_kv, S_eff]
    const int32_t* hit;       // [B, H_kv, S_eff] residual row of each selected token, or -1; null without residuals
    ResView res;
    float* partial;           // [B, H_q, n_chunks, d + 2]
    uint32_t* check;
};

// The second layer's operand: the chunk's hidden sums as bf16 hi + lo columns, 2g of them in n-tiles of 8.
__host__ __device__ constexpr int w2_ntiles(int g) { return (2 * g + 7) / 8; }
constexpr int kWoStride = 132;           // floats per row of the second layer's output (conflict-free stores)

// One epilogue team's scratch in 4-byte words, for g q-heads per kv-head: softmax weights [g][128], hidden sums
// [g][m], the second layer's output [8 nt][132] and operand [8 nt][m + 8] bf16, compacted hits (rows, slots),
// reductions [2][32] + counts [4]; a multiple of 4 words (16-byte aligned).
__host__ __device__ constexpr int team_words(int m, int g) {
    return (g * kRows + g * m + w2_ntiles(g) * 8 * kWoStride + w2_ntiles(g) * 4 * (m + 8) + 2 * kRows + 64 + 4 + 3) &
           ~3;
}
// Scratch beside the ring: two teams' scratch, then the barriers and the TMEM slot / abort flag.
size_t scratch_bytes(int m, int g) {
    return (size_t)8 * team_words(m, g) + 8 + 8 * (3 * kMaxStages + 2 * kFStage + 4 + 1) + 16;
}

struct VregenConfig {
    bool f_tmem, f_resident;
    int NS;
    size_t smem;
};

VregenConfig vregen_config(int m, int r, int g) {
    const int KC = r / 64;
    const size_t fres = (size_t)KC * m * 128, fixed = 1024 + scratch_bytes(m, g);
    VregenConfig c{};
    if (m == 128 && 2 * m + r / 2 <= 512) {
        // two accumulators and F_h fit the SM's 512 TMEM columns: F_h passes through kFStage 16 KB staging buffers
        const size_t fst = kFStage * (size_t)kCBytes;
        c.f_tmem = true;
        c.NS = (int)std::min<size_t>(kMaxStages, (kSmemMax - fst - fixed) / kCBytes);
        c.smem = fst + fixed + (size_t)c.NS * kCBytes;
    } else if (fres + fixed + 3 * (size_t)kCBytes <= kSmemMax) {
        c.f_resident = true;
        c.NS = (int)std::min<size_t>(kMaxStages, (kSmemMax - fres - fixed) / kCBytes);
        c.smem = fres + fixed + (size_t)c.NS * kCBytes;
    } else {
        const size_t stage = kCBytes + (size_t)m * 128;
        c.f_resident = false;
        c.NS = (int)std::min<size_t>(kMaxStages, (kSmemMax - fixed) / stage);
        c.smem = fixed + (size_t)c.NS * stage;
    }
    return c;
}

// SiLU(x) = x sigmoid(x), with sigmoid(x) = (1 + tanh(x / 2)) / 2 and tanh from the hardware approximation
// (tanh.approx.f32, relative error about 2^-11): one special-function operation per unit instead of an exponential
// and a reciprocal.  The error it adds is far below the bf16 rounding of the folded weights.
__device__ __forceinline__ float silu_tanh(float x) {
    const float h = 0.5f * x;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}


template <int G, int MB>
__global__ void __launch_bounds__(kVThreads, 1)
    vregen_tc_kernel(const __grid_constant__ CUtensorMap tmF, VregenTcParams p) {
    using namespace tc;
    constexpr int M = MB * 128;              // hidden units (TMEM lanes x column blocks)
    constexpr uint32_t kFChunk = M * 128;    // one k-chunk of F_h [M x 64]
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int NS = p.NS, KC = p.KC;
    const bool fres = p.f_resident != 0;
    const bool ftm = p.f_tmem != 0;
    const uint32_t tmem_cols = ftm ? 512u : (uint32_t)(2 * M);
    const uint32_t kStage = kCBytes + (fres || ftm ? 0u : kFChunk);
    uint8_t* Fres = smem;   // [KC][M x 64] when resident; [kFStage][M x 64] staging buffers in TMEM mode
    uint8_t* ring = smem + (fres ? (size_t)KC * kFChunk : ftm ? kFStage * (size_t)kFChunk : 0);   // NS stages: C
                                                                                               // chunk (+ F chunk)
    float* epi = (float*)(ring + (size_t)NS * kStage);           // [2 teams][team_words] epilogue scratch
    constexpr int NT = w2_ntiles(G);
    uint64_t* fullF = (uint64_t*)(((uintptr_t)(epi + 2 * team_words(M, G)) + 7) & ~(uintptr_t)7);   // streamed F
                                                                                                  // chunk landed
    uint64_t* fullC = fullF + kMaxStages;        // the 128 gathering threads' rows of the stage landed
    uint64_t* empty = fullC + kMaxStages;        // the MMAs are done with the stage
    uint64_t* f_full = empty + kMaxStages;       // resident F_h landed ([kFStage]: a staging buffer landed)
    uint64_t* f_empty = f_full + kFStage;        // the MMAs are done with the resident F_h ([kFStage]: in TMEM)
    uint64_t* t_full = f_empty + kFStage;        // [2] accumulator ready
    uint64_t* t_empty = t_full + 2;              // [2] epilogue done reading the accumulator
    uint64_t* m_drain = t_empty + 2;
    uint32_t* tmem_slot = (uint32_t*)(m_drain + 1);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
    if (layout_overflows(smem_raw, (const void*)(abort_flag + 1), p.check)) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int it_begin = (int)((int64_t)blockIdx.x * p.n_items / gridDim.x);
    const int it_end = (int)((int64_t)(blockIdx.x + 1) * p.n_items / gridDim.x);
    const int n_local = it_end - it_begin;
    // item -> (h, b, chunk), kv-head-major; the folded weights of an item sit at row fh(it) * M of the F map
    auto item_hbc = [&](int it, int& h, int& b, int& c) {
        c = it % p.n_chunks;
        const int hb = it / p.n_chunks;
        b = hb % p.B;
        h = hb / p.B;
    };
    auto item_fh = [&](int it) {
        int h, b, c;
        item_hbc(it, h, b, c);
        return (p.fold_per_seq ? b * p.H_kv : 0) + h;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&fullF[s], 1);
            mbar_init(&fullC[s], kGat);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < kFStage; ++i) {
            mbar_init(&f_full[i], 1);
            mbar_init(&f_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&t_full[i], 1);
            mbar_init(&t_empty[i], kTeam);
        }
        mbar_init(m_drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) prefetch_tmap(&tmF);
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dep_wait();     // selection, residual rows, folded weights and logits come from the kernels before

    if (warp < 8) {
        // warpgroups 0-1 drop to 56 registers a thread so that warpgroups 2-3 can rise to 200
        // (256 x 56 + 256 x 200 = 512 x 128, the registers the CTA was launched with)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProdRegs));
        if (warp == 0) {
            // ------------------------------------------------------------------ TMA: F_h
            if (lane == 0) {
                int n_seg = 0, cur_fh = -1;                 // resident: kv-head segments loaded
                uint32_t issued = 0;                        // streamed: stages issued; TMEM mode: chunks staged
                for (int j = 0; j < n_local && !*abort_flag; ++j) {
                    const int fh = item_fh(it_begin + j);
                    if (ftm) {
                        // TMEM mode: the segment's KC chunks through the staging buffers, each reused once the MMA
                        // thread has copied what it held into TMEM
                        if (fh == cur_fh) continue;
                        bool ok = true;
                        for (int kc = 0; kc < KC; ++kc, ++issued) {
                            const uint32_t fb = issued % kFStage, n = issued / kFStage;
                            if (!mbar_wait_lim(&f_empty[fb], (n & 1) ^ 1, abort_flag, p.wait_cycles)) {
                                ok = false;
                                break;
                            }
                            mbar_expect_tx(&f_full[fb], kFChunk);
                            tma_load_2d(Fres + fb * kFChunk, &tmF, &f_full[fb], kc * 64, fh * M);
                        }
                        if (!ok) break;
                        cur_fh = fh;
                    } else if (fres) {
                        if (fh == cur_fh) continue;
                        // the MMAs of the previous segment are done with F before it is overwritten
                        if (n_seg > 0 && !mbar_wait_lim(f_empty, (n_seg - 1) & 1, abort_flag, p.wait_cycles)) break;
                        mbar_expect_tx(f_full, (uint32_t)KC * kFChunk);
                        for (int kc = 0; kc < KC; ++kc)
#pragma unroll
                            for (int mb = 0; mb < MB; ++mb)
                                tma_load_2d(Fres + kc * kFChunk + mb * 16384, &tmF, f_full, kc * 64, fh * M + mb * 128);
                        cur_fh = fh;
                        ++n_seg;
                    } else {
                        bool ok = true;
                        for (int kc = 0; kc < KC; ++kc, ++issued) {
                            const uint32_t s = issued % NS, n = issued / NS;
                            if (!mbar_wait_lim(&empty[s], (n & 1) ^ 1, abort_flag, p.wait_cycles)) {
                                ok = false;
                                break;
                            }
                            mbar_expect_tx(&fullF[s], kFChunk);
#pragma unroll
                            for (int mb = 0; mb < MB; ++mb)
                                tma_load_2d(ring + s * kStage + kCBytes + mb * 16384, &tmF, &fullF[s], kc * 64,
                                            fh * M + mb * 128);
                        }
                        if (!ok) break;
                    }
                }
                if (*abort_flag) {   // copies issued complete before the CTA frees its shared memory
                    if (ftm)
                        for (uint32_t k = issued > (uint32_t)kFStage ? issued - kFStage : 0; k < issued; ++k)
                            mbar_wait_drain(&f_full[k % kFStage], (k / kFStage) & 1);
                    else if (fres && n_seg > 0)
                        mbar_wait_drain(f_full, (n_seg - 1) & 1);
                    else if (!fres)
                        for (uint32_t k = issued > (uint32_t)NS ? issued - NS : 0; k < issued; ++k)
                            mbar_wait_drain(&fullF[k % NS], (k / NS) & 1);
                }
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------------ MMA issuer
            if (lane == 0) {
                bool ok = true;
                int n_seg = 0, cur_fh = -1, n_drain = 0;
                uint32_t n_fst = 0;                                  // TMEM mode: staged F chunks copied
                uint32_t s = 0, par = 0;                             // ring slot and phase of the next stage
                for (int j = 0; j < n_local && ok; ++j) {
                    const int fh = item_fh(it_begin + j);
                    if ((fres || ftm) && fh != cur_fh) {
                        if (fres && !mbar_wait_lim(f_full, n_seg & 1, abort_flag, p.wait_cycles)) break;
                        if (ftm && n_seg > 0) {
                            // the MMAs of the kv-head before still read its F_h from TMEM: let them finish first (a copy
                            // is not ordered after earlier MMAs)
                            mma_commit(m_drain);
                            if (!mbar_wait_lim(m_drain, n_drain & 1, abort_flag, p.wait_cycles)) break;
                            ++n_drain;
                        }
                        cur_fh = fh;
                        ++n_seg;
                        // TMEM mode: F_h into TMEM columns [2M, 2M + r/2), k-chunk kc at column 32 kc, 8 columns per
                        // 16 k-values, from the staging buffers (each freed once its copies have read it)
                        for (int kc = 0; ftm && kc < KC; ++kc, ++n_fst) {
                            const uint32_t fb = n_fst % kFStage;
                            if (!mbar_wait_lim(&f_full[fb], (n_fst / kFStage) & 1, abort_flag, p.wait_cycles)) {
                                ok = false;
                                break;
                            }
                            fence_after();
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tmem_cp_128x256b(tmem + 2 * M + kc * 32 + k * 8,
                                                 sdesc_sw128(smem_u32(Fres + fb * kFChunk) + k * 32));
                            mma_commit(&f_empty[fb]);
                        }
                        if (!ok) break;
                    }
                    const uint32_t buf = j & 1;
                    if (!mbar_wait_lim(&t_empty[buf], ((j >> 1) & 1) ^ 1, abort_flag, p.wait_cycles)) break;
                    fence_after();
                    for (int kc = 0; kc < KC; ++kc) {
                        if (!mbar_wait_lim(&fullC[s], par, abort_flag, p.wait_cycles) ||
                            (!fres && !ftm && !mbar_wait_lim(&fullF[s], par, abort_flag, p.wait_cycles))) {
                            ok = false;
                            break;
                        }
                        // the gatherers' cp.async bytes (generic proxy) before the MMAs' reads (async proxy)
                        fence_proxy_async();
                        fence_after();
                        const uint32_t c_addr = smem_u32(ring + s * kStage);
                        if (ftm) {
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_bf16_ts(tmem + buf * M, tmem + 2 * M + kc * 32 + k * 8, sdesc_sw128(c_addr + k * 32),
                                            p.idesc, (kc | k) != 0);
                        } else {
                            const uint32_t f_addr = fres ? smem_u32(Fres + kc * kFChunk) : c_addr + kCBytes;
#pragma unroll
                            for (int mb = 0; mb < MB; ++mb)
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    mma_bf16(tmem + buf * M + mb * 128, sdesc_sw128(f_addr + mb * 16384 + k * 32),
                                             sdesc_sw128(c_addr + k * 32), p.idesc, (kc | k) != 0);
                        }
                        mma_commit(&empty[s]);
                        if (++s == (uint32_t)NS) {
                            s = 0;
                            par ^= 1;
                        }
                    }
                    if (!ok) break;
                    mma_commit(&t_full[buf]);
                    // the last item of a kv-head segment: its MMAs release the resident F_h
                    if (fres && (j + 1 == n_local || item_fh(it_begin + j + 1) != fh)) mma_commit(f_empty);
                }
                // every MMA issued completes before TMEM is released or shared memory is reused
                mma_commit(m_drain);
                mbar_wait_drain(m_drain, n_drain & 1);
            }
        } else if (warp < 4) {
            // warps 2-3 idle
        } else if (warp < 8) {
            // ------------------------------------------------------------------ gather (128 threads)
            // thread gt copies the 16-byte piece c16 of rows rsub + 16 rr (rr < 8) of every k-chunk; a padding slot
            // re-reads its sequence's token 0 (its softmax weight is 0).  The copies of a stage arrive on its full
            // barrier by themselves once they land (one arrival per thread), so the warps never wait for a copy:
            // they run ahead as far as the ring's free slots allow.
            const int gt = threadIdx.x - 128, c16 = gt & 7, rsub = gt >> 3;
            const uint32_t total = (uint32_t)n_local * KC;
            const __nv_bfloat16* srow[kGatRows];
            int nsel[kGatRows];   // the next item's selected tokens, loaded an item ahead
            auto load_sel = [&](int jl) {
                int h, b, c;
                item_hbc(it_begin + jl, h, b, c);
                const int64_t bh = (int64_t)b * p.H_kv + h;
#pragma unroll
                for (int rr = 0; rr < kGatRows; ++rr) {
                    const int jr = c * kRows + rr * (kGat / 8) + rsub;
                    nsel[rr] = jr < p.S_eff ? __ldg(p.sel + bh * p.S_eff + jr) : 0;
                }
            };
            if (n_local > 0) load_sel(0);
            for (uint32_t issued = 0; issued < total; ++issued) {
                const uint32_t s = issued % NS, n = issued / NS;
                const int kc = (int)(issued % KC);
                if (kc == 0) {   // the item's rows; then the next item's tokens
                    const int jl = (int)(issued / KC);
                    int h, b, c;
                    item_hbc(it_begin + jl, h, b, c);
#pragma unroll
                    for (int rr = 0; rr < kGatRows; ++rr) {
                        const int t = min(max(nsel[rr], 0), p.T - 1);
                        srow[rr] = p.coef + ((int64_t)b * p.T + t) * p.r + c16 * 8;
                    }
                    if (jl + 1 < n_local) load_sel(jl + 1);
                }
                // the slot frees when the MMAs of its previous round are done
                if (!mbar_wait_lim(&empty[s], (n & 1) ^ 1, abort_flag, p.wait_cycles)) break;
                const uint32_t A = smem_u32(ring + s * kStage);
#pragma unroll
                for (int rr = 0; rr < kGatRows; ++rr) {
                    const int row = rr * (kGat / 8) + rsub;
                    cp_async_16(A + row * 128 + ((c16 ^ (row & 7)) << 4), srow[rr] + kc * 64, 16u);
                }
                cp_async_mbar_arrive(&fullC[s]);
            }
            cp_async_wait<0>();
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs));
        // ------------------------------------------------------------------ epilogue (two teams of 128 threads)
        // Team tm (warps 8 + 4 tm .. 11 + 4 tm) takes the items j = tm, tm + 2, ... and TMEM buffer tm, with its
        // own scratch and named barrier, so that one team's barrier and load waits overlap the other's arithmetic.
        // Thread et of a team: token slot et for the softmax, hidden unit 32 q + lane (its TMEM lane) for the
        // hidden layer, output feature et for the residual rows and the record.
        const int tm = (warp - 8) >> 2, et = threadIdx.x - 256 - kTeam * tm;
        const int q = warp & 3;                      // TMEM lane quarter = slot quarter of the softmax
        const int slot = et, i_out = et;
        float* Ps = epi + (size_t)tm * team_words(M, G);        // [G][128] softmax weights (0 on padding slots)
        float* Z = Ps + G * kRows;                               // [G][M] hidden sums
        float* Wo = Z + G * M;                                   // [8 NT][132] second layer: rows n, features i
        __nv_bfloat16* Zs = reinterpret_cast<__nv_bfloat16*>(Wo + NT * 8 * kWoStride);   // [8 NT][M + 8] its operand
        int* HitRow = reinterpret_cast<int*>(Zs + NT * 8 * (M + 8));   // compacted residual rows of the chunk's slots
        int* HitSlot = HitRow + kRows;                           // ... and those slots, ascending
        float* redM = (float*)(HitSlot + kRows);                 // [4 slot quarters][8] partial max
        float* redL = redM + 32;                                 // [4][8] partial sums
        int* hcount = (int*)(redL + 32);                         // [4] residual hits per slot quarter
        auto team_sync = [&]() { named_bar_sync(1 + tm, kTeam); };
        auto chunk_max = [&](int jq) {
            return fmaxf(fmaxf(redM[jq], redM[8 + jq]), fmaxf(redM[16 + jq], redM[24 + jq]));
        };
        auto chunk_sum = [&](int jq) { return (redL[jq] + redL[8 + jq]) + (redL[16 + jq] + redL[24 + jq]); };
        const int64_t rw = 128 + 2;
        const int64_t qstride = (int64_t)p.n_chunks * rw;
        // this slot's selection data of an item, fetched a team item ahead in two steps so that no load waits on
        // the critical path: the token and its residual row when the item before starts, then (once the token
        // has landed) the scaled logits of the G q-heads
        auto fetch_sel = [&](int it, int& tok, int& hit) {
            int h, b, c;
            item_hbc(it, h, b, c);
            const int64_t bh = (int64_t)b * p.H_kv + h;
            const int jsel = c * kRows + slot;
            const bool valid = jsel < p.S_eff;
            tok = valid ? ldg_pin_s32(p.sel + bh * p.S_eff + jsel) : -1;
            hit = (valid && p.hit) ? ldg_pin_s32(p.hit + bh * p.S_eff + jsel) : -1;
        };
        auto fetch_logits = [&](int it, int& tok, float (&sv)[G]) {
            int h, b, c;
            item_hbc(it, h, b, c);
            if (tok >= p.T) tok = p.T - 1;   // the selection is always in range; keep the invariant explicit
            // the kv-head's G logits of the token are contiguous (vector loads where they align)
            const float* src = p.sall + ((int64_t)b * p.T + (tok >= 0 ? tok : 0)) * p.H_q + h * G;
            if constexpr (G % 4 == 0) {
#pragma unroll
                for (int v = 0; v < G; v += 4) {
                    const float4 x = ldg_pin_f32x4(src + v);
                    sv[v] = x.x;
                    sv[v + 1] = x.y;
                    sv[v + 2] = x.z;
                    sv[v + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int jq = 0; jq < G; ++jq) sv[jq] = ldg_pin_f32(src + jq);
            }
            if (tok < 0)
#pragma unroll
                for (int jq = 0; jq < G; ++jq) sv[jq] = -INFINITY;
        };
        // The second layer on warp MMAs: warp q of the team makes output features [32 q, 32 q + 32) of every
        // q-head (two m16 tiles), W[i][n] = sum_k w2[i][k] Zs[n][k], from its w2 rows in m16n8k16 A fragments.
        // With M = 128 the fragments stay in registers while the items' kv-head (and, with a predictor per
        // sequence, sequence) stays; with M = 256 they are loaded per item and tile.
        constexpr int KB = M / 16;
        constexpr int AT = M == 128 ? 2 : 1;                      // m16 tiles held at once
        const int fg = lane >> 2, ft = lane & 3;
        uint32_t af[AT][KB][4];
        auto load_af = [&](int h, int b, int mt, uint32_t (&a)[KB][4]) {
            const __nv_bfloat16* w = p.w2 + b * p.mlp_stride + ((int64_t)h * 128 + 32 * q + 16 * mt + fg) * M + 2 * ft;
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                // pinned where they stand (the item's start): they land during the accumulator wait
                a[kb][0] = ldg_pin_u32(w + kb * 16);
                a[kb][1] = ldg_pin_u32(w + 8 * M + kb * 16);
                a[kb][2] = ldg_pin_u32(w + kb * 16 + 8);
                a[kb][3] = ldg_pin_u32(w + 8 * M + kb * 16 + 8);
            }
        };
        int w2_key = -1;
        int nx_tok = -1, nx_hit = -1;
        float nx_sv[G];
        if (tm < n_local) {
            fetch_sel(it_begin + tm, nx_tok, nx_hit);
            fetch_logits(it_begin + tm, nx_tok, nx_sv);
        }
        for (int j = tm; j < n_local; j += 2) {
            int h, b, chunk;
            item_hbc(it_begin + j, h, b, chunk);
            const int64_t bh = (int64_t)b * p.H_kv + h;
            const int64_t bias_bh = p.mlp_stride ? bh : h;
            const int my_hit = nx_hit;
            float sv[G];
#pragma unroll
            for (int jq = 0; jq < G; ++jq) sv[jq] = nx_sv[jq];
            if (j + 2 < n_local) fetch_sel(it_begin + j + 2, nx_tok, nx_hit);
            if (M == 128) {
                const int key = p.mlp_stride ? (int)bh : h;
                if (key != w2_key) {
                    w2_key = key;
#pragma unroll
                    for (int mt = 0; mt < AT; ++mt) load_af(h, b, mt, af[mt]);
                }
            }
            team_sync();   // the previous item's readers of Ps, Z, the hits and the reductions are done
#pragma unroll
            for (int jq = 0; jq < G; ++jq) {
                const float mx = warp_max(sv[jq]);
                if (lane == 0) redM[q * 8 + jq] = mx;
            }
            const unsigned hb = __ballot_sync(0xffffffffu, my_hit >= 0);
            if (lane == 0) hcount[q] = __popc(hb);
            team_sync();
#pragma unroll
            for (int jq = 0; jq < G; ++jq) {
                const float mq = chunk_max(jq);
                const float pv = (sv[jq] == -INFINITY || mq == -INFINITY) ? 0.0f : __expf(sv[jq] - mq);
                Ps[jq * kRows + slot] = pv;
                const float ps = warp_sum(pv);
                if (lane == 0) redL[q * 8 + jq] = ps;
            }
            int n_hit = 0;
            {
                int before = 0;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    before += (w < q) ? hcount[w] : 0;
                    n_hit += hcount[w];
                }
                if (my_hit >= 0) {
                    const int at = before + __popc(hb & ((1u << lane) - 1u));
                    HitRow[at] = my_hit;
                    HitSlot[at] = slot;
                }
            }
            team_sync();

            // residual rows of the first 16 hits (feature i_out; int8 rows with their scales): loads issued now,
            // pinned here, their bits converted after the hidden units, so they land while the accumulator is read
            uint32_t rr[16], rs[16];
            const int64_t rbase = bh * p.n_res;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                rr[k] = 0u;
                rs[k] = 0u;
            }
            if (p.res.dtype == LOWRAM_BF16) {
                const unsigned short* rv16 = reinterpret_cast<const unsigned short*>(p.res.val);
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (k < n_hit) rr[k] = ldg_pin_u16(rv16 + (rbase + HitRow[k]) * 128 + i_out);
            } else if (p.res.dtype == LOWRAM_INT8_VEC) {
                const signed char* rv8 = reinterpret_cast<const signed char*>(p.res.val);
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (k < n_hit) {
                        const int64_t row = rbase + HitRow[k];
                        rr[k] = (uint32_t)ldg_pin_s8(rv8 + row * 128 + i_out);
                        rs[k] = ldg_pin_u16(p.res.scale + row);
                    }
            } else {
                const uint32_t* rv32 = reinterpret_cast<const uint32_t*>(p.res.val);
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (k < n_hit) rr[k] = ldg_pin_u32(rv32 + (rbase + HitRow[k]) * 128 + i_out);
            }

            // first- and second-layer biases of this thread's hidden units and output feature, pinned here too
            float bjs[MB];
#pragma unroll
            for (int mb = 0; mb < MB; ++mb)
                bjs[mb] = p.b1 ? ldg_pin_f32(p.b1 + bias_bh * M + mb * 128 + q * 32 + lane) : 0.0f;
            const float bias = p.b2 ? ldg_pin_f32(p.b2 + bias_bh * 128 + i_out) : 0.0f;

            // hidden units: thread = hidden unit jj of each 128-block, all 128 tokens;
            // z[jq] = sum over the tokens of p[jq, t] SiLU(D[jj, t] + b1[jj])
            const uint32_t buf = (uint32_t)tm;
            const bool have = mbar_wait_lim(&t_full[buf], (j >> 1) & 1, abort_flag, p.wait_cycles);
            if (have) {
                fence_after();
#pragma unroll 1
                for (int mb = 0; mb < MB; ++mb) {
                    const int jj = mb * 128 + q * 32 + lane;
                    const float bj = bjs[mb];
                    const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + buf * M + mb * 128;
                    float z[G];
#pragma unroll
                    for (int jq = 0; jq < G; ++jq) z[jq] = 0.0f;
                    constexpr int XG = G >= 7 ? 1 : 2;               // 32-column groups per TMEM wait (registers)
#pragma unroll 1
                    for (int c0 = 0; c0 < kRows; c0 += 32 * XG) {
                        float xv[XG][32];
                        if constexpr (XG == 2) {
                            tmem_ld_2x32(taddr + c0, taddr + c0 + 32, xv[0], xv[XG - 1]);
                        } else {
                            float (&x8)[4][8] = *reinterpret_cast<float (*)[4][8]>(&xv[0][0]);
                            tmem_ld_4x8(taddr + c0, taddr + c0 + 8, taddr + c0 + 16, taddr + c0 + 24, x8[0], x8[1], x8[2],
                                        x8[3]);
                        }
                        const float* pc = Ps + c0;
#pragma unroll
                        for (int g = 0; g < XG; ++g) {
#pragma unroll
                            for (int t4 = 0; t4 < 32; t4 += 4) {
                                float hv[4];
#pragma unroll
                                for (int u = 0; u < 4; ++u) hv[u] = silu_tanh(xv[g][t4 + u] + bj);
#pragma unroll
                                for (int jq = 0; jq < G; ++jq) {
                                    const float4 pw = *reinterpret_cast<const float4*>(pc + jq * kRows + g * 32 + t4);
                                    z[jq] = fmaf(pw.x, hv[0], z[jq]);
                                    z[jq] = fmaf(pw.y, hv[1], z[jq]);
                                    z[jq] = fmaf(pw.z, hv[2], z[jq]);
                                    z[jq] = fmaf(pw.w, hv[3], z[jq]);
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int jq = 0; jq < G; ++jq) Z[jq * M + jj] = z[jq];
                }
            }
            fence_before();
            mbar_arrive(&t_empty[buf]);   // the accumulator is read: the MMAs of item j + 2 may use it
            if (j + 2 < n_local) fetch_logits(it_begin + j + 2, nx_tok, nx_sv);

            // weighted residual rows, then the second layer on the chunk's hidden sums
            float acc[G];
#pragma unroll
            for (int jq = 0; jq < G; ++jq) acc[jq] = 0.0f;
            float rv[16];
            if (p.res.dtype == LOWRAM_INT8_VEC) {
#pragma unroll
                for (int k = 0; k < 16; ++k) rv[k] = (float)(int)rr[k] * __half2float(__ushort_as_half((unsigned short)rs[k]));
            } else {
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    rv[k] = p.res.dtype == LOWRAM_BF16 ? __uint_as_float(rr[k] << 16) : __uint_as_float(rr[k]);
            }
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                if (k < n_hit) {
                    const int t = HitSlot[k];
#pragma unroll
                    for (int jq = 0; jq < G; ++jq) acc[jq] = fmaf(Ps[jq * kRows + t], rv[k], acc[jq]);
                }
            }
            for (int k0 = 16; k0 < n_hit; k0 += 8) {    // more than 16 hits in the chunk
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int k = k0 + u;
                    v[u] = k < n_hit ? p.res.get(bh * p.n_res + HitRow[k], i_out) : 0.0f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int k = k0 + u;
                    if (k >= n_hit) break;
                    const int t = HitSlot[k];
#pragma unroll
                    for (int jq = 0; jq < G; ++jq) acc[jq] = fmaf(Ps[jq * kRows + t], v[u], acc[jq]);
                }
            }
            team_sync();   // every hidden sum is in Z
            if (have) {
                // the hidden sums as bf16 hi + lo: Zs[n][k] = hi(z[n][k]) for n < G, lo(z[n - G][k]) =
                // bf16(z - hi) for G <= n < 2G (hi + lo holds z to 2^-16), 0 beyond
                for (int e = et; e < NT * 8 * (M / 2); e += kTeam) {
                    const int n = e / (M / 2), k = (e - n * (M / 2)) * 2;
                    uint32_t packed = 0u;
                    if (n < 2 * G) {
                        const int jq = n < G ? n : n - G;
                        const float2 zz = *reinterpret_cast<const float2*>(Z + jq * M + k);
                        __nv_bfloat162 v = __floats2bfloat162_rn(zz.x, zz.y);
                        if (n >= G) {
                            const float2 hf = __bfloat1622float2(v);
                            v = __floats2bfloat162_rn(zz.x - hf.x, zz.y - hf.y);
                        }
                        packed = *reinterpret_cast<const uint32_t*>(&v);
                    }
                    *reinterpret_cast<uint32_t*>(Zs + n * (M + 8) + k) = packed;
                }
            }
            team_sync();
            if (have) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    uint32_t (&a)[KB][4] = af[AT == 2 ? mt : 0];
                    if (AT == 1) load_af(h, b, mt, a);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                        const __nv_bfloat16* zr = Zs + (nt * 8 + fg) * (M + 8) + 2 * ft;
#pragma unroll
                        for (int kb = 0; kb < KB; ++kb) {
                            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(zr + kb * 16);
                            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(zr + kb * 16 + 8);
                            mma_16816(d, a[kb][0], a[kb][1], a[kb][2], a[kb][3], b0, b1);
                        }
                        float* wo = Wo + (nt * 8 + 2 * ft) * kWoStride + 32 * q + 16 * mt + fg;
                        wo[0] = d[0];
                        wo[kWoStride] = d[1];
                        wo[8] = d[2];
                        wo[kWoStride + 8] = d[3];
                    }
                }
            }
            team_sync();
            float* rec = p.partial + (((int64_t)b * p.H_q + h * G) * p.n_chunks + chunk) * rw;
#pragma unroll
            for (int jq = 0; jq < G; ++jq)
                rec[jq * qstride + i_out] =
                    acc[jq] + (Wo[jq * kWoStride + i_out] + Wo[(G + jq) * kWoStride + i_out]) + chunk_sum(jq) * bias;
            if (i_out < G) {
                rec[i_out * qstride + 128] = chunk_max(i_out);
                rec[i_out * qstride + 129] = chunk_sum(i_out);
            }
        }
    }

    // ---------------------------------------------------------------------- teardown
    fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) flag(p.check, LOWRAM_CHECK_TIMEOUT);
    if (warp == 1) {
        fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

}  // namespace

bool tc_vregen_supported(const lowram_decode_shape& s) {
    return tc_score_supported(s) && (s.m == 128 || s.m == 256) && s.d == 128 && vregen_config(s.m, s.r, s.H_q / s.H_kv).NS >= 2;
}

int tc_partial_width(const lowram_decode_shape& s) { return s.d + 2; }


cudaError_t launch_vregen_tc(const DecodeArgs& a, cudaStream_t st) {
    const auto& s = a.s;
    VregenTcParams p{};
    p.B = s.B;
    p.T = s.T;
    p.H_q = s.H_q;
    p.H_kv = s.H_kv;
    p.m = s.m;
    p.r = s.r;
    p.coef = (const __nv_bfloat16*)a.coef;
    p.S_eff = a.S_eff;
    p.n_chunks = a.n_chunks;
    p.n_res = s.n_res;
    p.KC = s.r / 64;
    const VregenConfig cfg = vregen_config(s.m, s.r, s.H_q / s.H_kv);
    p.NS = cfg.NS;
    p.f_resident = cfg.f_resident ? 1 : 0;
    p.f_tmem = cfg.f_tmem ? 1 : 0;
    p.n_items = s.B * s.H_kv * a.n_chunks;
    const int copies = (s.basis_batch_stride || s.mlp_batch_stride) ? s.B : 1;
    p.fold_per_seq = copies > 1 ? 1 : 0;
    p.mlp_stride = s.mlp_batch_stride;
    const bool f16 = s.coef_dtype == kCoefF16;
    p.idesc = f16 ? tc::idesc_f16(128, 128) : tc::idesc_bf16(128, 128);
    p.wait_cycles = a.wait_cycles > 0 ? a.wait_cycles : tc::kWaitCycles;
    p.sall = a.sall;
    p.b1 = a.b1;
    p.b2 = a.b2;
    p.w2 = (const __nv_bfloat16*)a.w2;
    p.sel = a.sel;
    p.hit = a.hit;
    p.res = ResView{s.res_dtype, a.res_val, (const __half*)a.res_scale, s.d};
    p.partial = a.partial;
    p.check = a.check;
    if (p.n_items == 0) return cudaSuccess;
    if (!a.fold || cfg.NS < 2) return cudaErrorInvalidValue;
    CUtensorMap mF;
    const uint64_t dF[2] = {(uint64_t)s.r, (uint64_t)copies * s.H_kv * s.m};
    const uint32_t bF[2] = {64, 128};
    if (!tc::make_map(&mF, a.fold, 2, dF, bF, 0, f16)) return cudaErrorInvalidValue;
    const int grid = std::min(p.n_items, tc::sm_count());
    cudaError_t e = cudaSuccess;
    auto go = [&](auto kern) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.smem);
        if (e == cudaSuccess) e = launch_pdl(kern, dim3(grid), dim3(kVThreads), cfg.smem, st, mF, p);
    };
    const bool two = s.m == 256;
    switch (s.H_q / s.H_kv) {
        case 1: two ? go(vregen_tc_kernel<1, 2>) : go(vregen_tc_kernel<1, 1>); break;
        case 2: two ? go(vregen_tc_kernel<2, 2>) : go(vregen_tc_kernel<2, 1>); break;
        case 4: two ? go(vregen_tc_kernel<4, 2>) : go(vregen_tc_kernel<4, 1>); break;
        case 7: two ? go(vregen_tc_kernel<7, 2>) : go(vregen_tc_kernel<7, 1>); break;
        case 8: two ? go(vregen_tc_kernel<8, 2>) : go(vregen_tc_kernel<8, 1>); break;
        default: return cudaErrorNotSupported;
    }
    return e;
}

}  // namespace lowram
