// tc_evict.cu -- the window logits of the heavy-hitter eviction plan on the tensor cores (tcgen05), for bf16
// prompts: heavy hitters chosen from accumulated attention ("LowRAM: predict values from keys, store only the
// misses", Key points: sinks, recent tokens and heavy hitters are kept; "LowRAM Paper: Amortised Values and
// Low-Rank Keys for KV Compression", the quantisation / eviction composition).
//
// Per (sequence b, kv-head h) the logits of the W observation-window queries against the T prompt tokens are a
// dense product: L = Q_h K_h^T, Q_h [W*g x d] (the window query-heads of h, g = H_q / H_kv), K_h [T x d].  Both
// passes of the attention mass compute it tile by tile, 128 tokens and 128 query-heads at a time, with one
// tcgen05.mma chain (M = 128, N = 128, K = d) into a 128-column TMEM accumulator:
//   log-sum-exp pass  A = Q_h tile, B = K tile: TMEM lane = query-head, column = token, so each thread folds
//                     its query's logits over the tile's tokens into a running (max, sum of exp) and writes the
//                     pair once per chunk of tiles (the reduction kernel in evict.cu folds the chunks);
//   mass pass         A = K tile, B = Q_h tile: TMEM lane = token, column = query-head, so each thread sums
//                     exp(logit - lse) over its token's row; sums over kv-heads (and the two column halves)
//                     accumulate in shared memory.
// The window queries are first packed per kv-head, zero-padded to a multiple of 128 rows, so that one 2D TMA
// box is one operand tile.  K tiles come straight from the [B*T, H_kv, d] cache through a 3D TMA map (rows past
// the sequence's end are masked; past the cache's end TMA fills zeros).
//
// One CTA of 256 threads per (chunk of token tiles, b), two CTAs per SM.  Thread 0 issues the TMA loads and the
// MMAs; the next step's K tile is in flight (two stages) while the current step multiplies and all eight warps
// read TMEM: warp w takes lanes 32 (w % 4) .. + 31 and columns 64 (w / 4) .. + 63, so the two column halves of
// a row keep separate partial results, combined once per chunk through shared memory.  Exponentials are base 2
// on one fused multiply-add: exp(scale x - m) = 2^(x (scale log2 e) - m log2 e).  Every wait is bounded
// (tc_common.cuh): on a timeout the CTA sets LOWRAM_CHECK_TIMEOUT, waits for what it issued, frees TMEM and
// returns.
#include "evict.h"
#include "tc_common.cuh"

#include <algorithm>

namespace lowram {

namespace {

constexpr int kWThreads = 256;            // two warps per TMEM lane quarter, one per half of the columns
constexpr int kWTile = 128;               // tokens per K tile, query-heads per Q tile
constexpr int kWChunk = 16384;            // one 64-wide k-chunk of a 128-row tile, bf16, 128-byte swizzled
constexpr int kWMaxChunkTiles = 8;        // token tiles per CTA at most
constexpr int kWSmem = 1024 /* alignment */ + 2 * kWChunk /* Q */ + 4 * kWChunk /* K, two stages */ +
                       kWTile * 4 /* lse of the Q tile */ + 2 * kWMaxChunkTiles * kWTile * 4 /* token mass */ +
                       kWTile * 8 /* column-half exchange */ + 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x on the special-function unit (ex2.approx.ftz: relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// qp[(b*H_kv + h)*NQpad + n][:] = q_win[b, n / g, h*g + n % g, :] for n < NQ = W*g, zero rows up to NQpad.
__global__ void pack_window_kernel(const uint4* __restrict__ q, int B, int W, int H_q, int H_kv, int d, int NQpad,
                                   uint4* __restrict__ qp) {
    const int per_row = d / 8, g = H_q / H_kv, NQ = W * g;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * H_kv * NQpad * per_row) return;
    const int kk = (int)(i % per_row);
    const int64_t row = i / per_row;
    const int n = (int)(row % NQpad);
    const int64_t bh = row / NQpad;
    const int h = (int)(bh % H_kv), b = (int)(bh / H_kv);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < NQ) {
        const int iw = n / g, hq = h * g + (n - iw * g);
        v = __ldg(q + (((int64_t)b * W + iw) * H_q + hq) * per_row + kk);
    }
    qp[i] = v;
}

struct WindowTcParams {
    int T, W, H_q, H_kv, d, NQpad, chunk_tiles;
    float scale;
    float2* part;         // [B, n_chunks, W*H_q] (log-sum-exp pass)
    const float* lse;     // [B, W*H_q]           (mass pass)
    float* mass;          // [B, T]               (mass pass)
    uint32_t* check;
};

template <bool kMass>
__global__ void __launch_bounds__(kWThreads, 2)
    window_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     WindowTcParams p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* Qs = smem;                                        // [d/64][128 rows x 128 B]
    uint8_t* Ks = Qs + 2 * kWChunk;                            // [2 stages][d/64][128 rows x 128 B]
    float* lse_s = (float*)(Ks + 4 * kWChunk);                 // [128]
    float* mass_s = lse_s + kWTile;                            // [2 halves][chunk tiles][128]
    float2* xch = (float2*)(mass_s + 2 * kWMaxChunkTiles * kWTile);     // [128]
    uint64_t* kfull = (uint64_t*)(xch + kWTile);               // [2]
    uint64_t* qfull = kfull + 2;
    uint64_t* mdone = qfull + 1;
    uint32_t* tmem_slot = (uint32_t*)(mdone + 1);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
    if (layout_overflows(smem_raw, (const void*)(abort_flag + 1), p.check)) return;

    const int tid = threadIdx.x, warp = tid >> 5, row = tid & (kWTile - 1), half = warp >> 2;
    const int b = blockIdx.y, c = blockIdx.x;
    const int n_tiles = (int)cdiv(p.T, kWTile);
    const int tile_begin = c * p.chunk_tiles;
    const int ntl = min(p.chunk_tiles, n_tiles - tile_begin);
    const int g = p.H_q / p.H_kv, NQ = p.W * g, n_qc = p.NQpad / kWTile, KC = p.d / 64;
    const int S = p.H_kv * n_qc * ntl;
    const uint32_t kbytes = (uint32_t)KC * kWChunk;

    if (tid == 0) {
        mbar_init(&kfull[0], 1);
        mbar_init(&kfull[1], 1);
        mbar_init(qfull, 1);
        mbar_init(mdone, 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    if (kMass)
        for (int tl = 0; tl < ntl; ++tl) mass_s[(half * kWMaxChunkTiles + tl) * kWTile + row] = 0.0f;
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)half * 64;
    const float c2 = p.scale * kLog2e;       // logit in base-2 units per unit of q . k

    // thread 0's outstanding asynchronous work (and the phase parity each completes), for the drain after a
    // timeout
    bool k_out[2] = {false, false}, q_out = false, mma_out = false;
    uint32_t k_par[2] = {0u, 0u}, q_par = 0u, mma_par = 0u;

    // step i = (h * n_qc + qc) * ntl + tl
    auto step_h = [&](int i) { return i / (n_qc * ntl); };
    auto step_qc = [&](int i) { return (i / ntl) % n_qc; };
    auto step_tl = [&](int i) { return i % ntl; };
    auto issue_k = [&](int i) {
        const int s = i & 1, h = step_h(i);
        const int row = b * p.T + (tile_begin + step_tl(i)) * kWTile;
        mbar_expect_tx(&kfull[s], kbytes);
        for (int kc = 0; kc < KC; ++kc)
            tma_load_3d(Ks + (s * 2 + kc) * kWChunk, &tmK, &kfull[s], kc * 64, h, row);
        k_out[s] = true;
        k_par[s] = (uint32_t)(i >> 1) & 1u;
    };
    auto issue_q = [&](int i) {
        const int row = (b * p.H_kv + step_h(i)) * p.NQpad + step_qc(i) * kWTile;
        mbar_expect_tx(qfull, kbytes);
        for (int kc = 0; kc < KC; ++kc) tma_load_2d(Qs + kc * kWChunk, &tmQ, qfull, kc * 64, row);
        q_out = true;
        q_par = (uint32_t)(step_h(i) * n_qc + step_qc(i)) & 1u;
    };

    if (tid == 0 && S > 0) {
        issue_q(0);
        issue_k(0);
    }
    float run_m = -INFINITY, run_s = 0.0f;       // log-sum-exp pass: this thread's query and column half over
                                                 // the chunk, max in base-2 units
    bool aborted = false;
    for (int i = 0; i < S; ++i) {
        const int h = step_h(i), qc = step_qc(i), tl = step_tl(i);
        bool ok = true;
        if (tid == 0) {
            if (i + 1 < S) issue_k(i + 1);       // its stage was last read by step i-1's MMAs, which completed
            ok = mbar_wait(&kfull[i & 1], (i >> 1) & 1, abort_flag);
            if (ok) k_out[i & 1] = false;
            if (ok && tl == 0) {
                ok = mbar_wait(qfull, (h * n_qc + qc) & 1, abort_flag);
                if (ok) q_out = false;
            }
            if (ok) {
                fence_after();
                const uint32_t kb = smem_u32(Ks + (i & 1) * 2 * kWChunk), qb = smem_u32(Qs);
                const uint32_t idesc = idesc_bf16(kWTile, kWTile);
                for (int kc = 0; kc < KC; ++kc)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t ka = kb + kc * kWChunk + k * 32, qa = qb + kc * kWChunk + k * 32;
                        mma_bf16(tmem, sdesc_sw128(kMass ? ka : qa), sdesc_sw128(kMass ? qa : ka), idesc,
                                 (kc | k) != 0);
                    }
                mma_commit(mdone);
                mma_out = true;
                mma_par = (uint32_t)i & 1u;
            }
        }
        if (kMass && tl == 0 && tid < kWTile) {
            const int n = qc * kWTile + tid;
            float v = INFINITY;                  // padding query-heads: 2^(x c2 - inf) = 0
            if (n < NQ) {
                const int iw = n / g, hq = h * g + (n - iw * g);
                v = p.lse[((int64_t)b * p.W + iw) * p.H_q + hq] * kLog2e;
            }
            lse_s[tid] = v;
        }
        if (!__syncthreads_and(ok)) {
            aborted = true;
            break;
        }
        ok = mbar_wait(mdone, i & 1, abort_flag);
        if (!__syncthreads_and(ok)) {
            aborted = true;
            break;
        }
        if (tid == 0) mma_out = false;
        fence_after();
        if (tid == 0 && tl == ntl - 1 && i + 1 < S) issue_q(i + 1);   // step i's MMAs, Qs's last readers, are done
        const int t0 = (tile_begin + tl) * kWTile;
        const int nvalid = min(kWTile, p.T - t0);
        if (!kMass) {
            // lane = query-head qc*128 + row, columns = tokens half*64 .. half*64 + 63 of the tile
            const int cv = nvalid - half * 64;   // valid columns of this half
            float x[32], y[32];
            tmem_ld_2x32(taddr, taddr + 32, x, y);
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j < cv) mx = fmaxf(mx, x[j]);
                if (32 + j < cv) mx = fmaxf(mx, y[j]);
            }
            if (cv > 0) {
                const float m2 = mx * c2;        // scale > 0: the largest scaled logit, base 2
                float s = 0.0f;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if (j < cv) s += ex2(fmaf(x[j], c2, -m2));
                    if (32 + j < cv) s += ex2(fmaf(y[j], c2, -m2));
                }
                const float M = fmaxf(run_m, m2);
                run_s = (run_m == -INFINITY ? 0.0f : run_s * ex2(run_m - M)) + s * ex2(m2 - M);
                run_m = M;
            }
            if (tl == ntl - 1) {
                // the column halves of each query-head meet; the pair goes out in natural-log units
                if (half == 1) xch[row] = make_float2(run_m, run_s);
                __syncthreads();
                if (half == 0) {
                    const float2 o = xch[row];
                    const float M = fmaxf(run_m, o.x);
                    if (M != -INFINITY) {
                        run_s = (run_m == -INFINITY ? 0.0f : run_s * ex2(run_m - M)) +
                                (o.x == -INFINITY ? 0.0f : o.y * ex2(o.x - M));
                        run_m = M;
                    }
                    const int n = qc * kWTile + row;
                    if (n < NQ) {
                        const int iw = n / g, hq = h * g + (n - iw * g);
                        p.part[((int64_t)b * gridDim.x + c) * ((int64_t)p.W * p.H_q) + (int64_t)iw * p.H_q + hq] =
                            make_float2(run_m * kLn2, run_s);
                    }
                }
                run_m = -INFINITY;
                run_s = 0.0f;
            }
        } else {
            // lane = token t0 + row, columns = query-heads qc*128 + half*64 .. + 63
            float x[32], y[32];
            tmem_ld_2x32(taddr, taddr + 32, x, y);
            const float* ls = lse_s + half * 64;
            float acc = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                acc += ex2(fmaf(x[j], c2, -ls[j]));
                acc += ex2(fmaf(y[j], c2, -ls[32 + j]));
            }
            mass_s[(half * kWMaxChunkTiles + tl) * kWTile + row] += acc;
        }
        fence_before();
        __syncthreads();                          // TMEM and lse_s are read before the next step overwrites them
    }

    if (aborted && tid == 0) {
        for (int s = 0; s < 2; ++s)
            if (k_out[s]) mbar_wait_drain(&kfull[s], k_par[s]);
        if (q_out) mbar_wait_drain(qfull, q_par);
        if (mma_out) mbar_wait_drain(mdone, mma_par);
        flag(p.check, LOWRAM_CHECK_TIMEOUT);
    }
    if (kMass && !aborted && tid < kWTile)       // the last step's closing barrier ordered every half's sums
        for (int tl = 0; tl < ntl; ++tl) {
            const int t = (tile_begin + tl) * kWTile + tid;
            if (t < p.T)
                p.mass[(int64_t)b * p.T + t] = mass_s[tl * kWTile + tid] + mass_s[(kWMaxChunkTiles + tl) * kWTile + tid];
        }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, 128);
    }
}

}  // namespace

int window_tc_chunk_tiles(int B, int T) {
    const int64_t tiles = (int64_t)B * cdiv(T, kWTile);
    return (int)std::min<int64_t>(kWMaxChunkTiles, std::max<int64_t>(1, cdiv(tiles, 2 * 148)));
}

int window_tc_n_chunks(int B, int T) { return T > 0 ? (int)cdiv(cdiv(T, kWTile), window_tc_chunk_tiles(B, T)) : 0; }

int window_tc_qpad(int W, int H_q, int H_kv) { return (int)cdiv((int64_t)W * (H_q / H_kv), kWTile) * kWTile; }

cudaError_t launch_pack_window(int B, int W, int H_q, int H_kv, int d, const void* q_win, void* qp, cudaStream_t st) {
    const int NQpad = window_tc_qpad(W, H_q, H_kv);
    const int64_t n = (int64_t)B * H_kv * NQpad * (d / 8);
    if (n == 0) return cudaSuccess;
    pack_window_kernel<<<(unsigned)cdiv(n, 256), 256, 0, st>>>((const uint4*)q_win, B, W, H_q, H_kv, d, NQpad,
                                                               (uint4*)qp);
    return cudaGetLastError();
}

cudaError_t launch_window_tc(bool mass_pass, int B, int T, int W, int H_q, int H_kv, int d, float scale,
                             const void* qp, const void* k, float2* part, const float* lse, float* mass,
                             uint32_t* check, cudaStream_t st) {
    if ((int64_t)B * T == 0) return cudaSuccess;
    WindowTcParams p;
    p.T = T;
    p.W = W;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.d = d;
    p.NQpad = window_tc_qpad(W, H_q, H_kv);
    p.chunk_tiles = window_tc_chunk_tiles(B, T);
    p.scale = scale;
    p.part = part;
    p.lse = lse;
    p.mass = mass;
    p.check = check;
    CUtensorMap mQ, mK;
    const uint64_t dQ[2] = {(uint64_t)d, (uint64_t)B * H_kv * p.NQpad};
    const uint32_t bQ[2] = {64, (uint32_t)kWTile};
    const uint64_t dK[3] = {(uint64_t)d, (uint64_t)H_kv, (uint64_t)B * T};
    const uint32_t bK[3] = {64, 1, (uint32_t)kWTile};
    if (!tc::make_map(&mQ, qp, 2, dQ, bQ) || !tc::make_map(&mK, k, 3, dK, bK)) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)window_tc_n_chunks(B, T), (unsigned)B);
    cudaError_t e;
    if (mass_pass) {
        e = cudaFuncSetAttribute(window_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmem);
        if (e == cudaSuccess) window_tc_kernel<true><<<grid, kWThreads, kWSmem, st>>>(mQ, mK, p);
    } else {
        e = cudaFuncSetAttribute(window_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmem);
        if (e == cudaSuccess) window_tc_kernel<false><<<grid, kWThreads, kWSmem, st>>>(mQ, mK, p);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace lowram
