// tc_vregen.cu -- tensor-core (tcgen05) value regeneration for the selected tokens of bf16 caches (K3), and
// the merge of its softmax partials (K4).
//
// The method: each decode step rebuilds only a selected subset of KV pairs (LowRAM abstract); a selected
// token's value is predicted from its pre-RoPE key by the head's MLP, plus the stored residual when the
// token is one of the worst-predicted ("Value cache amortisation in plain language", LowRAM Paper:
// Amortised Values and Low-Rank Keys for KV Compression; flowchart "Values are mostly a function of keys"
// of the wiki page).  The key itself comes from the low-rank factors ("Asymmetric key compression with
// xKV").
//
// K3, one CTA per (sequence b, kv-head h, chunk of 128 selected tokens), 192 threads:
//   warp 0      TMA producer: the basis rows of head h [128 x r] in 64-wide k-chunks through an NS-stage
//               ring, and the head's first predictor layer w1[h] [m x d] (resident).
//   warp 1      TMEM owner and MMA issuer (one thread):
//                 MMA1  D1[128 tok x 128] = C_sel . basis_h^T   (M=128, N=128, K=r): pre-RoPE keys
//                 MMA2  D2[m x 128 tok]   = w1_h . K^T          (M=128 per 128 hidden units, N=128, K=d)
//               MMA2 runs transposed (hidden units on TMEM lanes, tokens on columns), so the softmax-weighted
//               sum over tokens is a loop over one thread's own TMEM row.
//   warps 2-5   gather + epilogue: cp.async of the selected latent rows into the 128B-swizzled operand
//               layout; D1 -> bf16 keys in shared memory (MMA2's B operand); softmax weights of the chunk
//               from the scaled logits the key pass stored; SiLU of D2 and the weighted sums
//               z[jq] = sum_t p[jq,t] SiLU(w1 k_t + b1); weighted sums of the chunk's residual rows.
// The second predictor layer is linear, so sum_t p_t (w2 h_t + b2 + r_t) = w2 (sum_t p_t h_t) + b2 sum_t p_t
// + sum_t p_t r_t: the merge kernel applies w2 and b2 once per (sequence, q-head) to the merged sums instead
// of once per selected token.  Values are never materialised; the result is the same up to rounding order.
//
// Every wait is bounded (tc_common.cuh).  On a timeout the kernel sets LOWRAM_CHECK_TIMEOUT, lets what it
// issued complete, frees TMEM and returns; every named barrier is reached on every path.
#include "kernels.h"
#include "predict.cuh"
#include "tc_common.cuh"

namespace lowram {

namespace {

constexpr int kVThreads = 192;
constexpr int kRows = 128;              // selected tokens per CTA
constexpr int kStageBytes = 32768;      // latent chunk [128 x 64] + basis chunk [128 x 64], bf16
constexpr int kHalf = 16384;
constexpr int kNS = 3;                  // ring stages; after MMA1 the ring holds the keys and w1[h]

struct VregenTcParams {
    int T, H_q, H_kv, r, m, S_eff, n_chunks, n_res, KC, PW;
    const __nv_bfloat16* coef;
    const float* sall;        // [B, H_q, T] scaled logits written by the key pass
    const float* b1;          // [H_kv, m] or null
    const float* b2;          // [H_kv, d] or null
    const __nv_bfloat16* w2;  // [H_kv, d, m]
    const int32_t* sel;       // [B, H_kv, S_eff]
    const int32_t* hit;       // [B, H_kv, S_eff] residual row of each selected token, or -1
    ResView res;
    float* partial;           // [B, H_q, n_chunks, PW]
    int32_t* cnt;             // [B, H_kv] chunks finished per (b, h); zeroed by the selection kernel
    float* out;               // [B, H_q, d]
    float* lse;               // [B, H_q] or null
    uint32_t* check;
};

size_t vregen_smem_bytes() {
    return 1024 + (size_t)kNS * kStageBytes + 8 * 128 * 4 + 3 * 128 * 4 + 72 * 4 + 8 * (3 * kNS + 5) + 16;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_16(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(tc::smem_u32(p)), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// The last CTA of a (sequence, kv-head) to finish merges the chunks' partials of its G q-heads (threads =
// the 128 epilogue threads, et = 0..127): W = max_c M_c, w_c = exp(M_c - W), L = sum_c w_c l_c,
// out = w2[h] (sum_c w_c z_c / L) + b2[h] + sum_c w_c rz_c / L,  lse = W + log L.
// It is the tail of the kernel's last wave, so its global reads are issued together: the thread's row of w2
// (output feature i = et) first, then the G q-heads' contiguous records in batches of 10 independent 16-byte
// loads (all G at once when they fit, else one q-head at a time); the chunk weights w_c are computed once per
// q-head.
template <int G>
__device__ __forceinline__ void merge_last(const VregenTcParams& p, int b, int h, int et, float* scratch) {
    const int64_t qstride = (int64_t)p.n_chunks * p.PW;
    const float* P0 = p.partial + ((int64_t)b * p.H_q + h * G) * qstride;
    const int ZW = p.m + 128;
    float* Z = scratch;                          // [G][m + 128] merged hidden sums, then residual sums
    float* Wc = Z + G * ZW;                      // [G][n_chunks] chunk weights exp(M_c - W)
    float* ML = Wc + G * p.n_chunks;             // [G][2] W and L
    float* Pb = ML + 2 * G;                      // [G][n_chunks][PW] staged records (16-byte aligned: see below)
    Pb = (float*)(((uintptr_t)Pb + 15) & ~(uintptr_t)15);
    // all G q-heads' records at once when they fit, else one q-head at a time (tc_fused_merge guarantees one fits)
    const size_t fixed = (size_t)(Pb - scratch) * sizeof(float);
    const int per = (fixed + G * qstride * sizeof(float) <= (size_t)kNS * kStageBytes) ? G : 1;

    constexpr int kW2Pre = 16;                   // 16-byte pieces of the w2 row fetched ahead (128 hidden units)
    constexpr int kRecBatch = 10;                // independent 16-byte record loads per thread per batch
    const uint4* W2r = reinterpret_cast<const uint4*>(p.w2 + ((int64_t)h * 128 + et) * p.m);
    uint4 wpre[kW2Pre];
#pragma unroll
    for (int u = 0; u < kW2Pre; ++u)
        if (u * 8 < p.m) wpre[u] = __ldg(W2r + u);

    for (int q0 = 0; q0 < G; q0 += per) {
        {   // records of q-heads q0 .. q0+per-1
            const float4* src = reinterpret_cast<const float4*>(P0 + q0 * qstride);
            float4* d4 = reinterpret_cast<float4*>(Pb);
            const int n4 = (int)(per * qstride / 4);
            for (int i0 = 0; i0 < n4; i0 += kRecBatch * kRows) {
                float4 v[kRecBatch];
#pragma unroll
                for (int u = 0; u < kRecBatch; ++u) {
                    const int i = i0 + u * kRows + et;
                    if (i < n4) v[u] = __ldcg(src + i);
                }
#pragma unroll
                for (int u = 0; u < kRecBatch; ++u) {
                    const int i = i0 + u * kRows + et;
                    if (i < n4) d4[i] = v[u];
                }
            }
            tc::named_bar_sync(1, kRows);
        }
        // one thread per q-head: W, L and the chunk weights
        if (et < per) {
            const int jq = q0 + et;
            const float* Pq = Pb + et * qstride;
            float mx = -INFINITY;
            for (int c = 0; c < p.n_chunks; ++c) mx = fmaxf(mx, Pq[(int64_t)c * p.PW + p.m + 128]);
            float l = 0.0f;
            for (int c = 0; c < p.n_chunks; ++c) {
                const float mc = Pq[(int64_t)c * p.PW + p.m + 128];
                const float w = mc == -INFINITY ? 0.0f : __expf(mc - mx);
                Wc[jq * p.n_chunks + c] = w;
                l = fmaf(w, Pq[(int64_t)c * p.PW + p.m + 129], l);
            }
            ML[jq * 2] = mx;
            ML[jq * 2 + 1] = l;
        }
        tc::named_bar_sync(1, kRows);
        for (int e = et; e < per * ZW; e += kRows) {
            const int jl = e / ZW, j = e - jl * ZW, jq = q0 + jl;
            const float* Pq = Pb + jl * qstride;
            const float l = ML[jq * 2 + 1];
            float acc = 0.0f;
            for (int c = 0; c < p.n_chunks; ++c) acc = fmaf(Wc[jq * p.n_chunks + c], Pq[(int64_t)c * p.PW + j], acc);
            Z[jq * ZW + j] = l > 0.0f ? acc / l : 0.0f;
        }
        tc::named_bar_sync(1, kRows);     // Pb is reused by the next group of q-heads; Z is complete
    }
    // thread et = output feature i: the second predictor layer on the merged hidden sums
    float acc[G];
#pragma unroll
    for (int jq = 0; jq < G; ++jq) acc[jq] = 0.0f;
    for (int j0 = 0; j0 < p.m; j0 += 8 * kW2Pre) {
#pragma unroll
        for (int u = 0; u < kW2Pre; ++u) {
            const int jb = j0 + u * 8;
            if (jb >= p.m) break;
            const uint4 wv = j0 == 0 ? wpre[u] : __ldg(W2r + jb / 8);
            const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&wv);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(pr[e]);
                const int j = jb + 2 * e;
#pragma unroll
                for (int jq = 0; jq < G; ++jq) {
                    acc[jq] = fmaf(f.x, Z[jq * ZW + j], acc[jq]);
                    acc[jq] = fmaf(f.y, Z[jq * ZW + j + 1], acc[jq]);
                }
            }
        }
    }
    const float bias = p.b2 ? __ldg(p.b2 + (int64_t)h * 128 + et) : 0.0f;
#pragma unroll
    for (int jq = 0; jq < G; ++jq) {
        const int64_t bhq = (int64_t)b * p.H_q + h * G + jq;
        const float Mq = ML[jq * 2], Lq = ML[jq * 2 + 1];
        p.out[bhq * 128 + et] = Lq > 0.0f ? acc[jq] + bias + Z[jq * ZW + p.m + et] : 0.0f;
        if (p.lse && et == jq) p.lse[bhq] = Lq > 0.0f ? Mq + logf(Lq) : -INFINITY;
    }
}

template <int G>
__global__ void __launch_bounds__(kVThreads, 2)
    vregen_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW1,
                     VregenTcParams p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* ring = smem;                        // MMA1: stages; then keys [0, 32K) and w1[h] [32K, 32K + m*256)
    uint8_t* W1s = ring + 2 * kHalf;
    float* Ps = (float*)(ring + kNS * kStageBytes);   // [G][128] softmax weights of the chunk
    int* Tok = (int*)(Ps + 8 * kRows);           // token of each slot, -1 past the selection
    int* Hit = Tok + kRows;                      // compacted: residual rows of the chunk's slots that have one
    int* HitSlot = Hit + kRows;                  // ... and those slots, ascending
    float* red = (float*)(HitSlot + kRows);      // [2][4 warps][8] partial max / sum, then 4 hit counts
    uint64_t* fullA = (uint64_t*)(red + 72);
    uint64_t* fullB = fullA + kNS;
    uint64_t* empty = fullB + kNS;
    uint64_t* w1_full = empty + kNS;
    uint64_t* d1_full = w1_full + 1;
    uint64_t* kbf_full = d1_full + 1;
    uint64_t* d2_full = kbf_full + 1;
    uint64_t* m_drain = d2_full + 1;
    uint32_t* tmem_slot = (uint32_t*)(m_drain + 1);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
    volatile int* last_flag = (volatile int*)(tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int64_t bh = (int64_t)b * p.H_kv + h;
    const uint32_t tcols = p.m > 128 ? 256u : 128u;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&fullA[s], kRows);
            mbar_init(&fullB[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(w1_full, 1);
        mbar_init(d1_full, 1);
        mbar_init(kbf_full, kRows);
        mbar_init(d2_full, 1);
        mbar_init(m_drain, 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmW1);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tcols);
        tmem_relinquish();
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dep_wait();     // selection, residual rows and logits come from the kernels before (launch_pdl)

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            bool w1_issued = false;
            for (int kc = 0; kc < p.KC; ++kc) {
                const int s = kc % kNS, n = kc / kNS;
                if (!mbar_wait(&empty[s], (n & 1) ^ 1, abort_flag)) break;
                mbar_expect_tx(&fullB[s], kHalf);
                tma_load_2d(ring + s * kStageBytes + kHalf, &tmW, &fullB[s], kc * 64, h * 128);
                ++issued;
            }
            // w1[h] goes into the ring once MMA1 is complete
            if (issued == p.KC && mbar_wait(d1_full, 0, abort_flag)) {
                mbar_expect_tx(w1_full, (uint32_t)p.m * 256u);
                for (int mb = 0; mb < p.m / 128; ++mb)
                    for (int kc2 = 0; kc2 < 2; ++kc2)
                        tma_load_2d(W1s + (mb * 2 + kc2) * kHalf, &tmW1, w1_full, kc2 * 64, h * p.m + mb * 128);
                w1_issued = true;
            }
            if (*abort_flag) {
                // loads older than the last kNS were consumed by MMAs, so they have landed
                for (int k = issued > kNS ? issued - kNS : 0; k < issued; ++k)
                    mbar_wait_drain(&fullB[k % kNS], (k / kNS) & 1);
                if (w1_issued) mbar_wait_drain(w1_full, 0);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, 128);
            bool ok = true;
            for (int kc = 0; kc < p.KC && ok; ++kc) {
                const int s = kc % kNS, n = kc / kNS;
                if (!mbar_wait(&fullB[s], n & 1, abort_flag) || !mbar_wait(&fullA[s], n & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t a = smem_u32(ring + s * kStageBytes), bb = a + kHalf;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem, sdesc_sw128(a + k * 32), sdesc_sw128(bb + k * 32), idesc, (kc | k) != 0);
                mma_commit(&empty[s]);
            }
            if (ok) {
                mma_commit(d1_full);
                if (mbar_wait(kbf_full, 0, abort_flag) && mbar_wait(w1_full, 0, abort_flag)) {
                    fence_after();
                    const uint32_t kb = smem_u32(ring);
                    for (int mb = 0; mb < p.m / 128; ++mb)
                        for (int kc2 = 0; kc2 < 2; ++kc2) {
                            const uint32_t a = smem_u32(W1s + (mb * 2 + kc2) * kHalf), bb = kb + kc2 * kHalf;
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_bf16(tmem + mb * 128, sdesc_sw128(a + k * 32), sdesc_sw128(bb + k * 32), idesc,
                                         (kc2 | k) != 0);
                        }
                    mma_commit(d2_full);
                }
            }
            // every MMA issued completes before TMEM is released
            mma_commit(m_drain);
            mbar_wait_drain(m_drain, 0);
        }
    } else {
        // ------------------------------------------------------------------ gather + epilogue
        const int et = threadIdx.x - 64;
        const int quarter = warp & 3;
        const int slot = quarter * 32 + lane;   // the TMEM lane (row) this thread reads
        int my_tok, my_hit;
        {
            const int j = chunk * kRows + slot;
            int tok = j < p.S_eff ? p.sel[bh * p.S_eff + j] : -1;
            if (tok >= p.T) tok = p.T - 1;      // the selection is always in range; keep the invariant explicit
            my_hit = (j < p.S_eff && p.hit && p.n_res > 0) ? p.hit[bh * p.S_eff + j] : -1;
            Tok[slot] = tok;
            my_tok = tok;
        }
        named_bar_sync(1, kRows);

        // gather the selected latent rows: 8 threads per 128-byte row segment, 16 rows per pass
        bool ok = true;
        {
            const int c16 = et & 7, rsub = et >> 3;
            for (int kc = 0; kc < p.KC; ++kc) {
                const int s = kc % kNS, n = kc / kNS;
                if (ok && !mbar_wait(&empty[s], (n & 1) ^ 1, abort_flag)) ok = false;
                if (ok) {
                    const uint32_t A = smem_u32(ring + s * kStageBytes);
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) {
                        const int row = rr * 16 + rsub;
                        const int tok = Tok[row];
                        const __nv_bfloat16* src =
                            p.coef + ((int64_t)b * p.T + (tok >= 0 ? tok : 0)) * p.r + kc * 64 + c16 * 8;
                        cp_async_16(A + row * 128 + ((c16 ^ (row & 7)) << 4), src, tok >= 0 ? 16u : 0u);
                    }
                }
                cp_async_commit();
                // up to kNS - 1 stages of gathers stay in flight; stage kc - (kNS - 1) has landed
                if (kc >= kNS - 1) {
                    cp_async_wait<kNS - 1>();
                    fence_proxy_async();
                    if (ok) mbar_arrive(&fullA[(kc - (kNS - 1)) % kNS]);
                }
            }
            cp_async_wait<0>();
            fence_proxy_async();
            if (ok)
                for (int kc = (p.KC > kNS - 1 ? p.KC - (kNS - 1) : 0); kc < p.KC; ++kc) mbar_arrive(&fullA[kc % kNS]);
        }

        // while MMA1 finishes: the scaled logits of this slot's token
        float sv[G];
#pragma unroll
        for (int jq = 0; jq < G; ++jq)
            sv[jq] = my_tok >= 0 ? __ldg(p.sall + ((int64_t)b * p.H_q + h * G + jq) * p.T + my_tok) : -INFINITY;

        // D1 -> bf16 pre-RoPE keys, K-major and swizzled, into the ring's first 32 KB (MMA1 is complete)
        bool have = ok && mbar_wait(d1_full, 0, abort_flag);
        if (have) {
            fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                float x[32], y[32];
                tmem_ld_2x32(taddr + c * 64, taddr + c * 64 + 32, x, y);
                uint8_t* row = ring + c * kHalf + slot * 128;
#pragma unroll
                for (int sg = 0; sg < 4; ++sg) {
                    st_shared_16(row + ((sg ^ (slot & 7)) << 4), pack_bf16x2(x[sg * 8], x[sg * 8 + 1]),
                                 pack_bf16x2(x[sg * 8 + 2], x[sg * 8 + 3]), pack_bf16x2(x[sg * 8 + 4], x[sg * 8 + 5]),
                                 pack_bf16x2(x[sg * 8 + 6], x[sg * 8 + 7]));
                    st_shared_16(row + (((sg + 4) ^ (slot & 7)) << 4), pack_bf16x2(y[sg * 8], y[sg * 8 + 1]),
                                 pack_bf16x2(y[sg * 8 + 2], y[sg * 8 + 3]), pack_bf16x2(y[sg * 8 + 4], y[sg * 8 + 5]),
                                 pack_bf16x2(y[sg * 8 + 6], y[sg * 8 + 7]));
                }
            }
        }
        fence_proxy_async();
        fence_before();
        mbar_arrive(kbf_full);

        // softmax weights of the chunk per q-head
        float M[G], l[G];
#pragma unroll
        for (int jq = 0; jq < G; ++jq) {
            const float mx = warp_max(sv[jq]);
            if (lane == 0) red[quarter * 8 + jq] = mx;
        }
        const unsigned hb = __ballot_sync(0xffffffffu, my_hit >= 0);
        int* hcount = (int*)(red + 64);
        if (lane == 0) hcount[quarter] = __popc(hb);
        named_bar_sync(1, kRows);
        int n_hit;
        {
            int before = 0;
            for (int w = 0; w < quarter; ++w) before += hcount[w];
            n_hit = hcount[0] + hcount[1] + hcount[2] + hcount[3];
            if (my_hit >= 0) {
                const int at = before + __popc(hb & ((1u << lane) - 1u));
                Hit[at] = my_hit;
                HitSlot[at] = slot;
            }
        }
#pragma unroll
        for (int jq = 0; jq < G; ++jq) {
            M[jq] = fmaxf(fmaxf(red[jq], red[8 + jq]), fmaxf(red[16 + jq], red[24 + jq]));
            const float pv = (sv[jq] == -INFINITY || M[jq] == -INFINITY) ? 0.0f : __expf(sv[jq] - M[jq]);
            Ps[jq * kRows + slot] = pv;
            const float ps = warp_sum(pv);
            if (lane == 0) red[32 + quarter * 8 + jq] = ps;
        }
        named_bar_sync(1, kRows);
#pragma unroll
        for (int jq = 0; jq < G; ++jq) l[jq] = (red[32 + jq] + red[40 + jq]) + (red[48 + jq] + red[56 + jq]);

        float* dst = p.partial + (((int64_t)b * p.H_q + h * G) * p.n_chunks + chunk) * p.PW;
        const int64_t jq_stride = (int64_t)p.n_chunks * p.PW;

        // residual rows of the chunk, weighted: thread = feature
        {
            float rz[G];
#pragma unroll
            for (int jq = 0; jq < G; ++jq) rz[jq] = 0.0f;
            for (int k0 = 0; k0 < n_hit; k0 += 16) {    // 16 independent row loads in flight
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) v[u] = k0 + u < n_hit ? p.res.get(bh * p.n_res + Hit[k0 + u], slot) : 0.0f;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    if (k0 + u >= n_hit) break;
                    const int t = HitSlot[k0 + u];
#pragma unroll
                    for (int jq = 0; jq < G; ++jq) rz[jq] = fmaf(Ps[jq * kRows + t], v[u], rz[jq]);
                }
            }
#pragma unroll
            for (int jq = 0; jq < G; ++jq) dst[jq * jq_stride + p.m + slot] = rz[jq];
#pragma unroll
            for (int jq = 0; jq < G; ++jq)
                if (slot == jq) {
                    dst[jq * jq_stride + p.m + 128] = M[jq];
                    dst[jq * jq_stride + p.m + 129] = l[jq];
                }
        }

        // hidden units: thread = unit j of each 128-block; z[jq] = sum_t p[jq,t] SiLU(D2[j,t] + b1[j])
        have = have && mbar_wait(d2_full, 0, abort_flag);
        if (have) {
            fence_after();
#pragma unroll 1
            for (int mb = 0; mb < p.m / 128; ++mb) {
                const int j = mb * 128 + slot;
                const float bj = p.b1 ? __ldg(p.b1 + (int64_t)h * p.m + j) : 0.0f;
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + mb * 128;
                float z[G];
#pragma unroll
                for (int jq = 0; jq < G; ++jq) z[jq] = 0.0f;
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    float x[32], y[32];
                    tmem_ld_2x32(taddr + c * 64, taddr + c * 64 + 32, x, y);
#pragma unroll
                    for (int tt = 0; tt < 32; tt += 4) {
                        float hx[4], hy[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            hx[u] = silu_fast(x[tt + u] + bj);
                            hy[u] = silu_fast(y[tt + u] + bj);
                        }
#pragma unroll
                        for (int jq = 0; jq < G; ++jq) {
                            const float4 px = *reinterpret_cast<const float4*>(Ps + jq * kRows + c * 64 + tt);
                            const float4 py = *reinterpret_cast<const float4*>(Ps + jq * kRows + c * 64 + 32 + tt);
                            z[jq] = fmaf(px.x, hx[0], z[jq]);
                            z[jq] = fmaf(px.y, hx[1], z[jq]);
                            z[jq] = fmaf(px.z, hx[2], z[jq]);
                            z[jq] = fmaf(px.w, hx[3], z[jq]);
                            z[jq] = fmaf(py.x, hy[0], z[jq]);
                            z[jq] = fmaf(py.y, hy[1], z[jq]);
                            z[jq] = fmaf(py.z, hy[2], z[jq]);
                            z[jq] = fmaf(py.w, hy[3], z[jq]);
                        }
                    }
                }
#pragma unroll
                for (int jq = 0; jq < G; ++jq) dst[jq * jq_stride + j] = z[jq];
            }
        }

        // the last CTA of this (b, h) to finish merges the chunks (partials made visible device-wide first);
        // without a counter array the separate merge kernel does it
        __threadfence();
        fence_before();
        named_bar_sync(1, kRows);
        if (et == 0 && p.cnt) *last_flag = (atomicAdd(p.cnt + bh, 1) == p.n_chunks - 1) ? 1 : 0;
        named_bar_sync(1, kRows);
        if (*last_flag) {
            __threadfence();
            // the ring is free: MMA2 has completed (or the call has aborted and its results are void)
            merge_last<G>(p, b, h, et, (float*)ring);
            if (et == 0) p.cnt[bh] = 0;
        }
    }

    // ---------------------------------------------------------------------- teardown
    fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) flag(p.check, LOWRAM_CHECK_TIMEOUT);
    if (warp == 1) {
        fence_after();
        tmem_dealloc(tmem, tcols);
    }
}

// ------------------------------------------------------------------------------------------------
// K4 for the tensor-core path: merge the chunks' partials of one (sequence, q-head), then apply the
// predictor's second layer and bias to the merged hidden-unit sums:
//   W = max_c M_c, w_c = exp(M_c - W), L = sum_c w_c l_c,
//   out = w2[h] (sum_c w_c z_c / L) + b2[h] + sum_c w_c rz_c / L,  lse = W + log L.
// One CTA of 128 threads per (sequence, q-head).
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float block_reduce_128(float v, float* red, bool is_max) {
    v = is_max ? warp_max(v) : warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = is_max ? fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])) : (red[0] + red[1]) + (red[2] + red[3]);
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(128) merge_w2_kernel(int H_q, int G, int n_chunks, int m, int PW,
                                                       const float* __restrict__ partial,
                                                       const __nv_bfloat16* __restrict__ w2,
                                                       const float* __restrict__ b2, float* __restrict__ out,
                                                       float* __restrict__ lse) {
    extern __shared__ float msm[];
    __shared__ float red[4];
    float* wts = msm;               // [n_chunks]
    float* zb = msm + n_chunks;     // [m + 128]: merged hidden sums, then merged residual sums
    const int bhq = blockIdx.x, h = (bhq % H_q) / G, tid = threadIdx.x;
    const float* P = partial + (int64_t)bhq * n_chunks * PW;
    float M = -INFINITY;
    for (int c = tid; c < n_chunks; c += 128) M = fmaxf(M, P[(int64_t)c * PW + m + 128]);
    M = block_reduce_128(M, red, true);
    float L = 0.0f;
    for (int c = tid; c < n_chunks; c += 128) {
        const float mc = P[(int64_t)c * PW + m + 128];
        const float w = (mc == -INFINITY) ? 0.0f : __expf(mc - M);
        wts[c] = w;
        L = fmaf(w, P[(int64_t)c * PW + m + 129], L);
    }
    L = block_reduce_128(L, red, false);
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    for (int j = tid; j < m + 128; j += 128) {
        float acc = 0.0f;
        for (int c = 0; c < n_chunks; ++c) acc = fmaf(wts[c], P[(int64_t)c * PW + j], acc);
        zb[j] = acc * inv;
    }
    __syncthreads();
    // thread i: out[i] = w2[h][i, :] . zbar; the row's 16-byte pieces are independent loads
    const __nv_bfloat16* W2 = w2 + ((int64_t)h * 128 + tid) * m;
    float acc = 0.0f;
    for (int j0 = 0; j0 < m; j0 += 64) {
        uint4 wv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) wv[u] = __ldg(reinterpret_cast<const uint4*>(W2 + j0 + u * 8));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&wv[u]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(pr[e]);
                acc = fmaf(f.x, zb[j0 + u * 8 + 2 * e], acc);
                acc = fmaf(f.y, zb[j0 + u * 8 + 2 * e + 1], acc);
            }
        }
    }
    out[(int64_t)bhq * 128 + tid] = L > 0.0f ? acc + (b2 ? b2[(int64_t)h * 128 + tid] : 0.0f) + zb[m + tid] : 0.0f;
    if (lse && tid == 0) lse[bhq] = L > 0.0f ? M + logf(L) : -INFINITY;
}


}  // namespace

bool tc_vregen_supported(const lowram_decode_shape& s) {
    return tc_score_supported(s) && (s.m == 128 || s.m == 256) && s.d == 128;
}

int tc_partial_width(const lowram_decode_shape& s) { return s.m + s.d + 4; }

// The last CTA of each (sequence, kv-head) merges in the value kernel when the merge's shared scratch
// (chunk weights and merged sums of the G q-heads) fits in the ring.
bool tc_fused_merge(const lowram_decode_shape& s, int n_chunks) {
    // merge_last's shared memory: Z [G][m+128], chunk weights [G][n_chunks], W and L [G][2], 16 bytes of
    // alignment, and one q-head's records [n_chunks][PW]
    const size_t g = s.H_q / s.H_kv, zw = s.m + 128, pw = tc_partial_width(s);
    return (g * zw + g * (size_t)n_chunks + 2 * g + 4 + (size_t)n_chunks * pw) * sizeof(float) <=
           (size_t)kNS * kStageBytes;
}

cudaError_t launch_vregen_tc(const DecodeArgs& a, cudaStream_t st) {
    const auto& s = a.s;
    VregenTcParams p{};
    p.T = s.T;
    p.H_q = s.H_q;
    p.H_kv = s.H_kv;
    p.r = s.r;
    p.m = s.m;
    p.S_eff = a.S_eff;
    p.n_chunks = a.n_chunks;
    p.n_res = s.n_res;
    p.KC = s.r / 64;
    p.PW = a.PW;
    p.coef = (const __nv_bfloat16*)a.coef;
    p.sall = a.sall;
    p.b1 = a.b1;
    p.b2 = a.b2;
    p.w2 = (const __nv_bfloat16*)a.w2;
    p.sel = a.sel;
    p.hit = a.hit;
    p.res = ResView{s.res_dtype, a.res_val, (const __half*)a.res_scale, s.d};
    p.partial = a.partial;
    p.cnt = a.cnt;
    p.out = a.out;
    p.lse = a.lse;
    p.check = a.check;
    if ((int64_t)s.B * a.n_chunks == 0) return cudaSuccess;
    CUtensorMap mW, mW1;
    const uint64_t dW[2] = {(uint64_t)s.r, (uint64_t)s.H_kv * s.d};
    const uint32_t bW[2] = {64, 128};
    const uint64_t dW1[2] = {(uint64_t)s.d, (uint64_t)s.H_kv * s.m};
    const uint32_t bW1[2] = {64, 128};
    if (!tc::make_map(&mW, a.basis, 2, dW, bW) || !tc::make_map(&mW1, a.w1, 2, dW1, bW1)) return cudaErrorInvalidValue;
    const size_t smem = vregen_smem_bytes();
    dim3 grid((unsigned)a.n_chunks, (unsigned)s.H_kv, (unsigned)s.B);
    cudaError_t e = cudaSuccess;
    auto go = [&](auto kern) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) {
            e = launch_pdl(kern, grid, dim3(kVThreads), smem, st, mW, mW1, p);
        }
    };
    switch (s.H_q / s.H_kv) {
        case 1: go(vregen_tc_kernel<1>); break;
        case 2: go(vregen_tc_kernel<2>); break;
        case 4: go(vregen_tc_kernel<4>); break;
        case 7: go(vregen_tc_kernel<7>); break;
        case 8: go(vregen_tc_kernel<8>); break;
        default: return cudaErrorNotSupported;
    }
    return e;
}

cudaError_t launch_merge_w2(const DecodeArgs& a, int n_chunks, cudaStream_t st) {
    const auto& s = a.s;
    const int BH = s.B * s.H_q;
    if (BH == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * ((size_t)n_chunks + s.m + 128);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(merge_w2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    merge_w2_kernel<<<(unsigned)BH, 128, smem, st>>>(s.H_q, a.g, n_chunks, s.m, a.PW, a.partial,
                                                     (const __nv_bfloat16*)a.w2, a.b2, a.out, a.lse);
    return cudaGetLastError();
}

}  // namespace lowram
