// dense.cu -- comparator: split-T decode attention over an explicit, uncompressed, already rotated
// K/V cache [B, T, H_kv, d]; sequence b's rows start at token b * Ts, so the exact tail of recent tokens is read
// in place from its [B, T_cap, H_kv, d] buffer with Ts = T_cap.  Same split-softmax partial layout and merge
// kernel as the compressed path.  This is the cache the compressed one replaces (LowRAM abstract: the KV
// cache's memory footprint caps batch size and throughput).
//
// HBM-bound: every K and V byte is read once, 16 bytes per lane, streamed through a per-thread cp.async
// ring in shared memory.  A group of d/VEC lanes holds one token (VEC elements per lane); the lanes of a
// group reduce the q.k dot products with xor shuffles and keep an online softmax state per q-head;
// groups, then warps, merge their states at the end.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace lowram {

constexpr int kDenseThreads = 128;
constexpr int kDenseU = 4;        // token steps per iteration
constexpr int kDenseStages = 4;   // iterations of loads in flight
constexpr size_t kDenseSmem = (size_t)kDenseStages * kDenseU * 2 * kDenseThreads * 16;

// 16-byte global -> shared copy through L2; zero-filled when !ok.
__device__ __forceinline__ void cp_async16(uint4* dst, const void* src, bool ok) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(ok ? 16u : 0u)
                 : "memory");
}

// 16-byte pieces of a row converted to float.
template <typename TE>
struct Vec16;
template <>
struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void cvt(const uint4& u, float (&x)[8]) {
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
    __device__ __forceinline__ static void cvt(const uint4& u, float (&x)[4]) {
        x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y); x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
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
__global__ void __launch_bounds__(kDenseThreads) dense_kernel(int T, int Ts, int H_q, int H_kv, float scale,
                                                              const TE* __restrict__ q, const TE* __restrict__ K,
                                                              const TE* __restrict__ V, float* __restrict__ partial,
                                                              int n_split) {
    constexpr int VEC = Vec16<TE>::N;
    constexpr int LPT = D / VEC;          // lanes per token
    constexpr int TPW = 32 / LPT;         // tokens per warp step
    constexpr int NW = kDenseThreads / 32;
    const int h = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
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
    // Deep pipeline without registers: every thread streams exactly the 16-byte pieces of K and V it will
    // use into its own shared-memory slots with cp.async, kDenseStages iterations ahead of the arithmetic,
    // so each SM keeps tens of KB of HBM reads in flight.  No slot is shared, so no CTA barrier is needed.
    constexpr int U = kDenseU;
    extern __shared__ uint4 ring[];   // [kDenseStages][U][2][kDenseThreads]
    const int tid = threadIdx.x;
    const int n_it = (int)cdiv(t_end - t_begin, NW * TPW * U);
    auto issue = [&](int it) {
        if (it < n_it) {
            const int s = it % kDenseStages;
            const int t0 = t_begin + (it * NW + warp) * TPW * U;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int t = t0 + u * TPW + grp;
                const bool ok = t < t_end;
                const int64_t off = (((int64_t)b * Ts + (ok ? t : t_begin)) * H_kv + h) * D + sub * VEC;
                cp_async16(&ring[((s * U + u) * 2 + 0) * kDenseThreads + tid], K + off, ok);
                cp_async16(&ring[((s * U + u) * 2 + 1) * kDenseThreads + tid], V + off, ok);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
#pragma unroll
    for (int it = 0; it < kDenseStages - 1; ++it) issue(it);
    for (int it = 0; it < n_it; ++it) {
        issue(it + kDenseStages - 1);
        asm volatile("cp.async.wait_group %0;" ::"n"(kDenseStages - 1) : "memory");
        const int s = it % kDenseStages;
        const int t0 = t_begin + (it * NW + warp) * TPW * U;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = t0 + u * TPW + grp;
            const bool valid = t < t_end;
            float kx[VEC], vx[VEC];
            Vec16<TE>::cvt(ring[((s * U + u) * 2 + 0) * kDenseThreads + tid], kx);
            Vec16<TE>::cvt(ring[((s * U + u) * 2 + 1) * kDenseThreads + tid], vx);
#pragma unroll
            for (int j = 0; j < G; ++j) {
                float sc = 0.0f;
                if (valid)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) sc = fmaf(qv[j][e], kx[e], sc);
#pragma unroll
                for (int o = LPT / 2; o > 0; o >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, o);
                if (valid) {
                    const float mn = fmaxf(m[j], sc);
                    const float corr = (m[j] == -INFINITY) ? 0.0f : __expf(m[j] - mn);
                    const float p = __expf(sc - mn);
                    l[j] = l[j] * corr + p;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) acc[j][e] = fmaf(p, vx[e], acc[j][e] * corr);
                    m[j] = mn;
                }
            }
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
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

// ------------------------------------------------------------------------------------------------
// bf16, d = 128.  Each warp streams blocks of 16 tokens of K and V through its own cp.async ring in shared memory
// and keeps an online softmax per q-head:
//   scores   eight lanes per token, 16 features each, four tokens per pass: the K row slices (read back swizzled)
//            against the q-heads held in registers (pre-scaled fp32 pairs), packed fp32x2 FMAs, three shuffles
//            to add;
//   weights  block max and sum by shuffles, one exp per (token, q-head);
//   values   lane = 4 features: each token's V row (8 bytes per lane) times its weight, broadcast by shuffle.
// Only K and V pass through shared memory (the queries never do), so its traffic is twice the bytes streamed.
// Up to four q-heads per kv-head: dense_bf16_pw_kernel (persistent, one record per warp and work item).  More
// q-heads (whose queries would not fit in registers) take dense_bf16_smemq_kernel: a CTA of four warps per
// (kv-head, token range, sequence), two ring stages per warp, the pre-scaled queries in shared memory read by two
// lanes per token, and the warps' states merged in shared memory into one record per (sequence, q-head).
// ------------------------------------------------------------------------------------------------
constexpr int kD2Warps = 4;
constexpr int kD2Threads = 32 * kD2Warps;
constexpr int kD2Rows = 16;                  // tokens per warp block
constexpr int kD2Stage = kD2Rows * 256;      // 16 token rows of 128 bf16

size_t dense2_smem(int G) {   // rings (they also hold the warps' final states); with more than four q-heads, the queries
    return (G > 4 ? (size_t)G * 128 * 4 : 0) + std::max((size_t)kD2Warps * 4 * kD2Stage, (size_t)kD2Warps * G * 130 * 4);
}

__device__ __forceinline__ void bf16x2_to_f2(uint32_t w, uint64_t& out) {
    out = tc::f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// One 16-token block of a warp's state: scores of tokens 4 ps + tg (every lane of a token group ends with the
// token's score), the online softmax update, and the weighted values.
template <int G, int J0 = 0, int GH = G>
__device__ __forceinline__ void dense_block_heads(const uint8_t* Kt, const uint8_t* Vt, int t0, int t_end, int tg, int fo,
                                                  int lane, const uint64_t (&q2)[G][8], float (&m)[G], float (&l)[G],
                                                  uint64_t (&acc)[G][2]) {
    using namespace tc;
    float sc[GH][4];
#pragma unroll
    for (int ps = 0; ps < 4; ++ps) {
        const int r = 4 * ps + tg;
        const uint4 ka = *reinterpret_cast<const uint4*>(Kt + r * 256 + (((2 * fo) ^ (r & 15)) << 4));
        const uint4 kb = *reinterpret_cast<const uint4*>(Kt + r * 256 + (((2 * fo + 1) ^ (r & 15)) << 4));
        const uint32_t kw[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
        uint64_t kp[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) bf16x2_to_f2(kw[e], kp[e]);
#pragma unroll
        for (int jj = 0; jj < GH; ++jj) {
            const int jq = J0 + jj;
            uint64_t s2 = 0ull;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                s2 = f2_fma(q2[jq][e], kp[e], s2);
            }
            const float2 sv = f2_unpack(s2);
            float v = sv.x + sv.y;
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            sc[jj][ps] = (t0 + r < t_end) ? v : -INFINITY;
        }
    }
    // online softmax over the block: max and weight sum across the four token groups (weights overwrite scores)
#pragma unroll
    for (int jj = 0; jj < GH; ++jj) {
        const int jq = J0 + jj;
        float bm = fmaxf(fmaxf(sc[jj][0], sc[jj][1]), fmaxf(sc[jj][2], sc[jj][3]));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
        const float mn = fmaxf(m[jq], bm);
        const float f = (m[jq] == -INFINITY) ? 0.0f : __expf(m[jq] - mn);
        float ls = 0.0f;
#pragma unroll
        for (int ps = 0; ps < 4; ++ps) {
            sc[jj][ps] = sc[jj][ps] == -INFINITY ? 0.0f : __expf(sc[jj][ps] - mn);
            ls += sc[jj][ps];
        }
        ls += __shfl_xor_sync(0xffffffffu, ls, 8);
        ls += __shfl_xor_sync(0xffffffffu, ls, 16);
        l[jq] = l[jq] * f + ls;
        const uint64_t f2 = f2_pack(f, f);
        acc[jq][0] = f2_mul(acc[jq][0], f2);
        acc[jq][1] = f2_mul(acc[jq][1], f2);
        m[jq] = mn;
    }
    // values: lane = features 4 lane .. 4 lane + 3; token 4 ps + g's weight sits in lanes 8 g .. 8 g + 7
#pragma unroll
    for (int t = 0; t < kD2Rows; ++t) {
        const uint2 vv = *reinterpret_cast<const uint2*>(Vt + t * 256 + lane * 8);
        uint64_t vp0, vp1;
        bf16x2_to_f2(vv.x, vp0);
        bf16x2_to_f2(vv.y, vp1);
#pragma unroll
        for (int jj = 0; jj < GH; ++jj) {
            const int jq = J0 + jj;
            const float pt = __shfl_sync(0xffffffffu, sc[jj][t >> 2], (t & 3) * 8);
            const uint64_t p2 = f2_pack(pt, pt);
            acc[jq][0] = f2_fma(p2, vp0, acc[jq][0]);
            acc[jq][1] = f2_fma(p2, vp1, acc[jq][1]);
        }
    }
}

// Persistent variant for up to four q-heads per kv-head: one CTA of 8 warps per SM, and every warp an independent
// stream over its own work items (a sequence, a kv-head and a token split each; items gw, gw + warps, ...), with
// a 3-stage ring of 16-token K/V blocks running across item boundaries, so two blocks (16 KB) per warp, 128 KB per
// SM, are in flight whenever the warp computes.  A warp writes one flash-decoding record per item: no CTA-wide
// merge, no barrier.
constexpr int kPwWarps = 8, kPwStages = 3;
constexpr size_t kPwSmem = (size_t)kPwWarps * kPwStages * 2 * kD2Stage;

template <int G>
__global__ void __launch_bounds__(32 * kPwWarps, 1) dense_bf16_pw_kernel(int B, int T, int Ts, int H_q, int H_kv,
                                                                         float scale, const __nv_bfloat16* __restrict__ q,
                                                                         const __nv_bfloat16* __restrict__ K,
                                                                         const __nv_bfloat16* __restrict__ V,
                                                                         float* __restrict__ partial, int n_split) {
    using namespace tc;
    extern __shared__ __align__(16) uint8_t dsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tg = lane >> 3, fo = lane & 7;
    uint8_t* wbase = dsm + (size_t)warp * kPwStages * 2 * kD2Stage;   // stage s: K at 2s, V at 2s + 1
    const int gw = blockIdx.x * kPwWarps + warp, nw = gridDim.x * kPwWarps;
    const int n_items = B * H_kv * n_split;
    const int per = (int)cdiv(T, n_split);
    // item -> (b, h, split): splits of one (b, h) adjacent, kv-heads of one sequence next
    auto item_of = [&](int it, int& b, int& h, int& sp, int& tb, int& te) {
        sp = it % n_split;
        const int bh = it / n_split;
        h = bh % H_kv;
        b = bh / H_kv;
        tb = sp * per;
        te = min(T, tb + per);
    };
    auto nblocks = [&](int tb, int te) { return te > tb ? (int)cdiv(te - tb, kD2Rows) : 0; };
    // issue cursor: the warp's item ordinal and block within it
    int iss_io = 0, iss_kb = 0, iss_n = 0;
    uint32_t iss_k = 0;   // blocks issued
    int ib = 0, ih = 0, isp = 0, itb = 0, ite = 0;
    auto iss_item = [&]() {
        const int it = gw + iss_io * nw;
        if (it < n_items) {
            item_of(it, ib, ih, isp, itb, ite);
            iss_n = nblocks(itb, ite);
        } else {
            iss_n = -1;
        }
    };
    iss_item();
    // issue the next block of the warp's sequence (or an empty group past its end)
    auto issue = [&]() {
        while (iss_n == 0) {   // an empty item (T split finer than the tokens): skip it
            ++iss_io;
            iss_kb = 0;
            iss_item();
        }
        if (iss_n > 0) {
            const int s = (int)(iss_k % kPwStages);
            uint8_t* Kt = wbase + (2 * s) * kD2Stage;
            uint8_t* Vt = wbase + (2 * s + 1) * kD2Stage;
            const int t0 = itb + iss_kb * kD2Rows;
#pragma unroll 4
            for (int i = lane; i < kD2Rows * 16; i += 32) {
                const int r = i >> 4, c = i & 15;
                const int t = t0 + r;
                const bool ok = t < ite;
                const int64_t off = (((int64_t)ib * Ts + (ok ? t : itb)) * H_kv + ih) * 128 + c * 8;
                cp_async16(reinterpret_cast<uint4*>(Kt + r * 256 + ((c ^ (r & 15)) << 4)), K + off, ok);
                cp_async16(reinterpret_cast<uint4*>(Vt + r * 256 + (c << 4)), V + off, ok);
            }
            if (++iss_kb == iss_n) {
                ++iss_io;
                iss_kb = 0;
                iss_item();
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        ++iss_k;
    };
    for (int k = 0; k < kPwStages - 1; ++k) issue();
    // compute cursor
    uint32_t cmp_k = 0;
    for (int io = 0;; ++io) {
        const int it = gw + io * nw;
        if (it >= n_items) break;
        int b, h, sp, tb, te;
        item_of(it, b, h, sp, tb, te);
        const int nb = nblocks(tb, te);
        // this item's queries: 16 features of every q-head per lane, pre-scaled
        uint64_t q2[G][8];
#pragma unroll
        for (int jq = 0; jq < G; ++jq) {
            const uint4* src = reinterpret_cast<const uint4*>(q + ((int64_t)b * H_q + h * G + jq) * 128 + 16 * fo);
            const uint4 u0 = __ldg(src), u1 = __ldg(src + 1);
            const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e)
                q2[jq][e] = f2_pack(__uint_as_float(w[e] << 16) * scale, __uint_as_float(w[e] & 0xffff0000u) * scale);
        }
        float m[G], l[G];
        uint64_t acc[G][2];
#pragma unroll
        for (int jq = 0; jq < G; ++jq) {
            m[jq] = -INFINITY;
            l[jq] = 0.0f;
            acc[jq][0] = acc[jq][1] = 0ull;
        }
        for (int kb = 0; kb < nb; ++kb, ++cmp_k) {
            issue();   // the block kPwStages - 1 ahead
            asm volatile("cp.async.wait_group %0;" ::"n"(kPwStages - 1) : "memory");
            __syncwarp();
            const int s = (int)(cmp_k % kPwStages);
            dense_block_heads<G>(wbase + (2 * s) * kD2Stage, wbase + (2 * s + 1) * kD2Stage, tb + kb * kD2Rows, te, tg,
                                 fo, lane, q2, m, l, acc);
            __syncwarp();   // this stage is read; a later issue refills it
        }
        // the item's record: weighted value sum (features 4 lane .. 4 lane + 3), max logit, weight sum
#pragma unroll
        for (int jq = 0; jq < G; ++jq) {
            float* dst = partial + (((int64_t)b * H_q + h * G + jq) * n_split + sp) * 130;
            const float2 a0 = f2_unpack(acc[jq][0]), a1 = f2_unpack(acc[jq][1]);
            *reinterpret_cast<float2*>(dst + lane * 4) = a0;
            *reinterpret_cast<float2*>(dst + lane * 4 + 2) = a1;
            if (lane == 0) {
                dst[128] = m[jq];
                dst[129] = l[jq];
            }
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

template <int G>
__global__ void __launch_bounds__(kD2Threads) dense_bf16_smemq_kernel(int T, int Ts, int H_q, int H_kv, float scale,
                                                                const __nv_bfloat16* __restrict__ q,
                                                                const __nv_bfloat16* __restrict__ K,
                                                                const __nv_bfloat16* __restrict__ V,
                                                                float* __restrict__ partial, int n_split) {
    using namespace tc;
    extern __shared__ __align__(16) uint8_t dsm[];
    float* Qs = reinterpret_cast<float*>(dsm);   // [G][128] pre-scaled queries
    const int h = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t* wbase = dsm + G * 128 * 4 + warp * 4 * kD2Stage;   // Kt[2], Vt[2]
    const int per = (int)cdiv(T, n_split);
    const int t_begin = split * per, t_end = min(T, t_begin + per);
    for (int e = tid; e < G * 128; e += kD2Threads)
        Qs[e] = __bfloat162float(q[((int64_t)b * H_q + h * G) * 128 + e]) * scale;
    __syncthreads();
    const int nblk = t_end > t_begin ? (int)cdiv(t_end - t_begin, kD2Rows) : 0;
    auto issue = [&](int k) {
        const int blk = warp + k * kD2Warps;
        if (blk < nblk) {
            const int t0 = t_begin + blk * kD2Rows;
            uint8_t* Kt = wbase + (k & 1) * kD2Stage;
            uint8_t* Vt = wbase + (2 + (k & 1)) * kD2Stage;
#pragma unroll 4
            for (int i = lane; i < kD2Rows * 16; i += 32) {
                const int r = i >> 4, c = i & 15;
                const int t = t0 + r;
                const bool ok = t < t_end;
                const int64_t off = (((int64_t)b * Ts + (ok ? t : t_begin)) * H_kv + h) * 128 + c * 8;
                cp_async16(reinterpret_cast<uint4*>(Kt + r * 256 + ((c ^ (r & 15)) << 4)), K + off, ok);
                cp_async16(reinterpret_cast<uint4*>(Vt + r * 256 + (c << 4)), V + off, ok);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    float m[G], l[G];
    uint64_t acc[G][2];
#pragma unroll
    for (int jq = 0; jq < G; ++jq) {
        m[jq] = -INFINITY;
        l[jq] = 0.0f;
        acc[jq][0] = acc[jq][1] = 0ull;
    }
    issue(0);
    for (int k = 0; warp + k * kD2Warps < nblk; ++k) {
        issue(k + 1);
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        __syncwarp();
        const uint8_t* Kt = wbase + (k & 1) * kD2Stage;
        const uint8_t* Vt = wbase + (2 + (k & 1)) * kD2Stage;
        const int t0 = t_begin + (warp + k * kD2Warps) * kD2Rows;
        const int r = lane >> 1, fh = lane & 1;          // scores: token r, feature half fh
        const bool valid = t0 + r < t_end;
        uint64_t s2[G];
#pragma unroll
        for (int jq = 0; jq < G; ++jq) s2[jq] = 0ull;
#pragma unroll 4
        for (int c8 = 0; c8 < 8; ++c8) {
            const int c = fh * 8 + c8;
            const uint4 kv = *reinterpret_cast<const uint4*>(Kt + r * 256 + ((c ^ (r & 15)) << 4));
            uint64_t kp[4];
            bf16x2_to_f2(kv.x, kp[0]);
            bf16x2_to_f2(kv.y, kp[1]);
            bf16x2_to_f2(kv.z, kp[2]);
            bf16x2_to_f2(kv.w, kp[3]);
#pragma unroll
            for (int jq = 0; jq < G; ++jq) {
                const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(Qs + jq * 128 + c * 8);
                const ulonglong2 qb = *reinterpret_cast<const ulonglong2*>(Qs + jq * 128 + c * 8 + 4);
                s2[jq] = f2_fma(qa.x, kp[0], s2[jq]);
                s2[jq] = f2_fma(qa.y, kp[1], s2[jq]);
                s2[jq] = f2_fma(qb.x, kp[2], s2[jq]);
                s2[jq] = f2_fma(qb.y, kp[3], s2[jq]);
            }
        }
        // weights of the block (both lanes of a token hold its score), online softmax update
        float p[G];
#pragma unroll
        for (int jq = 0; jq < G; ++jq) {
            const float2 sv = f2_unpack(s2[jq]);
            float part = sv.x + sv.y;
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            const float sc = valid ? part : -INFINITY;
            const float mn = fmaxf(m[jq], warp_max(sc));
            const float f = (m[jq] == -INFINITY) ? 0.0f : __expf(m[jq] - mn);
            p[jq] = valid ? __expf(sc - mn) : 0.0f;
            l[jq] = l[jq] * f + 0.5f * warp_sum(p[jq]);   // every token counted by its two lanes
            const uint64_t f2 = f2_pack(f, f);
            acc[jq][0] = f2_mul(acc[jq][0], f2);
            acc[jq][1] = f2_mul(acc[jq][1], f2);
            m[jq] = mn;
        }
        // values: lane = features 4*lane .. 4*lane+3; token t's weight sits in lane 2t
#pragma unroll 8
        for (int t = 0; t < kD2Rows; ++t) {
            const uint2 vv = *reinterpret_cast<const uint2*>(Vt + t * 256 + lane * 8);
            uint64_t vp0, vp1;
            bf16x2_to_f2(vv.x, vp0);
            bf16x2_to_f2(vv.y, vp1);
#pragma unroll
            for (int jq = 0; jq < G; ++jq) {
                const float pt = __shfl_sync(0xffffffffu, p[jq], 2 * t);
                const uint64_t p2 = f2_pack(pt, pt);
                acc[jq][0] = f2_fma(p2, vp0, acc[jq][0]);
                acc[jq][1] = f2_fma(p2, vp1, acc[jq][1]);
            }
        }
        __syncwarp();   // this stage is read; the next issue refills it
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    // combine the warps' softmax states through shared memory (the rings are free): one record per CTA
    __syncthreads();
    float* st = reinterpret_cast<float*>(dsm + G * 128 * 4);     // [kD2Warps][G][130]
#pragma unroll
    for (int jq = 0; jq < G; ++jq) {
        float* w = st + (warp * G + jq) * 130;
        const float2 a0 = f2_unpack(acc[jq][0]), a1 = f2_unpack(acc[jq][1]);
        *reinterpret_cast<float2*>(w + lane * 4) = a0;
        *reinterpret_cast<float2*>(w + lane * 4 + 2) = a1;
        if (lane == 0) {
            w[128] = m[jq];
            w[129] = l[jq];
        }
    }
    __syncthreads();
    for (int jq = warp; jq < G; jq += kD2Warps) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kD2Warps; ++w) M = fmaxf(M, st[(w * G + jq) * 130 + 128]);
        float L = 0.0f, a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int w = 0; w < kD2Warps; ++w) {
            const float* src = st + (w * G + jq) * 130;
            const float mw = src[128];
            const float f = (mw == -INFINITY) ? 0.0f : __expf(mw - M);
            L = fmaf(f, src[129], L);
#pragma unroll
            for (int e = 0; e < 4; ++e) a[e] = fmaf(f, src[lane * 4 + e], a[e]);
        }
        float* dst = partial + (((int64_t)b * H_q + h * G + jq) * n_split + split) * 130;
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[lane * 4 + e] = a[e];
        if (lane == 0) {
            dst[128] = M;
            dst[129] = L;
        }
    }
}

// Token splits per (sequence, kv-head), at least 128 tokens each: about two work items per warp of the persistent
// kernel (bf16, d = 128, up to four q-heads per kv-head; 8 warps on every SM), else about eight CTAs per SM.
static bool dense_persistent(int H_q, int H_kv, int d, int dtype) {
    return dtype == LOWRAM_BF16 && d == 128 && H_q / H_kv <= 4;
}
int dense_splits(int B, int T, int H_kv, int H_q, int d, int dtype) {
    const int64_t units = (int64_t)B * H_kv;
    if (units == 0 || T == 0) return 1;
    const int64_t target = dense_persistent(H_q, H_kv, d, dtype) ? 2 * (int64_t)tc::sm_count() * kPwWarps
                                                                 : 8 * (int64_t)tc::sm_count();
    int64_t s = cdiv(target, units);
    s = s < 1 ? 1 : s;
    const int64_t cap = cdiv(T, 128);
    return (int)(s > cap ? cap : s);
}

template <typename TE, int D>
static cudaError_t dense_g(int B, int T, int Ts, int H_q, int H_kv, float scale, const void* q, const void* k, const void* v,
                           float* partial, int n_split, cudaStream_t st) {
    // the kv-heads of one token range are adjacent in launch order: they run together and read the same
    // [H_kv, d] token rows of K and V, so DRAM sees whole rows rather than one head's 2*d bytes per row
    dim3 grid((unsigned)H_kv, (unsigned)n_split, (unsigned)B);
    const TE *Q = (const TE*)q, *K = (const TE*)k, *V = (const TE*)v;
    cudaError_t e = cudaSuccess;
    auto go = [&](auto kern) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDenseSmem);
        if (e == cudaSuccess) {
            kern<<<grid, kDenseThreads, kDenseSmem, st>>>(T, Ts, H_q, H_kv, scale, Q, K, V, partial, n_split);
            e = cudaGetLastError();
        }
    };
    switch (H_q / H_kv) {
        case 1: go(dense_kernel<TE, D, 1>); break;
        case 2: go(dense_kernel<TE, D, 2>); break;
        case 4: go(dense_kernel<TE, D, 4>); break;
        case 7: go(dense_kernel<TE, D, 7>); break;
        case 8: go(dense_kernel<TE, D, 8>); break;
        default: return cudaErrorNotSupported;
    }
    return e;
}

int dense_records_max(int B, int T, int H_kv, int H_q, int d) {
    return std::max(dense_splits(B, T, H_kv, H_q, d, LOWRAM_BF16), dense_splits(B, T, H_kv, H_q, d, LOWRAM_F32));
}

template <int G>
static cudaError_t dense2_go(int B, int T, int Ts, int H_q, int H_kv, float scale, const void* q, const void* k, const void* v,
                             float* partial, int n_split, cudaStream_t st) {
    const size_t smem = dense2_smem(G);
    // the kv-heads of one token range are adjacent in launch order (they read the same token rows)
    dim3 grid((unsigned)H_kv, (unsigned)n_split, (unsigned)B);
    auto go = [&](auto kern) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kD2Threads, smem, st>>>(T, Ts, H_q, H_kv, scale, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                                             (const __nv_bfloat16*)v, partial, n_split);
        return cudaGetLastError();
    };
    if constexpr (G <= 4) {
        const int n_items = B * H_kv * n_split;
        const int grid = std::min(tc::sm_count(), (int)cdiv(n_items, kPwWarps));
        cudaError_t e = cudaFuncSetAttribute(dense_bf16_pw_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kPwSmem);
        if (e != cudaSuccess) return e;
        dense_bf16_pw_kernel<G><<<grid, 32 * kPwWarps, kPwSmem, st>>>(B, T, Ts, H_q, H_kv, scale,
                                                                        (const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                                                                        (const __nv_bfloat16*)v, partial, n_split);
        return cudaGetLastError();
    } else {
        return go(dense_bf16_smemq_kernel<G>);
    }
}

cudaError_t launch_dense(int B, int T, int Ts, int H_q, int H_kv, int d, int dtype, float scale, const void* q, const void* k,
                         const void* v, float* partial, int n_split, cudaStream_t st) {
    if (B == 0) return cudaSuccess;
    if (dtype == LOWRAM_BF16 && d == 128) {
        switch (H_q / H_kv) {
            case 1: return dense2_go<1>(B, T, Ts, H_q, H_kv, scale, q, k, v, partial, n_split, st);
            case 2: return dense2_go<2>(B, T, Ts, H_q, H_kv, scale, q, k, v, partial, n_split, st);
            case 4: return dense2_go<4>(B, T, Ts, H_q, H_kv, scale, q, k, v, partial, n_split, st);
            case 7: return dense2_go<7>(B, T, Ts, H_q, H_kv, scale, q, k, v, partial, n_split, st);
            case 8: return dense2_go<8>(B, T, Ts, H_q, H_kv, scale, q, k, v, partial, n_split, st);
            default: return cudaErrorNotSupported;
        }
    }
    if (dtype == LOWRAM_BF16) {
        if (d == 128) return dense_g<__nv_bfloat16, 128>(B, T, Ts, H_q, H_kv, scale, q, k, v, partial, n_split, st);
        if (d == 64) return dense_g<__nv_bfloat16, 64>(B, T, Ts, H_q, H_kv, scale, q, k, v, partial, n_split, st);
    } else {
        if (d == 128) return dense_g<float, 128>(B, T, Ts, H_q, H_kv, scale, q, k, v, partial, n_split, st);
        if (d == 64) return dense_g<float, 64>(B, T, Ts, H_q, H_kv, scale, q, k, v, partial, n_split, st);
    }
    return cudaErrorNotSupported;
}

}  // namespace lowram
