// select.cu -- K2: exact top-n of each row of a float matrix, ties to the lower index, output
// ascending.  Used for the per-(sequence, kv-head) token selection of decode (the LowRAM abstract has each
// decoding step rebuild only a chosen subset of the cached tokens; taking the exactly largest scores is this
// library's reading) and for the worst-n_res residual tokens of the write side (the abstract keeps residuals
// for the tokens the predictor rebuilds worst).
//
// Radix select on order-preserving uint32 keys: four 8-bit digit passes narrow the candidates to
// the exact value of the n-th largest element (the threshold) and how many elements equal to it must
// be kept; a final pass in index order keeps every element above the threshold and the
// lowest-indexed equal ones, writing their indices ascending.
// Rows of up to 256K elements are held in registers across a cluster of up to eight CTAs; longer rows take
// one CTA each and stream from memory (rows up to 48K elements read once into shared memory).
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace lowram {

constexpr int kSelThreads = 1024;
constexpr int kSelMaxStaged = 48 * 1024;   // row elements staged in shared memory (192 KB)

// Residual lookup for the value pass: hit[row][j] = the position of token o[j] in the row's ascending
// residual list, or -1.  The list is checked (in range, strictly ascending; LOWRAM_CHECK_RES_INDEX on
// failure) and, when staged, copied into shared memory (free once the selection is written) for the
// binary searches.
struct SelectExtras {
    int32_t* hit;             // [rows][n_keep] residual row of each kept token, or null
    const int32_t* res_idx;   // [rows][n_res] ascending residual token indices
    int n_res;
    uint32_t* check;
    int rows;                 // CTAs that select; CTAs beyond them fold (FoldArgs)
    FoldArgs fold;
};

// Spare CTAs of the selection kernel fold the value predictor's first layer into the basis for the value pass:
// F[h][j][k] = sum_i w1[h][j][i] basis[h d + i][k] (float32 sums of bf16 products, rounded to bf16).  It is a small
// product (2 H_kv m d r FLOPs per call), run with warp-level bf16 MMAs (m16n8k16, float32 accumulation): a CTA of
// 1024 threads makes a tile of 128 hidden units x 256 rank columns of one head, warp w the 16 rows 16 (w % 8) and
// the 64 columns 64 (w / 8) of it.  The CTA reads only the caller's weights, so it does not wait for the kernel
// before.
constexpr int kFoldJ = 128, kFoldK = 256;
constexpr int kFoldPadA = 8, kFoldPadB = 8;   // bf16 of padding per shared row: conflict-free fragment loads
size_t fold_smem_bytes(int d) {
    return sizeof(uint16_t) * ((size_t)kFoldJ * (d + kFoldPadA) + (size_t)d * (kFoldK + kFoldPadB));
}
__host__ __device__ int fold_blocks(const FoldArgs& f) {
    return f.F ? f.copies * f.H_kv * (int)cdiv(f.m, kFoldJ) * (int)cdiv(f.r, kFoldK) : 0;
}

__device__ void fold_block(const FoldArgs& f, int blk, uint8_t* smem) {
    const int kb = (int)cdiv(f.r, kFoldK), jb = (int)cdiv(f.m, kFoldJ);
    const int per_copy = f.H_kv * jb * kb;
    const int c = blk / per_copy;
    blk -= c * per_copy;
    const int h = blk / (jb * kb), rem = blk % (jb * kb);
    const int j0 = (rem / kb) * kFoldJ, k0 = (rem % kb) * kFoldK;
    const int d = f.d, SA = d + kFoldPadA, SB = kFoldK + kFoldPadB;
    const uint16_t* w1 = reinterpret_cast<const uint16_t*>(f.w1 + c * f.mlp_stride);
    const uint16_t* basis = reinterpret_cast<const uint16_t*>(f.basis + c * f.basis_stride);
    uint16_t* As = reinterpret_cast<uint16_t*>(smem);           // [128 hidden units][d], rows padded
    uint16_t* Bs = As + kFoldJ * SA;                             // [d][256 rank columns], rows padded
    const int tid = threadIdx.x;
    // 16-byte pieces; rows past m and columns past r read as zero
    for (int e = tid; e < kFoldJ * (d / 8); e += kSelThreads) {
        const int j = e / (d / 8), i8 = (e % (d / 8)) * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (j0 + j < f.m) v = __ldg(reinterpret_cast<const uint4*>(w1 + ((int64_t)h * f.m + j0 + j) * d + i8));
        const uint32_t* pv = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
        for (int q = 0; q < 4; ++q) reinterpret_cast<uint32_t*>(As + j * SA + i8)[q] = pv[q];
    }
    for (int e = tid; e < d * (kFoldK / 8); e += kSelThreads) {
        const int i = e / (kFoldK / 8), c8 = (e % (kFoldK / 8)) * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (k0 + c8 < f.r) v = __ldg(reinterpret_cast<const uint4*>(basis + ((int64_t)h * d + i) * f.r + k0 + c8));
        const uint32_t* pv = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
        for (int q = 0; q < 4; ++q) reinterpret_cast<uint32_t*>(Bs + i * SB + c8)[q] = pv[q];
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, tq = lane & 3;
    const int jw = (warp & 7) * 16, kw = (warp >> 3) * 64;
    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
    auto pair = [](uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); };
    for (int ks = 0; ks < d; ks += 16) {
        // A fragment: rows jw + g and jw + g + 8, columns ks + 2tq (+1) and ks + 2tq + 8 (+1)
        const uint16_t* ar = As + (jw + g) * SA + ks + 2 * tq;
        const uint32_t a0 = *reinterpret_cast<const uint32_t*>(ar);
        const uint32_t a1 = *reinterpret_cast<const uint32_t*>(ar + 8 * SA);
        const uint32_t a2 = *reinterpret_cast<const uint32_t*>(ar + 8);
        const uint32_t a3 = *reinterpret_cast<const uint32_t*>(ar + 8 * SA + 8);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            // B fragment (k x n = 16 x 8): rows ks + 2tq (+1) and ks + 2tq + 8 (+1), column kw + 8nt + g
            const uint16_t* br = Bs + (ks + 2 * tq) * SB + kw + 8 * nt + g;
            const uint32_t b0 = pair(br[0], br[SB]);
            const uint32_t b1 = pair(br[8 * SB], br[9 * SB]);
            tc::mma_16816(acc[nt], a0, a1, a2, a3, b0, b1);
        }
    }
    // C fragment: rows jw + g (+8), columns kw + 8nt + 2tq (+1); stored bf16, or fp16 for an int4 cache's fp16 path
    uint16_t* F = reinterpret_cast<uint16_t*>(f.F) + (int64_t)c * f.H_kv * f.m * f.r;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        const int k = k0 + kw + 8 * nt + 2 * tq;
        if (k >= f.r) continue;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int j = j0 + jw + g + 8 * hh;
            if (j >= f.m) continue;
            uint32_t o;
            if (f.f16_out) {
                const __half2 v = __floats2half2_rn(acc[nt][2 * hh], acc[nt][2 * hh + 1]);
                o = *reinterpret_cast<const uint32_t*>(&v);
            } else {
                const __nv_bfloat162 v = __floats2bfloat162_rn(acc[nt][2 * hh], acc[nt][2 * hh + 1]);
                o = *reinterpret_cast<const uint32_t*>(&v);
            }
            *reinterpret_cast<uint32_t*>(F + ((int64_t)h * f.m + j) * f.r + k) = o;
        }
    }
}

template <bool Staged>
__device__ void match_residuals(int T, int n_keep, const int32_t* o, const SelectExtras& x, int row, uint32_t* staged) {
    const int tid = threadIdx.x;
    const int32_t* ri = x.res_idx + (int64_t)row * x.n_res;
    const bool in_smem = Staged && x.n_res <= kSelMaxStaged;
    __syncthreads();   // the kept indices o[] (global) and the staged keys are complete
    bool bad = false;
    for (int j = tid; j < x.n_res; j += kSelThreads) {
        const int v = ri[j];
        bad |= v < 0 || v >= T || (j > 0 && v <= ri[j - 1]);
        if (in_smem) staged[j] = (uint32_t)v;
    }
    if (bad) flag(x.check, LOWRAM_CHECK_RES_INDEX);
    __syncthreads();
    int32_t* hit = x.hit + (int64_t)row * n_keep;
    for (int j = tid; j < n_keep; j += kSelThreads) {
        const int tok = o[j];
        int lo = 0, hi = x.n_res - 1, found = -1;
        while (lo <= hi) {
            const int mid = (lo + hi) >> 1;
            const int v = in_smem ? (int)staged[mid] : ri[mid];
            if (v == tok) {
                found = mid;
                break;
            }
            if (v < tok) lo = mid + 1;
            else hi = mid - 1;
        }
        hit[j] = found;
    }
}

// Staged: the row's order keys are copied into shared memory once and every pass reads them there (rows of
// up to kSelMaxStaged elements); otherwise each pass streams the row from global memory (L2).  Histograms
// are kept per warp, which spreads the atomics of the first digit (few distinct exponents) over 32 copies.
template <bool Staged>
__global__ void __launch_bounds__(kSelThreads) select_topn_kernel(int T, int n_keep, const float* __restrict__ values,
                                                                  int32_t* __restrict__ out, SelectExtras x) {
    extern __shared__ uint32_t staged[];
    __shared__ uint32_t whist[kSelThreads / 32][256];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_prefix;
    __shared__ int s_need;
    __shared__ int warp_tot[33];
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    grid_dep_trigger();
    if (row >= x.rows) {   // a folding CTA: reads the caller's weights only
        fold_block(x.fold, row - x.rows, reinterpret_cast<uint8_t*>(staged));
        return;
    }
    const float* v = values + (int64_t)row * T;
    int32_t* o = out + (int64_t)row * n_keep;
    grid_dep_wait();     // the keys come from the kernel before (launched with launch_pdl)
    if (n_keep <= 0) return;
    if (n_keep >= T) {
        for (int t = tid; t < T; t += kSelThreads) o[t] = t;
        if (x.hit) match_residuals<Staged>(T, n_keep, o, x, row, staged);
        return;
    }
    if (Staged) {
        for (int t = tid; t < T; t += kSelThreads) staged[t] = order_key(v[t]);
        __syncthreads();
    }
    auto key_at = [&](int t) -> uint32_t { return Staged ? staged[t] : order_key(v[t]); };

    uint32_t prefix = 0, mask = 0;
    int need = n_keep;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        // each warp owns one histogram row: clearing and filling it need only the warp
        for (int i = lane; i < 256; i += 32) whist[warp][i] = 0;
        __syncwarp();
        for (int t = tid; t < T; t += kSelThreads) {
            const uint32_t u = key_at(t);
            if ((u & mask) == prefix) atomicAdd(&whist[warp][(u >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t c = 0;
#pragma unroll 8
            for (int w = 0; w < kSelThreads / 32; ++w) c += whist[w][tid];
            hist[tid] = c;
        }
        __syncthreads();
        if (warp == 0) {
            // lane L owns bins [8L, 8L+8); suffix sums over lanes from the top bin down
            uint32_t mine = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) mine += hist[lane * 8 + j];
            uint32_t suf = mine;
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
                uint32_t x = __shfl_down_sync(0xffffffffu, suf, o2);
                if (lane + o2 < 32) suf += x;
            }
            bool hit = suf >= (uint32_t)need && suf - mine < (uint32_t)need;
            unsigned bal = __ballot_sync(0xffffffffu, hit);
            int L = __ffs(bal) - 1;
            if (lane == L) {
                uint32_t above = suf - mine;
                for (int j = 7; j >= 0; --j) {
                    uint32_t c = hist[L * 8 + j];
                    if (above + c >= (uint32_t)need) {
                        s_prefix = prefix | ((uint32_t)(L * 8 + j) << shift);
                        s_need = need - (int)above;
                        break;
                    }
                    above += c;
                }
            }
        }
        __syncthreads();
        prefix = s_prefix;
        need = s_need;
        mask |= 0xFFu << shift;
    }
    // prefix is now the threshold key: keep every key above it and the `need` lowest-indexed equal ones.
    // Warp w owns the contiguous segment [s0, s1); one exchange of the warps' counts gives each warp its
    // output offset and the number of equal keys before it, so indices come out ascending.
    {
        constexpr int nw = kSelThreads / 32;
        const int seg = (T + nw - 1) / nw;
        const int s0 = min(T, warp * seg), s1 = min(T, s0 + seg);
        int n_gt = 0, n_eq = 0;
        for (int t = s0 + lane; t < s1; t += 32) {
            const uint32_t u = key_at(t);
            n_gt += u > prefix;
            n_eq += u == prefix;
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) {
            n_gt += __shfl_xor_sync(0xffffffffu, n_gt, o2);
            n_eq += __shfl_xor_sync(0xffffffffu, n_eq, o2);
        }
        if (lane == 0) {
            warp_tot[warp] = n_gt;
            (&whist[0][0])[warp] = (uint32_t)n_eq;
        }
        __syncthreads();
        int gt_before = 0, eq_before = 0;
        for (int w = 0; w < warp; ++w) {
            gt_before += warp_tot[w];
            eq_before += (int)(&whist[0][0])[w];
        }
        int at = gt_before + min(need, eq_before);
        int eq_rank = eq_before;
        const unsigned lt = (1u << lane) - 1u;
        for (int base = s0; base < s1; base += 32) {
            const int t = base + lane;
            const uint32_t u = t < s1 ? key_at(t) : 0u;
            const bool eq = t < s1 && u == prefix;
            const unsigned beq = __ballot_sync(0xffffffffu, eq);
            const bool take = (t < s1 && u > prefix) || (eq && eq_rank + __popc(beq & lt) < need);
            const unsigned btake = __ballot_sync(0xffffffffu, take);
            if (take) o[at + __popc(btake & lt)] = t;
            at += __popc(btake);
            eq_rank += __popc(beq);
        }
    }
    if (x.hit) match_residuals<Staged>(T, n_keep, o, x, row, staged);
}

// cluster helpers: the cluster's CTA count, and loads from a cluster CTA's shared memory (address from mapa)
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void ld_cluster_8(uint32_t addr, uint32_t (&v)[8]) {   // 32 bytes, 16-byte aligned
    asm volatile(
        "ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%8];\n\t"
        "ld.shared::cluster.v4.u32 {%4, %5, %6, %7}, [%9];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
        : "r"(addr), "r"(addr + 16)
        : "memory");
}
__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Rows of up to 256K elements, each split over a cluster of CL CTAs (CL = 1, 2, 4 or 8, the cluster's size; more
// than one only for rows longer than 8192 elements, where the keys of one CTA would not fit its registers):
// CTA c of a row holds elements [c Tc, c Tc + Tc), Tc = 1024 E, thread t the E consecutive ones from c Tc + t E,
// as order keys in registers, so no pass reads memory.  Each pass builds a 256-bin histogram per CTA (the first
// digit's atomics aggregated per warp: its few distinct exponents would otherwise collide), the cluster barrier
// publishes it, and every CTA sums the CL histograms through distributed shared memory and finds the same
// threshold bin (three histogram buffers in rotation: the one a pass clears was last read two barriers ago).  The
// passes stop early once the threshold bin is kept whole.  Each CTA then counts its (above, equal) elements, the
// cluster barrier publishes the counts, and a CTA's output starts after the lower-ranked CTAs' kept elements.
// The residual row of a kept token is its rank in the row's ascending residual list: a bitmap of the list's
// tokens in the CTA's range and the running count of its words (both built before the keys exist) give it in
// constant time.  The kept tokens and their residual rows are staged in shared memory and written out coalesced.
template <int E>
__global__ void __launch_bounds__(kSelThreads) select_cl_kernel(int T, int n_keep, int cap, const float* __restrict__ values,
                                                               int32_t* __restrict__ out, SelectExtras x) {
    constexpr int Tc = E * kSelThreads, kWords = Tc / 32;   // elements and bitmap words per CTA
    extern __shared__ uint32_t dyn[];   // fold tiles, or: bitmap [kWords], word prefix [kWords], staged output [2][cap]
    __shared__ uint32_t hist[3][256];
    __shared__ uint32_t s_prefix[3];
    __shared__ int s_need[3], s_whole[3];
    __shared__ int wsum_gt[32], wsum_eq[32];
    __shared__ int s_tot[2];            // this CTA's elements above the threshold and equal to it (read by the peers)
    __shared__ int s_res_below;         // residual tokens before this CTA's range
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int CL = (int)cluster_size(), crank = (int)tc::cluster_rank();
    grid_dep_trigger();
    const int row = blockIdx.x / CL;
    if (row >= x.rows) {   // a folding CTA: reads the caller's weights only (no cluster traffic)
        const int fi = blockIdx.x - x.rows * CL;
        if (fi < fold_blocks(x.fold)) fold_block(x.fold, fi, reinterpret_cast<uint8_t*>(dyn));
        return;
    }
    const int lo = crank * Tc, hi = min(T, lo + Tc);   // this CTA's elements (lo may be >= T: an idle CTA)
    uint32_t* bm = dyn;
    uint32_t* bpre = dyn + kWords;
    int32_t* so = reinterpret_cast<int32_t*>(dyn + 2 * kWords);
    int32_t* sh = so + cap;
    // before the keys exist: clear the first histogram; mark the residual list's tokens of this range, check the
    // list (caller input; this CTA checks every CL-th entry) and count its tokens before the range
    const bool want_hit = x.hit != nullptr;
    if (tid < 256) hist[0][tid] = 0;
    if (tid == 0) s_res_below = 0;
    if (want_hit)
        for (int w = tid; w < kWords; w += kSelThreads) bm[w] = 0;
    __syncthreads();
    if (want_hit) {
        const int32_t* ri = x.res_idx + (int64_t)row * x.n_res;
        bool bad = false;
        int below = 0;
        for (int j = tid; j < x.n_res; j += kSelThreads) {
            const int v = __ldg(ri + j);
            if (j % CL == crank) bad |= v < 0 || v >= T || (j > 0 && v <= __ldg(ri + j - 1));
            if (v >= lo && v < hi) atomicOr(&bm[(v - lo) >> 5], 1u << ((v - lo) & 31));
            below += v < lo;
        }
        if (bad) flag(x.check, LOWRAM_CHECK_RES_INDEX);
        below = warp_sum_int(below);
        if (lane == 0 && below) atomicAdd(&s_res_below, below);
        __syncthreads();
        // bpre[w] = marked tokens in words before w (kWords <= 1024: one word per thread)
        const int c = tid < kWords ? __popc(bm[tid]) : 0;
        int incl = c;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o2);
            if (lane >= o2) incl += y;
        }
        if (lane == 31) wsum_gt[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int a = wsum_gt[lane];
            int s = a;
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, s, o2);
                if (lane >= o2) s += y;
            }
            wsum_gt[lane] = s - a;
        }
        __syncthreads();
        if (tid < kWords) bpre[tid] = wsum_gt[warp] + incl - c;
        __syncthreads();   // wsum_gt is free again (the passes may be skipped)
    }
    grid_dep_wait();     // the keys come from the kernel before (launched with launch_pdl)
    if (n_keep <= 0) return;   // uniform over the cluster: no CTA touched another's memory
    const int t0 = lo + tid * E;
    uint32_t k[E];
    {
        const float* v = values + (int64_t)row * T + t0;
        if (t0 + E <= hi && (((uintptr_t)v) & 15u) == 0) {
#pragma unroll
            for (int i = 0; i < E; i += 4) {
                const float4 f = __ldcg(reinterpret_cast<const float4*>(v + i));
                k[i] = order_key(f.x);
                k[i + 1] = order_key(f.y);
                k[i + 2] = order_key(f.z);
                k[i + 3] = order_key(f.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < E; ++i) k[i] = t0 + i < hi ? order_key(__ldcg(v + i)) : 0u;
        }
    }
    // elements past the range hold key 0 and are never counted (counting stops at hi) nor taken
    uint32_t prefix = 0, mask = 0;
    int need = n_keep;
    bool whole = n_keep >= T;       // every element is kept
    for (int pass = 0; pass < 4 && !whole; ++pass) {
        const int shift = 24 - 8 * pass, cur = pass % 3, nxt = (pass + 1) % 3;
        if (tid < 256) hist[nxt][tid] = 0;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const bool in = t0 + i < hi && (k[i] & mask) == prefix;
            const uint32_t dg = (k[i] >> shift) & 255u;
            if (pass == 0) {
                const unsigned act = __ballot_sync(0xffffffffu, in);
                if (in) {
                    const unsigned peers = __match_any_sync(act, dg);
                    if (lane == __ffs(peers) - 1) atomicAdd(&hist[cur][dg], (uint32_t)__popc(peers));
                }
            } else if (in) {
                atomicAdd(&hist[cur][dg], 1u);
            }
        }
        if (CL > 1) tc::cluster_sync();   // every CTA's histogram of this pass is complete and visible
        else __syncthreads();
        if (warp == 0) {
            // lane L owns bins [8L, 8L+8), summed over the cluster; suffix sums over lanes from the top bin down
            uint32_t c8[8], mine = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) c8[j] = 0;
            for (int r = 0; r < CL; ++r) {
                uint32_t v8[8];
                ld_cluster_8(tc::peer_smem(&hist[cur][lane * 8], (uint32_t)r), v8);
#pragma unroll
                for (int j = 0; j < 8; ++j) c8[j] += v8[j];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) mine += c8[j];
            uint32_t suf = mine;
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
                const uint32_t y = __shfl_down_sync(0xffffffffu, suf, o2);
                if (lane + o2 < 32) suf += y;
            }
            const bool here = suf >= (uint32_t)need && suf - mine < (uint32_t)need;
            if (here) {
                uint32_t above = suf - mine;
                for (int j = 7; j >= 0; --j) {
                    if (above + c8[j] >= (uint32_t)need) {
                        s_prefix[cur] = prefix | ((uint32_t)(lane * 8 + j) << shift);
                        s_need[cur] = need - (int)above;
                        s_whole[cur] = (above + c8[j] == (uint32_t)need) ? 1 : 0;
                        break;
                    }
                    above += c8[j];
                }
            }
        }
        __syncthreads();
        prefix = s_prefix[cur];
        need = s_need[cur];
        mask |= 0xFFu << shift;
        if (s_whole[cur]) whole = true;   // the threshold bin is kept whole: keep all that reach the bin
    }
    // take: above the threshold (resolved digits), or in the threshold bin -- all of it when the bin is kept whole,
    // else the `need` lowest-indexed equal keys of the row (the bin is one key value once all digits are resolved)
    const bool all_T = n_keep >= T;
    int n_gt = 0, n_eq = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        if (t0 + i >= hi) break;
        const uint32_t u = k[i] & mask;
        if (all_T || u > prefix || (whole && u == prefix)) ++n_gt;
        else if (u == prefix) ++n_eq;
    }
    // block-wide exclusive scan of (n_gt, n_eq), then the cluster's: the counts of the lower-ranked CTAs
    int gi = n_gt, ei = n_eq;
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, gi, o2), c = __shfl_up_sync(0xffffffffu, ei, o2);
        if (lane >= o2) {
            gi += a;
            ei += c;
        }
    }
    if (lane == 31) {
        wsum_gt[warp] = gi;
        wsum_eq[warp] = ei;
    }
    __syncthreads();
    if (warp == 0) {
        int a = wsum_gt[lane], c = wsum_eq[lane];
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
            const int a2 = __shfl_up_sync(0xffffffffu, a, o2), c2 = __shfl_up_sync(0xffffffffu, c, o2);
            if (lane >= o2) {
                a += a2;
                c += c2;
            }
        }
        if (lane == 31) {
            s_tot[0] = a;
            s_tot[1] = c;
        }
        wsum_gt[lane] = a - wsum_gt[lane];     // exclusive prefix over warps
        wsum_eq[lane] = c - wsum_eq[lane];
    }
    if (CL > 1) tc::cluster_sync();   // every CTA's totals are visible
    else __syncthreads();
    int gt_base = 0, eq_base = 0;
    for (int r = 0; r < crank; ++r) {
        gt_base += (int)ld_cluster_u32(tc::peer_smem(&s_tot[0], (uint32_t)r));
        eq_base += (int)ld_cluster_u32(tc::peer_smem(&s_tot[1], (uint32_t)r));
    }
    const int out_base = gt_base + min(need, eq_base);
    const int n_out = gt_base + s_tot[0] + min(need, eq_base + s_tot[1]) - out_base;
    const int gt_before = gt_base + wsum_gt[warp] + gi - n_gt, eq_before = eq_base + wsum_eq[warp] + ei - n_eq;
    int at = gt_before + min(need, eq_before);
    int eq_rank = eq_before;
    int32_t* o = out + (int64_t)row * n_keep;
    int32_t* hit = want_hit ? x.hit + (int64_t)row * n_keep : nullptr;
    const int res_below = want_hit ? s_res_below : 0;
    const bool staged = n_out <= cap;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const int t = t0 + i;
        if (t >= hi) break;
        const uint32_t u = k[i] & mask;
        bool take = all_T || u > prefix || (whole && u == prefix);
        if (!take && u == prefix) take = eq_rank++ < need;
        if (take) {
            int found = -1;
            if (want_hit) {
                const int w = (t - lo) >> 5, b = (t - lo) & 31;
                const uint32_t word = bm[w];
                if ((word >> b) & 1u) found = res_below + (int)bpre[w] + __popc(word & ((1u << b) - 1u));
            }
            if (staged) {
                so[at - out_base] = t;
                sh[at - out_base] = found;
            } else {
                o[at] = t;
                if (want_hit) hit[at] = found;
            }
            ++at;
        }
    }
    if (staged) {
        __syncthreads();
        for (int i = tid; i < n_out; i += kSelThreads) {
            o[out_base + i] = so[i];
            if (want_hit) hit[out_base + i] = sh[i];
        }
    }
    if (CL > 1) tc::cluster_sync();   // no CTA leaves while a peer may still read its counts
}

size_t select_scratch_bytes(int, int, int) { return 0; }

cudaError_t launch_select_topn(int P, int T, int n_keep, const float* values, int32_t* out, cudaStream_t st,
                               int32_t* hit, const int32_t* res_idx, int n_res, uint32_t* check,
                               const FoldArgs* fold) {
    if (P == 0) return cudaSuccess;
    SelectExtras x{(hit && n_res > 0) ? hit : nullptr, res_idx, n_res, check, P, FoldArgs{}};
    if (fold) x.fold = *fold;
    const int nf = fold_blocks(x.fold);
    const size_t fold_smem = nf ? fold_smem_bytes(x.fold.d) : 0;
    // rows split over clusters while the CTAs stay within one wave and each keeps more than 4096 elements
    // a row stays in one CTA up to 8 keys a thread (the barriers of a cluster cost more than the extra keys); longer
    // rows split over a cluster while the CTAs still fit one wave
    int CL = 1;
    const int sms = tc::sm_count();
    while (CL < 8 && (int64_t)P * CL * 2 <= sms && T > CL * 8 * kSelThreads) CL *= 2;
    int E = 4;
    while (E < 32 && (int64_t)E * kSelThreads * CL < T) E *= 2;
    if ((int64_t)E * kSelThreads * CL >= T) {
        const int Tc = E * kSelThreads;
        const int cap = std::min(Tc, std::max(n_keep, 0)) <= 12288 ? std::min(Tc, std::max(n_keep, 0)) : 0;
        size_t smem = sizeof(uint32_t) * (2 * (size_t)(Tc / 32) + 2 * (size_t)cap);
        if (fold_smem > smem) smem = fold_smem;
        const int nfc = (int)cdiv(nf, CL) * CL;
        auto go = [&](auto kern) -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(P * CL + nfc));
            cfg.blockDim = dim3(kSelThreads);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = st;
            cudaLaunchAttribute attr[2];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = (unsigned)CL;
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 2;
            e = cudaLaunchKernelEx(&cfg, kern, T, n_keep, cap, values, out, x);
            return e != cudaSuccess ? e : cudaGetLastError();
        };
        switch (E) {
            case 4: return go(select_cl_kernel<4>);
            case 8: return go(select_cl_kernel<8>);
            case 16: return go(select_cl_kernel<16>);
            default: return go(select_cl_kernel<32>);
        }
    }
    const dim3 grid((unsigned)(P + nf));
    const bool staged = n_keep > 0 && T <= kSelMaxStaged;
    size_t smem = staged ? sizeof(uint32_t) * (size_t)T : 0;   // the staged keys also hold the residual list (n_res <= T)
    if (fold_smem > smem) smem = fold_smem;
    auto kern = staged ? select_topn_kernel<true> : select_topn_kernel<false>;
    const size_t smax = staged ? sizeof(uint32_t) * kSelMaxStaged : fold_smem;
    if (smax > 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smax);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_pdl(kern, grid, dim3(kSelThreads), smem, st, T, n_keep, values, out, x);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace lowram
