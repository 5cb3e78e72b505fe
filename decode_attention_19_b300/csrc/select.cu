// select.cu -- K2: exact top-n of each row of a float matrix, ties to the lower index, output
// ascending.  Used for the per-(sequence, kv-head) token selection of decode (LowRAM abstract:
// "reconstructing only a selected subset of KV pairs at each decoding step"; the rule -- exact
// largest scores -- is this library's reading) and for the worst-n_res residual tokens of the write
// side ("stores residuals only for the tokens it reconstructs worst").
//
// Radix select on order-preserving uint32 keys: four 8-bit digit passes narrow the candidates to
// the exact value of the n-th largest element (the threshold) and how many elements equal to it must
// be kept; a final pass in index order keeps every element above the threshold and the
// lowest-indexed equal ones, writing their indices ascending (each warp compacts a contiguous segment
// after one exchange of per-warp counts).
// One CTA per row; rows up to 48K elements are read once into shared memory.
#include "common.cuh"
#include "kernels.h"

namespace lowram {

constexpr int kSelThreads = 1024;
constexpr int kSelMaxStaged = 48 * 1024;   // row elements staged in shared memory (192 KB)

// Residual lookup for the value pass: hit[row][j] = the position of token o[j] in the row's ascending
// residual list, or -1.  The list is checked (in range, strictly ascending; LOWRAM_CHECK_RES_INDEX on
// failure) and, when staged, copied into shared memory (free once the selection is written) for the
// binary searches.
struct SelectExtras {
    int32_t* zero_cnt;        // [rows] set to 0, or null
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
int fold_blocks(const FoldArgs& f) {
    return f.F ? f.copies * f.H_kv * (int)cdiv(f.m, kFoldJ) * (int)cdiv(f.r, kFoldK) : 0;
}

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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
            mma_16816(acc[nt], a0, a1, a2, a3, b0, b1);
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
    if (x.zero_cnt && tid == 0) x.zero_cnt[row] = 0;
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

// Rows of up to 32K elements: each of the 1024 threads holds E consecutive elements' order keys in registers
// (thread t: elements [t E, t E + E)), so no pass reads memory.  One shared 256-bin histogram per pass
// (double-buffered: the next pass's is cleared during this one), the first digit's atomics aggregated per warp
// (its few distinct exponents would otherwise collide), two barriers per pass, and an early stop once the
// threshold bin is kept whole.  One block-wide scan of (above, equal) counts gives each thread its output offset,
// and the residual list (a caller input, staged in shared memory before waiting for the keys) is searched for the
// thread's own kept tokens.
template <int E>
__global__ void __launch_bounds__(kSelThreads) select_reg_kernel(int T, int n_keep, const float* __restrict__ values,
                                                                int32_t* __restrict__ out, SelectExtras x) {
    extern __shared__ uint32_t dyn[];               // the row's residual list (n_res ints), or the fold's tiles
    __shared__ uint32_t hist[2][256];
    __shared__ uint32_t s_prefix[2];
    __shared__ int s_need[2], s_whole[2];
    __shared__ int wsum_gt[32], wsum_eq[32];
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    grid_dep_trigger();
    if (row >= x.rows) {   // a folding CTA: reads the caller's weights only
        fold_block(x.fold, row - x.rows, reinterpret_cast<uint8_t*>(dyn));
        return;
    }
    // before the keys exist: clear the first histogram, stage and check the residual list (caller inputs)
    if (tid < 256) hist[0][tid] = 0;
    const bool want_hit = x.hit != nullptr;
    const int32_t* ri = want_hit ? x.res_idx + (int64_t)row * x.n_res : nullptr;
    if (want_hit) {
        bool bad = false;
        for (int j = tid; j < x.n_res; j += kSelThreads) {
            const int v = __ldg(ri + j);
            bad |= v < 0 || v >= T || (j > 0 && v <= __ldg(ri + j - 1));
            dyn[j] = (uint32_t)v;
        }
        if (bad) flag(x.check, LOWRAM_CHECK_RES_INDEX);
    }
    __syncthreads();     // the cleared histogram and the staged list before any use
    grid_dep_wait();     // the keys come from the kernel before (launched with launch_pdl)
    if (x.zero_cnt && tid == 0) x.zero_cnt[row] = 0;
    if (n_keep <= 0) return;
    int32_t* o = out + (int64_t)row * n_keep;
    const int t0 = tid * E;
    uint32_t k[E];
    {
        const float* v = values + (int64_t)row * T + t0;
        if (t0 + E <= T && (((uintptr_t)v) & 15u) == 0) {
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
            for (int i = 0; i < E; ++i) k[i] = t0 + i < T ? order_key(__ldcg(v + i)) : 0u;
        }
    }
    // keys past T are 0, the smallest order key: they are never counted (counting stops at T) nor taken
    uint32_t prefix = 0, mask = 0;
    int need = n_keep;
    bool whole = n_keep >= T;       // every element is kept
    for (int pass = 0; pass < 4 && !whole; ++pass) {
        const int shift = 24 - 8 * pass, cur = pass & 1;
        if (tid < 256) hist[cur ^ 1][tid] = 0;      // the next pass's histogram (last read two barriers ago)
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const bool in = t0 + i < T && (k[i] & mask) == prefix;
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
        __syncthreads();
        if (warp == 0) {
            // lane L owns bins [8L, 8L+8); suffix sums over lanes from the top bin down
            uint32_t c8[8], mine = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c8[j] = hist[cur][lane * 8 + j];
                mine += c8[j];
            }
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
        if (s_whole[cur]) {
            // the threshold bin is kept whole: keep every element whose resolved digits reach the bin
            whole = true;
        }
    }
    // take: above the threshold (resolved digits), or in the threshold bin -- all of it when the bin is kept whole,
    // else the `need` lowest-indexed equal keys (the bin is one key value once all four digits are resolved)
    const bool all_T = n_keep >= T;
    int n_gt = 0, n_eq = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        if (t0 + i >= T) break;
        const uint32_t u = k[i] & mask;
        if (all_T || u > prefix || (whole && u == prefix)) ++n_gt;
        else if (u == prefix) ++n_eq;
    }
    // block-wide exclusive scan of (n_gt, n_eq)
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
        wsum_gt[lane] = a - wsum_gt[lane];     // exclusive prefix over warps
        wsum_eq[lane] = c - wsum_eq[lane];
    }
    __syncthreads();
    const int gt_before = wsum_gt[warp] + gi - n_gt, eq_before = wsum_eq[warp] + ei - n_eq;
    int at = gt_before + min(need, eq_before);
    int eq_rank = eq_before;
    int32_t* hit = want_hit ? x.hit + (int64_t)row * n_keep : nullptr;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const int t = t0 + i;
        if (t >= T) break;
        const uint32_t u = k[i] & mask;
        bool take = all_T || u > prefix || (whole && u == prefix);
        if (!take && u == prefix) take = eq_rank++ < need;
        if (take) {
            o[at] = t;
            if (want_hit) {
                int lo = 0, hi = x.n_res - 1, found = -1;
                while (lo <= hi) {
                    const int mid = (lo + hi) >> 1;
                    const int v = (int)dyn[mid];
                    if (v == t) {
                        found = mid;
                        break;
                    }
                    if (v < t) lo = mid + 1;
                    else hi = mid - 1;
                }
                hit[at] = found;
            }
            ++at;
        }
    }
}

size_t select_scratch_bytes(int, int, int) { return 0; }

cudaError_t launch_select_topn(int P, int T, int n_keep, const float* values, int32_t* out, cudaStream_t st,
                               int32_t* zero_cnt, int32_t* hit, const int32_t* res_idx, int n_res, uint32_t* check,
                               const FoldArgs* fold) {
    if (P == 0) return cudaSuccess;
    SelectExtras x{zero_cnt, (hit && n_res > 0) ? hit : nullptr, res_idx, n_res, check, P, FoldArgs{}};
    if (fold) x.fold = *fold;
    const int nf = fold_blocks(x.fold);
    const size_t fold_smem = nf ? fold_smem_bytes(x.fold.d) : 0;
    const dim3 grid((unsigned)(P + nf));
    if (T <= 32 * kSelThreads) {
        // register-resident rows; the residual list (n_res <= T ints) or the fold's tiles in dynamic shared memory
        size_t smem = x.hit ? sizeof(uint32_t) * (size_t)n_res : 0;
        if (fold_smem > smem) smem = fold_smem;
        auto go = [&](auto kern) -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)(sizeof(uint32_t) * 32 * kSelThreads));
            if (e != cudaSuccess) return e;
            e = launch_pdl(kern, grid, dim3(kSelThreads), smem, st, T, n_keep, values, out, x);
            return e != cudaSuccess ? e : cudaGetLastError();
        };
        if (T <= 4 * kSelThreads) return go(select_reg_kernel<4>);
        if (T <= 8 * kSelThreads) return go(select_reg_kernel<8>);
        if (T <= 16 * kSelThreads) return go(select_reg_kernel<16>);
        return go(select_reg_kernel<32>);
    }
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
