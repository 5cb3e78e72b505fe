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
};

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
    const float* v = values + (int64_t)row * T;
    int32_t* o = out + (int64_t)row * n_keep;
    grid_dep_trigger();
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

size_t select_scratch_bytes(int, int, int) { return 0; }

cudaError_t launch_select_topn(int P, int T, int n_keep, const float* values, int32_t* out, cudaStream_t st,
                               int32_t* zero_cnt, int32_t* hit, const int32_t* res_idx, int n_res, uint32_t* check) {
    if (P == 0) return cudaSuccess;
    const SelectExtras x{zero_cnt, (hit && n_res > 0) ? hit : nullptr, res_idx, n_res, check};
    if (n_keep > 0 && T <= kSelMaxStaged) {
        const size_t smem = sizeof(uint32_t) * (size_t)T;   // also holds the residual list (n_res <= T)
        cudaError_t e = cudaFuncSetAttribute(select_topn_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(sizeof(uint32_t) * kSelMaxStaged));
        if (e != cudaSuccess) return e;
        e = launch_pdl(select_topn_kernel<true>, dim3((unsigned)P), dim3(kSelThreads), smem, st, T, n_keep, values, out, x);
        if (e != cudaSuccess) return e;
    } else {
        cudaError_t e = launch_pdl(select_topn_kernel<false>, dim3((unsigned)P), dim3(kSelThreads), 0, st, T, n_keep,
                                   values, out, x);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace lowram
