// lowram_abi.cu -- the C ABI of liblowram.so: argument and alignment checks, workspace carving,
// and the launch sequence of each call.  See include/lowram.h for the contract of every entry point.
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "kernels.h"
#include "predict_fit.h"
#include "evict.h"

using namespace lowram;

namespace {

// A named NVTX range around a library call or one stage of its launch sequence, for timeline tools (Nsight Systems,
// Nsight Compute's range filters); without a tool attached a push and a pop cost a call through a null hook each.
struct Range {
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range&) = delete;
    Range& operator=(const Range&) = delete;
};

thread_local char g_msg[512] = "";

// Pipeline wait limit of the tensor-core value pass in SM clock cycles (0: the kernels' default of ~1 s); set by
// lowram_set_wait_limit, a testing aid for the timeout path.
long long g_wait_cycles = 0;

lowram_status fail(lowram_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

lowram_status cuda_fail(cudaError_t e, const char* where) {
    return fail(LOWRAM_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

constexpr size_t kHeader = 256;
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool is_act(int dt) { return dt == LOWRAM_F32 || dt == LOWRAM_BF16; }

// Kernels that give each sequence its own grid row (y or z) take at most 65535 sequences per call, and token
// rows b*T + t are 32-bit TMA coordinates and loop indices, so B*T stays below 2^31.
constexpr int32_t kMaxGridRows = 65535;
lowram_status check_grid_rows(int32_t B) {
    return B > kMaxGridRows ? fail(LOWRAM_ERR_UNSUPPORTED, "B=%d > %d sequences per call", B, kMaxGridRows) : LOWRAM_OK;
}
lowram_status check_token_rows(int32_t B, int32_t T) {
    return (int64_t)B * T > (int64_t)INT32_MAX
               ? fail(LOWRAM_ERR_UNSUPPORTED, "B*T=%lld token rows per call (below 2^31)", (long long)B * T)
               : LOWRAM_OK;
}

// ------------------------------------------------------------------------------------------------
// decode
// ------------------------------------------------------------------------------------------------
lowram_status check_decode_shape(const lowram_decode_shape* s) {
    if (!s) return fail(LOWRAM_ERR_INVALID_ARG, "shape is NULL");
    if (s->B < 0 || s->T < 0 || s->S < 0 || s->n_res < 0)
        return fail(LOWRAM_ERR_INVALID_ARG, "negative size (B=%d T=%d S=%d n_res=%d)", s->B, s->T, s->S, s->n_res);
    if (check_grid_rows(s->B) != LOWRAM_OK || check_token_rows(s->B, s->T) != LOWRAM_OK) return LOWRAM_ERR_UNSUPPORTED;
    if (s->H_kv < 1 || s->H_q < 1 || s->H_q % s->H_kv != 0)
        return fail(LOWRAM_ERR_INVALID_ARG, "H_q=%d must be a positive multiple of H_kv=%d", s->H_q, s->H_kv);
    if (s->H_q / s->H_kv > 8) return fail(LOWRAM_ERR_UNSUPPORTED, "H_q/H_kv=%d > 8", s->H_q / s->H_kv);
    if (s->d != 64 && s->d != 128) return fail(LOWRAM_ERR_UNSUPPORTED, "d=%d (64 or 128 supported)", s->d);
    if (s->r < 32 || s->r % 32 != 0 || s->r > 1024)
        return fail(LOWRAM_ERR_UNSUPPORTED, "r=%d (multiple of 32, <= 1024)", s->r);
    if (s->m < 32 || s->m % 32 != 0 || s->m > 256)
        return fail(LOWRAM_ERR_UNSUPPORTED, "m=%d (multiple of 32, <= 256)", s->m);
    if (s->n_res > s->T) return fail(LOWRAM_ERR_INVALID_ARG, "n_res=%d > T=%d", s->n_res, s->T);
    if (!is_act(s->act_dtype)) return fail(LOWRAM_ERR_INVALID_ARG, "act_dtype=%d", s->act_dtype);
    if (s->coef_dtype == LOWRAM_F32 || s->coef_dtype == LOWRAM_BF16) {
        if (s->coef_dtype != s->act_dtype)
            return fail(LOWRAM_ERR_UNSUPPORTED, "coef_dtype %d must equal act_dtype %d", s->coef_dtype, s->act_dtype);
    } else if (s->coef_dtype != LOWRAM_INT4_G32) {
        return fail(LOWRAM_ERR_INVALID_ARG, "coef_dtype=%d", s->coef_dtype);
    }
    if (s->res_dtype != LOWRAM_F32 && s->res_dtype != LOWRAM_BF16 && s->res_dtype != LOWRAM_INT8_VEC)
        return fail(LOWRAM_ERR_INVALID_ARG, "res_dtype=%d", s->res_dtype);
    if (s->T > 0 && s->max_pos < 1) return fail(LOWRAM_ERR_INVALID_ARG, "max_pos=%d", s->max_pos);
    if ((int64_t)s->B * s->T * s->r > ((int64_t)1 << 40)) return fail(LOWRAM_ERR_UNSUPPORTED, "cache too large");
    const int64_t nb = (int64_t)s->H_kv * s->d * s->r, nm = (int64_t)s->H_kv * s->m * s->d;
    if (s->basis_batch_stride != 0 && (s->basis_batch_stride < nb || s->basis_batch_stride % 8 != 0))
        return fail(LOWRAM_ERR_INVALID_ARG, "basis_batch_stride=%lld (0, or >= H_kv*d*r = %lld and a multiple of 8)",
                    (long long)s->basis_batch_stride, (long long)nb);
    if (s->mlp_batch_stride != 0 && (s->mlp_batch_stride < nm || s->mlp_batch_stride % 8 != 0))
        return fail(LOWRAM_ERR_INVALID_ARG, "mlp_batch_stride=%lld (0, or >= H_kv*m*d = %lld and a multiple of 8)",
                    (long long)s->mlp_batch_stride, (long long)nm);
    if (s->flags & ~LOWRAM_FLAG_INT4_EXACT_SPLIT) return fail(LOWRAM_ERR_INVALID_ARG, "flags=0x%x", s->flags);
    return LOWRAM_OK;
}

struct DecodeLayout {
    bool tc_score, tc_vregen;
    bool split;                 // int4 cache run on the tensor cores through the exact bf16 split (dequant.cu)
    bool f16;                   // int4 cache run on the tensor cores through an fp16 copy (the default)
    lowram_decode_shape sx;     // the shape the kernels see: with split, bf16 coefficients of rank 2r; with f16,
                                // fp16 coefficients (kCoefF16) and an fp16 basis
    int chunk, n_chunks, S_eff, PW;
    size_t off_key, off_sel, off_partial, off_sall, off_hit, off_fold, off_asplit, off_bsplit, total;
};

DecodeLayout decode_layout(const lowram_decode_shape& s) {
    DecodeLayout L{};
    L.S_eff = s.S < s.T ? s.S : s.T;
    L.sx = s;
    if (s.coef_dtype == LOWRAM_INT4_G32 && s.act_dtype == LOWRAM_BF16) {
        lowram_decode_shape x = s;
        const bool exact = (s.flags & LOWRAM_FLAG_INT4_EXACT_SPLIT) != 0;
        x.coef_dtype = exact ? LOWRAM_BF16 : kCoefF16;
        x.r = exact ? 2 * s.r : s.r;
        // the repeated bases [W | W] (or the fp16 bases) are packed in the workspace, one per sequence when they differ
        x.basis_batch_stride = s.basis_batch_stride ? (int64_t)s.H_kv * s.d * x.r : 0;
        if (tc_score_supported(x) && tc_vregen_supported(x)) {
            (exact ? L.split : L.f16) = true;
            L.sx = x;
        }
    }
    L.tc_score = tc_score_supported(L.sx);
    L.tc_vregen = tc_vregen_supported(L.sx);
    L.chunk = L.tc_vregen ? kTcChunk : kSimtChunk;
    L.n_chunks = (int)cdiv(L.S_eff, L.chunk);
    L.PW = L.tc_vregen ? tc_partial_width(L.sx) : s.d + 2;
    size_t off = kHeader;
    L.off_key = off;
    off += align256(sizeof(float) * (size_t)s.B * s.H_kv * s.T);
    L.off_sel = off;
    off += align256(sizeof(int32_t) * (size_t)s.B * s.H_kv * L.S_eff);
    L.off_partial = off;
    off += align256(sizeof(float) * (size_t)s.B * s.H_q * L.n_chunks * L.PW);
    L.off_sall = off;
    off += L.tc_vregen ? align256(sizeof(float) * (size_t)s.B * s.H_q * s.T) : 0;
    L.off_hit = off;
    off += L.tc_vregen ? align256(sizeof(int32_t) * (size_t)s.B * s.H_kv * L.S_eff) : 0;
    L.off_fold = off;
    const size_t copies = (s.basis_batch_stride || s.mlp_batch_stride) ? (size_t)s.B : 1;
    off += L.tc_vregen ? align256(sizeof(uint16_t) * copies * s.H_kv * s.m * L.sx.r) : 0;
    L.off_asplit = off;
    off += (L.split || L.f16) ? align256(sizeof(uint16_t) * (size_t)s.B * s.T * L.sx.r) : 0;
    L.off_bsplit = off;
    off += (L.split || L.f16)
               ? align256(sizeof(uint16_t) * (s.basis_batch_stride ? (size_t)s.B : 1) * s.H_kv * s.d * L.sx.r)
               : 0;
    L.total = off;
    return L;
}

}  // namespace

namespace lowram {
// Set the calling thread's lowram_last_error() message (for entry points defined in other files).
void set_error_message(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
}
}  // namespace lowram

extern "C" {

int32_t lowram_version(void) { return 200; }

lowram_status lowram_set_wait_limit(int64_t cycles) {
    if (cycles < 0) return fail(LOWRAM_ERR_INVALID_ARG, "cycles=%lld", (long long)cycles);
    g_wait_cycles = (long long)cycles;
    return LOWRAM_OK;
}

const char* lowram_last_error(void) { return g_msg; }

const char* lowram_status_string(lowram_status st) {
    switch (st) {
        case LOWRAM_OK: return "ok";
        case LOWRAM_ERR_INVALID_ARG: return "invalid argument";
        case LOWRAM_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case LOWRAM_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case LOWRAM_ERR_WORKSPACE: return "workspace missing or too small";
        case LOWRAM_ERR_CUDA: return "CUDA error";
        case LOWRAM_ERR_DEVICE_CHECK: return "device check failed";
    }
    return "unknown status";
}

lowram_status lowram_decode_workspace_size(const lowram_decode_shape* shape, size_t* bytes) {
    lowram_status st = check_decode_shape(shape);
    if (st != LOWRAM_OK) return st;
    if (!bytes) return fail(LOWRAM_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = decode_layout(*shape).total;
    return LOWRAM_OK;
}

lowram_status lowram_decode_uses_tensor_cores(const lowram_decode_shape* shape, int32_t* yes) {
    lowram_status st = check_decode_shape(shape);
    if (st != LOWRAM_OK) return st;
    if (!yes) return fail(LOWRAM_ERR_INVALID_ARG, "yes is NULL");
    *yes = decode_layout(*shape).tc_score ? 1 : 0;
    return LOWRAM_OK;
}

lowram_status lowram_rope_table(int32_t d, double theta, int32_t max_pos, float* cos_out, float* sin_out,
                                void* stream) {
    const Range nvtx_range(__func__);
    if (d <= 0 || d % 2 || max_pos < 0 || !(theta > 0.0)) return fail(LOWRAM_ERR_INVALID_ARG, "d=%d max_pos=%d theta=%g", d, max_pos, theta);
    if (max_pos == 0) return LOWRAM_OK;
    if (!cos_out || !sin_out) return fail(LOWRAM_ERR_INVALID_ARG, "NULL table pointer");
    cudaError_t e = launch_rope_table(d, theta, max_pos, cos_out, sin_out, (cudaStream_t)stream);
    return e == cudaSuccess ? LOWRAM_OK : cuda_fail(e, "rope_table");
}

static lowram_status decode_impl(const lowram_decode_shape* shape, const void* q, const void* coef,
                                 const void* coef_scale, const int32_t* pos, const float* rope_cos,
                                 const float* rope_sin, const void* basis, const void* w1, const void* w2,
                                 const float* b1, const float* b2, const int32_t* res_idx, const void* res_val,
                                 const void* res_scale, float* out, float* lse, int32_t* sel_out, float* key_out,
                                 void* workspace, size_t workspace_bytes, void* stream, void* const* events) {
    lowram_status st = check_decode_shape(shape);
    if (st != LOWRAM_OK) return st;
    const lowram_decode_shape& s = *shape;
    const cudaStream_t cs = (cudaStream_t)stream;
    const bool any = (int64_t)s.B * s.H_q > 0;
    if (any && !out) return fail(LOWRAM_ERR_INVALID_ARG, "out is NULL");
    if ((int64_t)s.B * s.T > 0) {
        if (!q || !coef || !rope_cos || !rope_sin || !basis || !w1 || !w2)
            return fail(LOWRAM_ERR_INVALID_ARG, "a required tensor pointer is NULL");
        if (s.coef_dtype == LOWRAM_INT4_G32 && !coef_scale) return fail(LOWRAM_ERR_INVALID_ARG, "coef_scale is NULL");
        if (s.n_res > 0 && (!res_idx || !res_val)) return fail(LOWRAM_ERR_INVALID_ARG, "residual list is NULL");
        if (s.n_res > 0 && s.res_dtype == LOWRAM_INT8_VEC && !res_scale)
            return fail(LOWRAM_ERR_INVALID_ARG, "res_scale is NULL");
    }
    const void* ptrs[] = {q, coef, coef_scale, pos, rope_cos, rope_sin, basis, w1, w2, b1, b2, res_idx, res_val,
                          res_scale, out, lse, sel_out, key_out, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(LOWRAM_ERR_ALIGNMENT, "pointer %p is not 16-byte aligned", p);
    const DecodeLayout L = decode_layout(s);
    if (!workspace || workspace_bytes < L.total)
        return fail(LOWRAM_ERR_WORKSPACE, "workspace %zu bytes, %zu needed", workspace ? workspace_bytes : 0, L.total);

    char* ws = (char*)workspace;
    DecodeArgs a{};
    a.s = L.sx;
    a.g = s.H_q / s.H_kv;
    a.S_eff = L.S_eff;
    a.scale = s.sm_scale > 0.0f ? s.sm_scale : 1.0f / sqrtf((float)s.d);
    a.q = q; a.coef = coef; a.coef_scale = coef_scale; a.pos = pos;
    a.rope_cos = rope_cos; a.rope_sin = rope_sin; a.basis = basis; a.w1 = w1; a.w2 = w2; a.b1 = b1; a.b2 = b2;
    a.res_idx = res_idx; a.res_val = res_val; a.res_scale = res_scale; a.out = out; a.lse = lse;
    a.key = key_out ? key_out : (float*)(ws + L.off_key);
    a.sel = sel_out ? sel_out : (int32_t*)(ws + L.off_sel);
    a.partial = (float*)(ws + L.off_partial);
    a.n_chunks = L.n_chunks;
    a.PW = L.PW;
    a.sall = L.tc_vregen ? (float*)(ws + L.off_sall) : nullptr;
    a.hit = (L.tc_vregen && s.n_res > 0) ? (int32_t*)(ws + L.off_hit) : nullptr;
    a.fold = L.tc_vregen ? (void*)(ws + L.off_fold) : nullptr;
    a.wait_cycles = g_wait_cycles;
    a.check = (uint32_t*)ws;
    if (L.split || L.f16) {   // the kernels read [hi | lo] and [W | W] (bf16, rank 2r, exactly C W^T), or fp16 copies
        a.coef = ws + L.off_asplit;
        a.coef_scale = nullptr;
        a.basis = ws + L.off_bsplit;
    }

    // optional timing marks: before K1, after K1, after K2, after K3, after K4
    auto mark = [&](int i) -> cudaError_t {
        return (events && events[i]) ? cudaEventRecord((cudaEvent_t)events[i], cs) : cudaSuccess;
    };
    cudaError_t e = mark(0);
    if (e == cudaSuccess && L.split && (int64_t)s.B * s.T > 0) {
        const Range stage("lowram int4 split");
        e = launch_int4_split(coef, coef_scale, (int64_t)s.B * s.T, s.r, ws + L.off_asplit, cs);
        if (e == cudaSuccess)
            e = launch_dup_cols(basis, (int64_t)s.H_kv * s.d, s.r, ws + L.off_bsplit, cs,
                                s.basis_batch_stride ? s.B : 1, s.basis_batch_stride);
        if (e != cudaSuccess) return cuda_fail(e, "int4 split");
    }
    if (e == cudaSuccess && L.f16 && (int64_t)s.B * s.T > 0) {
        const Range stage("lowram int4 to fp16");
        e = launch_int4_f16_copies(coef, coef_scale, (int64_t)s.B * s.T, s.r, ws + L.off_asplit, basis,
                                   (int64_t)s.H_kv * s.d, s.basis_batch_stride ? s.B : 1, s.basis_batch_stride,
                                   ws + L.off_bsplit, cs);
        if (e != cudaSuccess) return cuda_fail(e, "int4 to fp16");
    }
    if (e == cudaSuccess && (int64_t)s.B * s.T > 0 && (L.S_eff > 0 || key_out)) {
        const Range stage("lowram key pass");
        e = L.tc_score ? launch_score_tc(a, cs) : launch_score_simt(a, cs);
    }
    if (e != cudaSuccess) return cuda_fail(e, "score");
    if ((e = mark(1)) != cudaSuccess) return cuda_fail(e, "event");
    // the fold takes bf16 bases: the caller's with an fp16 copy for the kernels, else the ones the kernels read
    const FoldArgs fold{(const __nv_bfloat16*)a.w1, (const __nv_bfloat16*)(L.f16 ? basis : a.basis), a.fold, s.H_kv,
                        s.d, s.m, L.sx.r, (s.basis_batch_stride || s.mlp_batch_stride) ? s.B : 1,
                        L.f16 ? s.basis_batch_stride : L.sx.basis_batch_stride, s.mlp_batch_stride, L.f16};
    if ((int64_t)s.B * L.S_eff > 0) {
        const Range stage("lowram selection");
        e = launch_select_topn(s.B * s.H_kv, s.T, L.S_eff, a.key, a.sel, cs, a.hit, res_idx, s.n_res, a.check,
                               L.tc_vregen ? &fold : nullptr);
    }
    if (e != cudaSuccess) return cuda_fail(e, "select");
    if ((e = mark(2)) != cudaSuccess) return cuda_fail(e, "event");
    if ((int64_t)s.B * L.S_eff > 0) {
        const Range stage("lowram value pass");
        e = L.tc_vregen ? launch_vregen_tc(a, cs) : launch_vregen_simt(a, cs);
    }
    if (e != cudaSuccess) return cuda_fail(e, "vregen");
    if ((e = mark(3)) != cudaSuccess) return cuda_fail(e, "event");
    if (any) {
        const int nc = (int64_t)s.B * L.S_eff > 0 ? L.n_chunks : 0;
        e = launch_merge(s.B, s.H_q, nc, s.d, a.partial, out, lse, cs);
    }
    if (e != cudaSuccess) return cuda_fail(e, "merge");
    if ((e = mark(4)) != cudaSuccess) return cuda_fail(e, "event");
    return LOWRAM_OK;
}

lowram_status lowram_decode_attn(const lowram_decode_shape* shape, const void* q, const void* coef,
                                 const void* coef_scale, const int32_t* pos, const float* rope_cos,
                                 const float* rope_sin, const void* basis, const void* w1, const void* w2,
                                 const float* b1, const float* b2, const int32_t* res_idx, const void* res_val,
                                 const void* res_scale, float* out, float* lse, int32_t* sel_out, float* key_out,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    const Range nvtx_range(__func__);
    return decode_impl(shape, q, coef, coef_scale, pos, rope_cos, rope_sin, basis, w1, w2, b1, b2, res_idx, res_val,
                       res_scale, out, lse, sel_out, key_out, workspace, workspace_bytes, stream, nullptr);
}

lowram_status lowram_decode_attn_events(const lowram_decode_shape* shape, const void* q, const void* coef,
                                        const void* coef_scale, const int32_t* pos, const float* rope_cos,
                                        const float* rope_sin, const void* basis, const void* w1, const void* w2,
                                        const float* b1, const float* b2, const int32_t* res_idx,
                                        const void* res_val, const void* res_scale, float* out, float* lse,
                                        int32_t* sel_out, float* key_out, void* workspace, size_t workspace_bytes,
                                        void* stream, void* const* events) {
    const Range nvtx_range(__func__);
    return decode_impl(shape, q, coef, coef_scale, pos, rope_cos, rope_sin, basis, w1, w2, b1, b2, res_idx, res_val,
                       res_scale, out, lse, sel_out, key_out, workspace, workspace_bytes, stream, events);
}

// ------------------------------------------------------------------------------------------------
// compress
// ------------------------------------------------------------------------------------------------
static lowram_status check_compress_shape(const lowram_compress_shape* s) {
    if (!s) return fail(LOWRAM_ERR_INVALID_ARG, "shape is NULL");
    if (s->B < 0 || s->T < 0 || s->n_res < 0 || s->n_res > s->T)
        return fail(LOWRAM_ERR_INVALID_ARG, "bad sizes (B=%d T=%d n_res=%d)", s->B, s->T, s->n_res);
    if (check_grid_rows(s->B) != LOWRAM_OK || check_token_rows(s->B, s->T) != LOWRAM_OK) return LOWRAM_ERR_UNSUPPORTED;
    if (s->G < 1 || s->G > 16) return fail(LOWRAM_ERR_UNSUPPORTED, "G=%d (1..16)", s->G);
    if (s->H_kv < 1) return fail(LOWRAM_ERR_INVALID_ARG, "H_kv=%d", s->H_kv);
    if (s->d != 64 && s->d != 128) return fail(LOWRAM_ERR_UNSUPPORTED, "d=%d (64 or 128 supported)", s->d);
    if (s->r < 32 || s->r % 32 != 0 || s->r > 1024) return fail(LOWRAM_ERR_UNSUPPORTED, "r=%d", s->r);
    if (s->m < 32 || s->m % 32 != 0 || s->m > 256) return fail(LOWRAM_ERR_UNSUPPORTED, "m=%d", s->m);
    if (!is_act(s->act_dtype)) return fail(LOWRAM_ERR_INVALID_ARG, "act_dtype=%d", s->act_dtype);
    if (s->coef_dtype != LOWRAM_F32 && s->coef_dtype != LOWRAM_BF16 && s->coef_dtype != LOWRAM_INT4_G32)
        return fail(LOWRAM_ERR_INVALID_ARG, "coef_dtype=%d", s->coef_dtype);
    if (s->res_dtype != LOWRAM_F32 && s->res_dtype != LOWRAM_BF16 && s->res_dtype != LOWRAM_INT8_VEC)
        return fail(LOWRAM_ERR_INVALID_ARG, "res_dtype=%d", s->res_dtype);
    if (s->keys_post_rope && s->T > 0 && s->max_pos < 1) return fail(LOWRAM_ERR_INVALID_ARG, "max_pos=%d", s->max_pos);
    return LOWRAM_OK;
}

// ------------------------------------------------------------------------------------------------
// heavy hitters from accumulated attention (eviction plan)
// ------------------------------------------------------------------------------------------------
static lowram_status check_mass_shape(int32_t B, int32_t T, int32_t W, int32_t H_q, int32_t H_kv, int32_t d) {
    if (B < 0 || T < 0 || W < 1 || H_kv < 1 || H_q < 1 || H_q % H_kv != 0)
        return fail(LOWRAM_ERR_INVALID_ARG, "B=%d T=%d W=%d H_q=%d H_kv=%d", B, T, W, H_q, H_kv);
    if (check_grid_rows(B) != LOWRAM_OK || check_token_rows(B, T) != LOWRAM_OK) return LOWRAM_ERR_UNSUPPORTED;
    const int g = H_q / H_kv;
    if (g != 1 && g != 2 && g != 4 && g != 7 && g != 8) return fail(LOWRAM_ERR_UNSUPPORTED, "H_q/H_kv=%d", g);
    if (d != 64 && d != 128) return fail(LOWRAM_ERR_UNSUPPORTED, "d=%d (64 or 128 supported)", d);
    return LOWRAM_OK;
}

lowram_status lowram_attention_mass_workspace_size(int32_t B, int32_t T, int32_t W, int32_t H_q, int32_t H_kv,
                                                   int32_t d, int32_t dtype, size_t* bytes) {
    lowram_status st = check_mass_shape(B, T, W, H_q, H_kv, d);
    if (st != LOWRAM_OK) return st;
    if (!is_act(dtype)) return fail(LOWRAM_ERR_INVALID_ARG, "dtype=%d", dtype);
    if (!bytes) return fail(LOWRAM_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = kHeader + align256(mass_workspace_bytes(B, T, W, H_q, H_kv, d, dtype));
    return LOWRAM_OK;
}

lowram_status lowram_attention_mass(int32_t B, int32_t T, int32_t W, int32_t H_q, int32_t H_kv, int32_t d,
                                    int32_t dtype, float sm_scale, const void* q_win, const void* k, float* mass_out,
                                    void* workspace, size_t workspace_bytes, void* stream) {
    const Range nvtx_range(__func__);
    size_t need = 0;
    lowram_status st = lowram_attention_mass_workspace_size(B, T, W, H_q, H_kv, d, dtype, &need);
    if (st != LOWRAM_OK) return st;
    if (!workspace || workspace_bytes < need || !aligned16(workspace))
        return fail(LOWRAM_ERR_WORKSPACE, "workspace %zu bytes, %zu needed", workspace ? workspace_bytes : 0, need);
    if ((int64_t)B * T == 0) return LOWRAM_OK;
    if (!q_win || !k || !mass_out) return fail(LOWRAM_ERR_INVALID_ARG, "a required pointer is NULL");
    const void* ptrs[] = {q_win, k, mass_out};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(LOWRAM_ERR_ALIGNMENT, "pointer %p is not 16-byte aligned", p);
    const float scale = sm_scale > 0.0f ? sm_scale : 1.0f / sqrtf((float)d);
    const cudaError_t e = launch_attention_mass(B, T, W, H_q, H_kv, d, dtype, scale, q_win, k, mass_out,
                                                (char*)workspace + kHeader, (uint32_t*)workspace, (cudaStream_t)stream);
    return e == cudaSuccess ? LOWRAM_OK : cuda_fail(e, "attention_mass");
}

lowram_status lowram_evict_plan_workspace_size(int32_t B, int32_t T, size_t* bytes) {
    if (B < 0 || T < 0) return fail(LOWRAM_ERR_INVALID_ARG, "B=%d T=%d", B, T);
    if (!bytes) return fail(LOWRAM_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = kHeader + align256(sizeof(float) * (size_t)B * T);
    return LOWRAM_OK;
}

lowram_status lowram_evict_plan(int32_t B, int32_t T, int32_t n_sink, int32_t n_recent, int32_t T_keep,
                                const float* mass, int32_t* keep_out, void* workspace, size_t workspace_bytes,
                                void* stream) {
    const Range nvtx_range(__func__);
    size_t need = 0;
    lowram_status st = lowram_evict_plan_workspace_size(B, T, &need);
    if (st != LOWRAM_OK) return st;
    if (n_sink < 0 || n_recent < 0 || T_keep < 0 || T_keep > T ||
        T_keep < (n_sink + n_recent < T ? n_sink + n_recent : T))
        return fail(LOWRAM_ERR_INVALID_ARG, "n_sink=%d n_recent=%d T_keep=%d T=%d (need sinks + recents <= T_keep <= T)",
                    n_sink, n_recent, T_keep, T);
    if (!workspace || workspace_bytes < need || !aligned16(workspace))
        return fail(LOWRAM_ERR_WORKSPACE, "workspace %zu bytes, %zu needed", workspace ? workspace_bytes : 0, need);
    if ((int64_t)B * T_keep == 0) return LOWRAM_OK;
    if (!mass || !keep_out) return fail(LOWRAM_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!aligned16(mass) || !aligned16(keep_out)) return fail(LOWRAM_ERR_ALIGNMENT, "a pointer is not 16-byte aligned");
    const cudaError_t e = launch_evict_plan(B, T, n_sink, n_recent, T_keep, mass,
                                            (float*)((char*)workspace + kHeader), keep_out, (uint32_t*)workspace,
                                            (cudaStream_t)stream);
    return e == cudaSuccess ? LOWRAM_OK : cuda_fail(e, "evict_plan");
}

// ------------------------------------------------------------------------------------------------
// test-time fit of the value predictor
// ------------------------------------------------------------------------------------------------
static lowram_status check_predictor_shape(int32_t B, int32_t T, int32_t H_kv, int32_t d, int32_t m, int32_t dtype) {
    if (B < 0 || T < 0 || H_kv < 1) return fail(LOWRAM_ERR_INVALID_ARG, "B=%d T=%d H_kv=%d", B, T, H_kv);
    if (check_token_rows(B, T) != LOWRAM_OK) return LOWRAM_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return fail(LOWRAM_ERR_UNSUPPORTED, "d=%d (64 or 128 supported)", d);
    if (m < 32 || m % 32 != 0 || m > 256) return fail(LOWRAM_ERR_UNSUPPORTED, "m=%d", m);
    if (!is_act(dtype)) return fail(LOWRAM_ERR_INVALID_ARG, "dtype=%d", dtype);
    return LOWRAM_OK;
}

static size_t predictor_params(int32_t H_kv, int32_t d, int32_t m) {
    return (size_t)H_kv * ((size_t)2 * m * d + m + d);
}

lowram_status lowram_predictor_grad(int32_t B, int32_t T, int32_t H_kv, int32_t d, int32_t m, int32_t dtype,
                                    const void* keys, const void* values, const float* w1, const float* b1,
                                    const float* w2, const float* b2, float* loss_out, float* g_w1, float* g_b1,
                                    float* g_w2, float* g_b2, void* stream) {
    const Range nvtx_range(__func__);
    lowram_status st = check_predictor_shape(B, T, H_kv, d, m, dtype);
    if (st != LOWRAM_OK) return st;
    const void* need[] = {w1, b1, w2, b2, loss_out, g_w1, g_b1, g_w2, g_b2};
    for (const void* p : need)
        if (!p) return fail(LOWRAM_ERR_INVALID_ARG, "a required pointer is NULL");
    if ((int64_t)B * T > 0 && (!keys || !values)) return fail(LOWRAM_ERR_INVALID_ARG, "keys or values is NULL");
    const void* ptrs[] = {keys, values, w1, b1, w2, b2, loss_out, g_w1, g_b1, g_w2, g_b2};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(LOWRAM_ERR_ALIGNMENT, "pointer %p is not 16-byte aligned", p);
    PredictorFitArgs a{B, T, H_kv, d, m, dtype == LOWRAM_BF16, keys, values, w1, b1, w2, b2, loss_out,
                       g_w1, g_b1, g_w2, g_b2};
    const cudaError_t e = launch_predictor_grad(a, (cudaStream_t)stream);
    return e == cudaSuccess ? LOWRAM_OK : cuda_fail(e, "predictor_grad");
}

lowram_status lowram_fit_predictor_workspace_size(int32_t B, int32_t T, int32_t H_kv, int32_t d, int32_t m,
                                                  size_t* bytes) {
    lowram_status st = check_predictor_shape(B, T, H_kv, d, m, LOWRAM_F32);
    if (st != LOWRAM_OK) return st;
    if ((int64_t)B * T > predictor_tc_max_tokens())
        return fail(LOWRAM_ERR_UNSUPPORTED, "B*T=%lld prompt tokens (at most %lld for the fit)", (long long)B * T,
                    (long long)predictor_tc_max_tokens());
    if (!bytes) return fail(LOWRAM_ERR_INVALID_ARG, "bytes is NULL");
    // gradient, first and second moments of every parameter, a loss row, and the tensor-core products' scratch
    *bytes = kHeader + 3 * align256(sizeof(float) * predictor_params(H_kv, d, m)) + align256(sizeof(float) * H_kv) +
             align256(predictor_tc_scratch_bytes((int64_t)B * T, H_kv, d, m));
    return LOWRAM_OK;
}

lowram_status lowram_fit_predictor(int32_t B, int32_t T, int32_t H_kv, int32_t d, int32_t m, int32_t dtype,
                                   const void* keys, const void* values, int32_t steps, float lr, float beta1,
                                   float beta2, float eps, float* w1, float* b1, float* w2, float* b2,
                                   float* losses_out, void* workspace, size_t workspace_bytes, void* stream) {
    const Range nvtx_range(__func__);
    lowram_status st = check_predictor_shape(B, T, H_kv, d, m, dtype);
    if (st != LOWRAM_OK) return st;
    size_t need = 0;
    if ((st = lowram_fit_predictor_workspace_size(B, T, H_kv, d, m, &need)) != LOWRAM_OK) return st;
    if (!workspace || workspace_bytes < need || !aligned16(workspace))
        return fail(LOWRAM_ERR_WORKSPACE, "workspace %zu bytes, %zu needed", workspace ? workspace_bytes : 0, need);
    if (steps < 0) return fail(LOWRAM_ERR_INVALID_ARG, "steps=%d", steps);
    if (!(lr > 0.0f) || !(beta1 >= 0.0f && beta1 < 1.0f) || !(beta2 >= 0.0f && beta2 < 1.0f) || !(eps > 0.0f))
        return fail(LOWRAM_ERR_INVALID_ARG, "Adam hyper-parameters lr=%g beta1=%g beta2=%g eps=%g", lr, beta1, beta2, eps);
    if (!w1 || !b1 || !w2 || !b2) return fail(LOWRAM_ERR_INVALID_ARG, "a parameter pointer is NULL");
    if ((int64_t)B * T > 0 && (!keys || !values)) return fail(LOWRAM_ERR_INVALID_ARG, "keys or values is NULL");
    const void* ptrs[] = {keys, values, w1, b1, w2, b2, losses_out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(LOWRAM_ERR_ALIGNMENT, "pointer %p is not 16-byte aligned", p);
    const cudaStream_t cs = (cudaStream_t)stream;
    const size_t np = predictor_params(H_kv, d, m), seg = align256(sizeof(float) * np);
    char* ws = (char*)workspace + kHeader;
    float* grad = (float*)ws;
    float* mom = (float*)(ws + seg);
    float* vel = (float*)(ws + 2 * seg);
    float* loss_tmp = (float*)(ws + 3 * seg);
    void* tc_scratch = ws + 3 * seg + align256(sizeof(float) * H_kv);
    uint32_t* check = (uint32_t*)workspace;   // the header's check word: LOWRAM_CHECK_TIMEOUT from the products
    // the four parameter tensors and their slices of the gradient / moment buffers
    const size_t n1 = (size_t)H_kv * m * d, nb1 = (size_t)H_kv * m, nb2 = (size_t)H_kv * d;
    float* params[4] = {w1, b1, w2, b2};
    const size_t count[4] = {n1, nb1, n1, nb2};
    size_t off[4];
    off[0] = 0;
    for (int i = 1; i < 4; ++i) off[i] = off[i - 1] + count[i - 1];
    cudaError_t e = cudaMemsetAsync(mom, 0, 2 * seg, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(check, 0, sizeof(uint32_t), cs);
    if (e == cudaSuccess && steps > 0) {
        const PredictorFitArgs a0{B, T, H_kv, d, m, dtype == LOWRAM_BF16, keys, values, w1, b1, w2, b2, loss_tmp,
                                  grad + off[0], grad + off[1], grad + off[2], grad + off[3]};
        e = launch_predictor_prep_tc(a0, tc_scratch, cs);
    }
    for (int s_ = 0; s_ < steps && e == cudaSuccess; ++s_) {
        PredictorFitArgs a{B, T, H_kv, d, m, dtype == LOWRAM_BF16, keys, values, w1, b1, w2, b2,
                           losses_out ? losses_out + (size_t)s_ * H_kv : loss_tmp, grad + off[0], grad + off[1],
                           grad + off[2], grad + off[3]};
        e = launch_predictor_grad_tc(a, tc_scratch, check, cs);
        for (int i = 0; i < 4 && e == cudaSuccess; ++i)
            e = launch_adam(params[i], grad + off[i], mom + off[i], vel + off[i], (int64_t)count[i], lr, beta1, beta2,
                            eps, s_ + 1, cs);
    }
    return e == cudaSuccess ? LOWRAM_OK : cuda_fail(e, "fit_predictor");
}

// ------------------------------------------------------------------------------------------------
// fitted basis
// ------------------------------------------------------------------------------------------------
static lowram_status check_fit_shape(const lowram_compress_shape* s) {
    if (!s) return fail(LOWRAM_ERR_INVALID_ARG, "shape is NULL");
    if (s->B < 0 || s->T < 0) return fail(LOWRAM_ERR_INVALID_ARG, "bad sizes (B=%d T=%d)", s->B, s->T);
    if (check_token_rows(s->B, s->T) != LOWRAM_OK) return LOWRAM_ERR_UNSUPPORTED;
    if (s->G < 1 || s->G > 16) return fail(LOWRAM_ERR_UNSUPPORTED, "G=%d (1..16)", s->G);
    if (s->H_kv < 1) return fail(LOWRAM_ERR_INVALID_ARG, "H_kv=%d", s->H_kv);
    if (s->d != 64 && s->d != 128) return fail(LOWRAM_ERR_UNSUPPORTED, "d=%d (64 or 128 supported)", s->d);
    const int64_t D = (int64_t)s->G * s->H_kv * s->d;
    if (s->r < 32 || s->r % 32 != 0 || s->r > 1024 || s->r > D) return fail(LOWRAM_ERR_UNSUPPORTED, "r=%d", s->r);
    if (D > 16384) return fail(LOWRAM_ERR_UNSUPPORTED, "G*H_kv*d=%lld (at most 16384)", (long long)D);
    if ((int64_t)s->B * s->T < s->r)
        return fail(LOWRAM_ERR_INVALID_ARG, "B*T=%lld tokens, fewer than the rank r=%d", (long long)s->B * s->T, s->r);
    if (!is_act(s->act_dtype)) return fail(LOWRAM_ERR_INVALID_ARG, "act_dtype=%d", s->act_dtype);
    if (s->keys_post_rope && s->max_pos < 1) return fail(LOWRAM_ERR_INVALID_ARG, "max_pos=%d", s->max_pos);
    return LOWRAM_OK;
}

lowram_status lowram_fit_basis_workspace_size(const lowram_compress_shape* shape, size_t* bytes) {
    lowram_status st = check_fit_shape(shape);
    if (st != LOWRAM_OK) return st;
    if (!bytes) return fail(LOWRAM_ERR_INVALID_ARG, "bytes is NULL");
    const int64_t N = (int64_t)shape->B * shape->T;
    *bytes = kHeader + align256(fit_workspace_bytes(N, shape->G * shape->H_kv * shape->d, shape->r));
    return LOWRAM_OK;
}

lowram_status lowram_fit_basis(const lowram_compress_shape* shape, const void* keys, const int32_t* pos,
                               const float* rope_cos, const float* rope_sin, int32_t iters, uint64_t seed,
                               float* proj_out, void* const* basis_out, void* workspace, size_t workspace_bytes,
                               void* stream) {
    const Range nvtx_range(__func__);
    size_t need = 0;
    lowram_status st = lowram_fit_basis_workspace_size(shape, &need);
    if (st != LOWRAM_OK) return st;
    const lowram_compress_shape& s = *shape;
    if (!workspace || workspace_bytes < need || !aligned16(workspace))
        return fail(LOWRAM_ERR_WORKSPACE, "workspace %zu bytes, %zu needed", workspace ? workspace_bytes : 0, need);
    if (iters < 1 || iters > 1000) return fail(LOWRAM_ERR_INVALID_ARG, "iters=%d (1..1000)", iters);
    if (!keys || !proj_out || !basis_out) return fail(LOWRAM_ERR_INVALID_ARG, "a required pointer is NULL");
    if (s.keys_post_rope && (!rope_cos || !rope_sin)) return fail(LOWRAM_ERR_INVALID_ARG, "RoPE tables are NULL");
    const void* ptrs[] = {keys, pos, rope_cos, rope_sin, proj_out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(LOWRAM_ERR_ALIGNMENT, "pointer %p is not 16-byte aligned", p);
    for (int l = 0; l < s.G; ++l) {
        if (!basis_out[l]) return fail(LOWRAM_ERR_INVALID_ARG, "basis_out[%d] is NULL", l);
        if (!aligned16(basis_out[l])) return fail(LOWRAM_ERR_ALIGNMENT, "basis_out[%d] is not 16-byte aligned", l);
    }
    FitArgs f{};
    f.B = s.B; f.T = s.T; f.G = s.G; f.H_kv = s.H_kv; f.d = s.d; f.r = s.r;
    f.max_pos = s.max_pos; f.post_rope = s.keys_post_rope ? 1 : 0; f.iters = iters;
    f.bf16 = s.act_dtype == LOWRAM_BF16;
    f.seed = seed;
    f.keys = keys; f.pos = pos; f.rope_cos = rope_cos; f.rope_sin = rope_sin;
    f.proj_out = proj_out;
    for (int l = 0; l < s.G; ++l) f.basis_out[l] = basis_out[l];
    f.scratch = (char*)workspace + kHeader;
    f.check = (uint32_t*)workspace;
    const cudaError_t e = launch_fit_basis(f, (cudaStream_t)stream);
    return e == cudaSuccess ? LOWRAM_OK : cuda_fail(e, "fit_basis");
}

lowram_status lowram_compress_workspace_size(const lowram_compress_shape* shape, size_t* bytes) {
    lowram_status st = check_compress_shape(shape);
    if (st != LOWRAM_OK) return st;
    if (!bytes) return fail(LOWRAM_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = kHeader + align256(sizeof(float) * (size_t)shape->B * shape->H_kv * shape->T);
    return LOWRAM_OK;
}

lowram_status lowram_compress(const lowram_compress_shape* shape, const void* keys, const void* const* values,
                              const float* proj, const int32_t* pos, const float* rope_cos, const float* rope_sin,
                              const void* const* basis, const void* const* w1, const void* const* w2,
                              const float* const* b1, const float* const* b2, void* coef_out, void* coef_scale_out,
                              int32_t* const* res_idx_out, void* const* res_val_out, void* const* res_scale_out,
                              float* const* err_out, void* workspace, size_t workspace_bytes, void* stream) {
    const Range nvtx_range(__func__);
    lowram_status st = check_compress_shape(shape);
    if (st != LOWRAM_OK) return st;
    const lowram_compress_shape& s = *shape;
    const cudaStream_t cs = (cudaStream_t)stream;
    size_t need = 0;
    lowram_compress_workspace_size(shape, &need);
    if (!workspace || workspace_bytes < need || !aligned16(workspace))
        return fail(LOWRAM_ERR_WORKSPACE, "workspace %zu bytes, %zu needed", workspace ? workspace_bytes : 0, need);
    if ((int64_t)s.B * s.T == 0) return LOWRAM_OK;
    if (!keys || !values || !proj || !basis || !w1 || !w2 || !coef_out)
        return fail(LOWRAM_ERR_INVALID_ARG, "a required pointer is NULL");
    if (s.coef_dtype == LOWRAM_INT4_G32 && !coef_scale_out) return fail(LOWRAM_ERR_INVALID_ARG, "coef_scale_out is NULL");
    if (s.keys_post_rope && (!rope_cos || !rope_sin)) return fail(LOWRAM_ERR_INVALID_ARG, "RoPE tables are NULL");
    if (s.n_res > 0 && (!res_idx_out || !res_val_out)) return fail(LOWRAM_ERR_INVALID_ARG, "residual outputs are NULL");
    if (s.n_res > 0 && s.res_dtype == LOWRAM_INT8_VEC && !res_scale_out)
        return fail(LOWRAM_ERR_INVALID_ARG, "res_scale_out is NULL");

    CompressArgs a{};
    a.s = s;
    a.keys = keys; a.proj = proj; a.pos = pos; a.rope_cos = rope_cos; a.rope_sin = rope_sin;
    a.coef_out = coef_out; a.coef_scale_out = coef_scale_out;
    a.check = (uint32_t*)workspace;
    a.err_scratch = (float*)((char*)workspace + kHeader);
    const void* top[] = {keys, proj, pos, rope_cos, rope_sin, coef_out, coef_scale_out};
    for (const void* p : top)
        if (p && !aligned16(p)) return fail(LOWRAM_ERR_ALIGNMENT, "pointer %p is not 16-byte aligned", p);
    for (int l = 0; l < s.G; ++l) {
        a.values[l] = values[l]; a.basis[l] = basis[l]; a.w1[l] = w1[l]; a.w2[l] = w2[l];
        a.b1[l] = b1 ? b1[l] : nullptr; a.b2[l] = b2 ? b2[l] : nullptr;
        a.res_idx_out[l] = s.n_res > 0 ? res_idx_out[l] : nullptr;
        a.res_val_out[l] = s.n_res > 0 ? res_val_out[l] : nullptr;
        a.res_scale_out[l] = (s.n_res > 0 && res_scale_out) ? res_scale_out[l] : nullptr;
        a.err_out[l] = err_out ? err_out[l] : nullptr;
        if (!a.values[l] || !a.basis[l] || !a.w1[l] || !a.w2[l])
            return fail(LOWRAM_ERR_INVALID_ARG, "layer %d: a required pointer is NULL", l);
        if (s.n_res > 0 && (!a.res_idx_out[l] || !a.res_val_out[l]))
            return fail(LOWRAM_ERR_INVALID_ARG, "layer %d: residual output is NULL", l);
        if (s.n_res > 0 && s.res_dtype == LOWRAM_INT8_VEC && !a.res_scale_out[l])
            return fail(LOWRAM_ERR_INVALID_ARG, "layer %d: res_scale_out is NULL", l);
        const void* lp[] = {a.values[l], a.basis[l], a.w1[l], a.w2[l], a.b1[l], a.b2[l], a.res_idx_out[l],
                            a.res_val_out[l], a.res_scale_out[l], a.err_out[l]};
        for (const void* p : lp)
            if (p && !aligned16(p)) return fail(LOWRAM_ERR_ALIGNMENT, "layer %d: pointer %p is not 16-byte aligned", l, p);
    }
    cudaError_t e = launch_project(a, cs);
    if (e != cudaSuccess) return cuda_fail(e, "project");
    for (int l = 0; l < s.G; ++l) {
        float* err = a.err_out[l] ? a.err_out[l] : a.err_scratch;
        e = launch_predict_err(a, l, err, cs);
        if (e != cudaSuccess) return cuda_fail(e, "predict_err");
        if (s.n_res > 0) {
            e = launch_select_topn(s.B * s.H_kv, s.T, s.n_res, err, a.res_idx_out[l], cs);
            if (e != cudaSuccess) return cuda_fail(e, "select residuals");
            e = launch_residual_rows(a, l, cs);
            if (e != cudaSuccess) return cuda_fail(e, "residual rows");
        }
    }
    return LOWRAM_OK;
}

// ------------------------------------------------------------------------------------------------
// dense comparator
// ------------------------------------------------------------------------------------------------
lowram_status lowram_dense_workspace_size(int32_t B, int32_t T, int32_t H_q, int32_t H_kv, int32_t d, size_t* bytes) {
    if (B < 0 || T < 0 || H_q < 1 || H_kv < 1 || H_q % H_kv || (d != 64 && d != 128) || !bytes)
        return fail(LOWRAM_ERR_INVALID_ARG, "bad dense shape");
    if (check_grid_rows(B) != LOWRAM_OK || check_token_rows(B, T) != LOWRAM_OK) return LOWRAM_ERR_UNSUPPORTED;
    const int nr = dense_records_max(B, T, H_kv, H_q, d);
    *bytes = kHeader + align256(sizeof(float) * (size_t)B * H_q * nr * (d + 2));
    return LOWRAM_OK;
}

// Attention over explicit K/V rows [B, *, H_kv, d] whose sequence b starts at token b * Ts (Ts = T for a plain
// cache, T_cap for the exact tail's buffers).
static lowram_status dense_impl(int32_t B, int32_t T, int32_t Ts, int32_t H_q, int32_t H_kv, int32_t d,
                                int32_t dtype, float sm_scale, const void* q, const void* k, const void* v, float* out,
                                float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    size_t need = 0;
    lowram_status st = lowram_dense_workspace_size(B, T, H_q, H_kv, d, &need);
    if (st != LOWRAM_OK) return st;
    if (!is_act(dtype)) return fail(LOWRAM_ERR_INVALID_ARG, "dtype=%d", dtype);
    const int g = H_q / H_kv;
    if (g != 1 && g != 2 && g != 4 && g != 7 && g != 8) return fail(LOWRAM_ERR_UNSUPPORTED, "H_q/H_kv=%d", g);
    if (!workspace || workspace_bytes < need) return fail(LOWRAM_ERR_WORKSPACE, "workspace too small (%zu needed)", need);
    if ((int64_t)B * H_q == 0) return LOWRAM_OK;
    if (!out || (T > 0 && (!q || !k || !v))) return fail(LOWRAM_ERR_INVALID_ARG, "a required pointer is NULL");
    const void* ptrs[] = {q, k, v, out, lse, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(LOWRAM_ERR_ALIGNMENT, "pointer %p is not 16-byte aligned", p);
    const cudaStream_t cs = (cudaStream_t)stream;
    const int ns = dense_splits(B, T, H_kv, H_q, d, dtype);
    float* partial = (float*)((char*)workspace + kHeader);
    const float scale = sm_scale > 0.0f ? sm_scale : 1.0f / sqrtf((float)d);
    cudaError_t e = cudaSuccess;
    if (T > 0) {
        e = launch_dense(B, T, Ts, H_q, H_kv, d, dtype, scale, q, k, v, partial, ns, cs);
        if (e != cudaSuccess) return cuda_fail(e, "dense");
    }
    e = launch_merge(B, H_q, T > 0 ? ns : 0, d, partial, out, lse, cs);
    return e == cudaSuccess ? LOWRAM_OK : cuda_fail(e, "merge");
}

lowram_status lowram_dense_decode_attn(int32_t B, int32_t T, int32_t H_q, int32_t H_kv, int32_t d, int32_t dtype,
                                       float sm_scale, const void* q, const void* k, const void* v, float* out,
                                       float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    const Range nvtx_range(__func__);
    return dense_impl(B, T, T, H_q, H_kv, d, dtype, sm_scale, q, k, v, out, lse, workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------------------------------------------
// exact tail
// ------------------------------------------------------------------------------------------------
lowram_status lowram_tail_append(int32_t B, int32_t T_cap, int32_t H_kv, int32_t d, int32_t dtype, int32_t t,
                                 const void* k_new, const void* v_new, void* tail_k, void* tail_v, void* stream) {
    const Range nvtx_range(__func__);
    if (B < 0 || T_cap < 1 || H_kv < 1 || (d != 64 && d != 128))
        return fail(LOWRAM_ERR_INVALID_ARG, "B=%d T_cap=%d H_kv=%d d=%d", B, T_cap, H_kv, d);
    if (!is_act(dtype)) return fail(LOWRAM_ERR_INVALID_ARG, "dtype=%d", dtype);
    if (t < 0 || t >= T_cap) return fail(LOWRAM_ERR_INVALID_ARG, "row t=%d outside the tail's capacity %d", t, T_cap);
    if (B == 0) return LOWRAM_OK;
    if (!k_new || !v_new || !tail_k || !tail_v) return fail(LOWRAM_ERR_INVALID_ARG, "a required pointer is NULL");
    const void* ptrs[] = {k_new, v_new, tail_k, tail_v};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(LOWRAM_ERR_ALIGNMENT, "pointer %p is not 16-byte aligned", p);
    const cudaError_t e = launch_tail_append(B, T_cap, H_kv, d, dtype == LOWRAM_BF16 ? 2 : 4, t, k_new, v_new, tail_k,
                                             tail_v, (cudaStream_t)stream);
    return e == cudaSuccess ? LOWRAM_OK : cuda_fail(e, "tail_append");
}

lowram_status lowram_tail_decode_attn(int32_t B, int32_t T_cap, int32_t t_len, int32_t H_q, int32_t H_kv, int32_t d,
                                      int32_t dtype, float sm_scale, const void* q, const void* tail_k,
                                      const void* tail_v, float* out, float* lse, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    const Range nvtx_range(__func__);
    if (t_len < 0 || t_len > T_cap)
        return fail(LOWRAM_ERR_INVALID_ARG, "t_len=%d outside the tail's capacity %d", t_len, T_cap);
    return dense_impl(B, t_len, T_cap, H_q, H_kv, d, dtype, sm_scale, q, tail_k, tail_v, out, lse, workspace,
                      workspace_bytes, stream);
}

lowram_status lowram_merge_attn(int32_t B, int32_t H_q, int32_t d, const float* out_a, const float* lse_a,
                                const float* out_b, const float* lse_b, float* out, float* lse, void* stream) {
    const Range nvtx_range(__func__);
    if (B < 0 || H_q < 1 || d < 1) return fail(LOWRAM_ERR_INVALID_ARG, "B=%d H_q=%d d=%d", B, H_q, d);
    if (B == 0) return LOWRAM_OK;
    if (!out_a || !lse_a || !out_b || !lse_b || !out) return fail(LOWRAM_ERR_INVALID_ARG, "a required pointer is NULL");
    const void* ptrs[] = {out_a, lse_a, out_b, lse_b, out, lse};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(LOWRAM_ERR_ALIGNMENT, "pointer %p is not 16-byte aligned", p);
    const cudaError_t e = launch_merge_attn(B, H_q, d, out_a, lse_a, out_b, lse_b, out, lse, (cudaStream_t)stream);
    return e == cudaSuccess ? LOWRAM_OK : cuda_fail(e, "merge_attn");
}

// ------------------------------------------------------------------------------------------------
// status
// ------------------------------------------------------------------------------------------------
lowram_status lowram_get_error(void* workspace, void* stream, uint32_t* check_word) {
    if (!workspace || !check_word) return fail(LOWRAM_ERR_INVALID_ARG, "NULL argument");
    const cudaStream_t cs = (cudaStream_t)stream;
    uint32_t w = 0;
    cudaError_t e = cudaMemcpyAsync(&w, workspace, sizeof(w), cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "get_error");
    *check_word = w;
    return w ? fail(LOWRAM_ERR_DEVICE_CHECK, "device check word 0x%x", w) : LOWRAM_OK;
}

lowram_status lowram_clear_error(void* workspace, void* stream) {
    if (!workspace) return fail(LOWRAM_ERR_INVALID_ARG, "workspace is NULL");
    cudaError_t e = cudaMemsetAsync(workspace, 0, kHeader, (cudaStream_t)stream);
    return e == cudaSuccess ? LOWRAM_OK : cuda_fail(e, "clear_error");
}

}  // extern "C"
