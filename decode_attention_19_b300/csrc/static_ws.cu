// static_ws.cu -- lowram_decode_attn_static: the decode call for callers that cannot allocate device
// memory.
//
// Some callers of this library cannot call cudaMalloc or hand over a workspace: code that runs inside
// another runtime's memory pool or arena (which owns every allocation and forbids outside ones),
// plug-ins loaded into a host that gives them no allocator, and code paths that must not allocate
// between setup and teardown.  For them this entry point takes the same inputs and outputs as
// lowram_decode_attn, but its scratch (selection keys, selected indices, softmax partials and the
// device check word) lives in one file-scope device array of kStaticBytes bytes that every GPU loading
// the library holds until the process exits.  Nothing here calls cudaMalloc, cudaFree or any allocating
// library routine.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kStaticBytes = (size_t)32 << 20;   // 32 MiB
constexpr int kMaxDevices = 64;

// The scratch array.  In host code this name is a host-side stand-in, not a device address: host code
// must use the address cudaGetSymbolAddress returns for the current device.  A module's __device__ arrays
// start zeroed, so the device check word in its first bytes starts clear.
static __device__ __align__(256) unsigned char g_static_ws[kStaticBytes];

std::mutex g_mu[kMaxDevices];
void* g_addr[kMaxDevices] = {};

// With the caller's device current: the array's device address on that device.  Only a successful lookup
// is kept; a failed one (during a stream capture, say) is retried by the next call.
cudaError_t static_scratch(void** addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu[dev]);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
    }
    *addr = g_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" LOWRAM_API lowram_status lowram_decode_attn_static(
    const lowram_decode_shape* shape, const void* q, const void* coef, const void* coef_scale, const int32_t* pos,
    const float* rope_cos, const float* rope_sin, const void* basis, const void* w1, const void* w2, const float* b1,
    const float* b2, const int32_t* res_idx, const void* res_val, const void* res_scale, float* out, float* lse,
    int32_t* sel_out, float* key_out, void* stream) {
    size_t need = 0;
    lowram_status st = lowram_decode_workspace_size(shape, &need);
    if (st != LOWRAM_OK) return st;
    if (need > kStaticBytes) {
        lowram::set_error_message("lowram_decode_attn_static: this shape needs %zu bytes of scratch, more than the "
                                  "%zu bytes (32 MiB) of the static scratch; use lowram_decode_attn with a workspace",
                                  need, kStaticBytes);
        return LOWRAM_ERR_WORKSPACE;
    }
    void* ws = nullptr;
    cudaError_t e = static_scratch(&ws);
    if (e != cudaSuccess || ws == nullptr) {
        lowram::set_error_message("lowram_decode_attn_static: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
        return LOWRAM_ERR_CUDA;
    }
    // the device check word is sticky across calls until lowram_decode_attn_static_get_error reads it; the rest of
    // the scratch is written before it is read
    return lowram_decode_attn(shape, q, coef, coef_scale, pos, rope_cos, rope_sin, basis, w1, w2, b1, b2, res_idx,
                              res_val, res_scale, out, lse, sel_out, key_out, ws, kStaticBytes, stream);
}

extern "C" LOWRAM_API lowram_status lowram_decode_attn_static_get_error(void* stream, uint32_t* check_word) {
    if (!check_word) {
        lowram::set_error_message("lowram_decode_attn_static_get_error: check_word is NULL");
        return LOWRAM_ERR_INVALID_ARG;
    }
    void* ws = nullptr;
    cudaError_t e = static_scratch(&ws);
    if (e != cudaSuccess || ws == nullptr) {
        lowram::set_error_message("lowram_decode_attn_static_get_error: cudaGetSymbolAddress failed: %s",
                                  cudaGetErrorString(e));
        return LOWRAM_ERR_CUDA;
    }
    return lowram_get_error(ws, stream, check_word);
}
