// evict.h -- launchers of the heavy-hitter eviction plan (evict.cu): attention mass of an observation window over
// the prompt's tokens, and the kept tokens (sinks, recents, heaviest).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace lowram {

size_t mass_workspace_bytes(int B, int T, int W, int H_q, int H_kv, int d, int dtype);
cudaError_t launch_attention_mass(int B, int T, int W, int H_q, int H_kv, int d, int dtype, float scale,
                                  const void* q_win, const void* k, float* mass, void* scratch, uint32_t* check,
                                  cudaStream_t st);

// tc_evict.cu: the window logits on the tensor cores (bf16).  Token tiles of 128, chunk_tiles of them per CTA;
// the window query-heads of each kv-head packed into qp [B, H_kv, NQpad, d] (NQpad = W*g rounded up to 128).
int window_tc_chunk_tiles(int B, int T);
int window_tc_n_chunks(int B, int T);
int window_tc_qpad(int W, int H_q, int H_kv);
cudaError_t launch_pack_window(int B, int W, int H_q, int H_kv, int d, const void* q_win, void* qp, cudaStream_t st);
// mass_pass false: part[b, chunk, i*H_q + hq] = (max, sum of exp) of the scaled logits over the chunk's tokens;
// mass_pass true: mass[b, t] = sum over window query-heads of exp(scaled logit - lse[b, i*H_q + hq]).
cudaError_t launch_window_tc(bool mass_pass, int B, int T, int W, int H_q, int H_kv, int d, float scale,
                             const void* qp, const void* k, float2* part, const float* lse, float* mass,
                             uint32_t* check, cudaStream_t st);
cudaError_t launch_evict_plan(int B, int T, int n_sink, int n_recent, int T_keep, const float* mass, float* scores,
                              int32_t* keep, uint32_t* check, cudaStream_t st);

}  // namespace lowram
