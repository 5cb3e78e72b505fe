// evict.h -- launchers of the heavy-hitter eviction plan (evict.cu): attention mass of an observation window over
// the prompt's tokens, and the kept tokens (sinks, recents, heaviest).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace lowram {

size_t mass_workspace_bytes(int B, int T, int W, int H_q, int H_kv, int d, int dtype);
cudaError_t launch_attention_mass(int B, int T, int W, int H_q, int H_kv, int d, int dtype, float scale,
                                  const void* q_win, const void* k, float* mass, void* scratch, cudaStream_t st);
cudaError_t launch_evict_plan(int B, int T, int n_sink, int n_recent, int T_keep, const float* mass, float* scores,
                              int32_t* keep, uint32_t* check, cudaStream_t st);

}  // namespace lowram
