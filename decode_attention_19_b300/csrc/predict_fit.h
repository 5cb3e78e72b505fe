// predict_fit.h -- launchers of the test-time fit of the value predictor (predict_fit.cu): loss and gradient of
// every kv-head's MLP over the prompt's (pre-RoPE key, value) pairs, and one Adam step on a flat parameter array.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lowram {

struct PredictorFitArgs {
    int B, T, H_kv, d, m;
    bool bf16;
    const void* keys;      // [B, T, H_kv, d]
    const void* values;    // [B, T, H_kv, d]
    const float *w1, *b1, *w2, *b2;          // [H_kv, m, d], [H_kv, m], [H_kv, d, m], [H_kv, d]
    float* loss;                             // [H_kv]
    float *g_w1, *g_b1, *g_w2, *g_b2;        // shaped like the parameters
};
cudaError_t launch_predictor_grad(const PredictorFitArgs& a, cudaStream_t st);
cudaError_t launch_adam(float* p, const float* g, float* mom, float* vel, int64_t n, float lr, float beta1, float beta2,
                        float eps, int step, cudaStream_t st);

}  // namespace lowram
