// predict_fit.h -- launchers of the test-time fit of the value predictor (predict_fit.cu, tc_predict_fit.cu): loss
// and gradient of every kv-head's MLP over the prompt's (pre-RoPE key, value) pairs, and one Adam step on a flat
// parameter array.
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
// The same loss and gradient with the five products on the tensor cores (tc_predict_fit.cu), in scratch of
// predictor_tc_scratch_bytes; launch_predictor_prep_tc writes the keys' terms into it once per fit (the keys do not
// change between steps).  A pipeline timeout sets LOWRAM_CHECK_TIMEOUT in *check.
size_t predictor_tc_scratch_bytes(int64_t N, int H_kv, int d, int m);
int64_t predictor_tc_max_tokens();   // B*T above it: LOWRAM_ERR_UNSUPPORTED
cudaError_t launch_predictor_prep_tc(const PredictorFitArgs& a, void* scratch, cudaStream_t st);
cudaError_t launch_predictor_grad_tc(const PredictorFitArgs& a, void* scratch, uint32_t* check, cudaStream_t st);
cudaError_t launch_adam(float* p, const float* g, float* mom, float* vel, int64_t n, float lr, float beta1, float beta2,
                        float eps, int step, cudaStream_t st);

}  // namespace lowram
