// tc_decode.cu -- tensor-core (tcgen05) kernels of the decode path for bf16 / int4 caches.
#include "kernels.h"

namespace lowram {

bool tc_supported(const DecodeArgs&) { return false; }
size_t tc_scratch_bytes(const lowram_decode_shape&) { return 0; }
cudaError_t launch_score_tc(const DecodeArgs&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_vregen_tc(const DecodeArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace lowram
