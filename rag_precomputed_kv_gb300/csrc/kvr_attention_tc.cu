// kvr_attention_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) query prefill attention.
#include "kvr_internal.cuh"

namespace kvr {

bool attention_tc_supported(int, int) { return false; }

cudaError_t launch_attention_tc(const TcAttnArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace kvr
