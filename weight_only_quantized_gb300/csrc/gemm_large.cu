// Large-M GEMM (prefill): tcgen05 / TMEM / TMA kernel.  Not yet part of this build; gptq_gemm
// routes every M to the small-M kernel (which tiles M by 16) until it is.
#include "internal.cuh"

namespace gptq {

bool large_m_available() { return false; }
int large_m_launches(const Handle&, int) { return -1; }
cudaError_t launch_gemm_large(const Handle&, const void*, void*, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gptq
