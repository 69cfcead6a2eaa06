// bf16-operand instantiations of the CUDA-core grouped GEMM (fp32 accumulate),
// and the mixed fp32 x bf16 weight-gradient form used by the router.
#include "gemm_simt.cuh"

namespace moe {

cudaError_t launch_gemm_simt_bf16(const GemmArgs& g, cudaStream_t st) {
  using namespace simt;
  if (g.a_type == 0 && g.b_type == 1) {
    if (g.ragged_k && g.epi == EPI_STORE) return launch_form<float, bf16, 2, EPI_STORE>(g, st);
    return cudaErrorInvalidValue;
  }
  return launch_expert_forms<bf16, bf16>(g, st);
}

}  // namespace moe
