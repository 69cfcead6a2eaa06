// fp32 instantiations of the CUDA-core grouped GEMM.
#include "gemm_simt.cuh"

namespace moe {

cudaError_t launch_gemm_simt_f32(const GemmArgs& g, cudaStream_t st) {
  return simt::launch_expert_forms<float, float>(g, st);
}

}  // namespace moe
