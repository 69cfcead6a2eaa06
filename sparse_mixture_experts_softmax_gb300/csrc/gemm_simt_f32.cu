// fp32 instantiations of the CUDA-core grouped GEMM, and the router's
// dX = dlogits W_g product with the scatter-back of the expert rows fused in.
#include "gemm_simt.cuh"

namespace moe {

cudaError_t launch_gemm_simt_f32(const GemmArgs& g, cudaStream_t st) {
  using namespace simt;
  if (g.epi == EPI_SCATTER_ADD && !g.ragged_k && !g.b_kcontig)
    return launch_form<float, float, 1, EPI_SCATTER_ADD>(g, st);
  return launch_expert_forms<float, float>(g, st);
}

}  // namespace moe
