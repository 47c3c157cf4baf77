// Weight-streaming GEMM instances: the Medusa FC1 step (bf16 SiLU + residual
// epilogue), alone or chained with the vocabulary projection in one launch.
#include "wgemm_kernel.cuh"

namespace sv {
namespace wg {

int launch_silu(const SvGemmPlan &p, const CUtensorMap *maps, const WArgs &a, bool pdl, cudaStream_t stream) {
  return launch_nt<kEpiSiluRes, -1>(p, maps, a, pdl, stream);
}

int launch_silu_f32(const SvGemmPlan &p, const CUtensorMap *maps, const WArgs &a, bool pdl, cudaStream_t stream) {
  return launch_nt<kEpiSiluRes, kEpiF32>(p, maps, a, pdl, stream);
}

}  // namespace wg
}  // namespace sv
