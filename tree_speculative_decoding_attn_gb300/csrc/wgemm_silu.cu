// Weight-streaming GEMM instances: the Medusa FC1 step (bf16 SiLU + residual
// epilogue).
#include "wgemm_kernel.cuh"

namespace sv {
namespace wg {

int launch_silu(const SvGemmPlan &p, const CUtensorMap *maps, const WArgs &a, bool pdl, cudaStream_t stream) {
  return launch_nt<kEpiSiluRes>(p, maps, a, pdl, stream);
}

}  // namespace wg
}  // namespace sv
