// Weight-streaming GEMM instances: float32 logits.
#include "wgemm_kernel.cuh"

namespace sv {
namespace wg {

int launch_f32(const SvGemmPlan &p, const CUtensorMap *maps, const WArgs &a, bool pdl, cudaStream_t stream) {
  return launch_nt<kEpiF32>(p, maps, a, pdl, stream);
}

}  // namespace wg
}  // namespace sv
