// Weight-streaming GEMM instances: softmax-statistics records (fused LM head + acceptance).
#include "wgemm_kernel.cuh"

namespace sv {
namespace wg {

int launch_stats(const SvGemmPlan &p, const CUtensorMap *maps, const WArgs &a, bool pdl, cudaStream_t stream) {
  return launch_nt<kEpiStats>(p, maps, a, pdl, stream);
}

}  // namespace wg
}  // namespace sv
