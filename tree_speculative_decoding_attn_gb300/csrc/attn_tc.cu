// Tree attention on the tcgen05 tensor cores (bf16, head_dim 128).
// Not yet enabled: the plan never selects it.
#include "common.cuh"
#include "kernels.h"

SvAttnPlan sv_attn_tc_plan(const SvAttnShape &, int, bool *ok) {
  *ok = false;
  return SvAttnPlan{};
}

int sv_attn_tc(const SvAttnShape &, const SvAttnPlan &, const void *, const void *, const void *,
               const void *, const void *, const int32_t *, const uint64_t *, void *, float,
               void *, int32_t *, cudaStream_t) {
  return SPEC_ERR_UNSUPPORTED;
}
