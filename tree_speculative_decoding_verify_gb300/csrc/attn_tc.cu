// tcgen05 / TMEM / TMA tree-verification attention (bf16, head_dim 128).
#include "attn_common.cuh"
#include "common.cuh"

namespace tsv {

bool tc_supported(const AttnPlan& p) { return false; }

int launch_attn_tc(const AttnPlan&, const AttnArgs&, float, void*, cudaStream_t) {
  return TSV_ERR_UNSUPPORTED;
}

}  // namespace tsv
