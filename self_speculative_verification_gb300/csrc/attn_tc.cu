// Tensor-core verify-attention kernel: not yet enabled in this build.
#include "attn_tc.cuh"

namespace sv {

bool tc_supported(const AttnParams &, int) { return false; }

int tc_rows_per_block(const AttnParams &) { return 64; }

spec_status_t launch_attn_tc(const AttnParams &, cudaStream_t) { return SPEC_ERR_UNSUPPORTED; }

}  // namespace sv
