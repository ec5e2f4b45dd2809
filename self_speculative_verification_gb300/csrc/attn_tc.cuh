// Tensor-core verify-attention kernel (bf16): entry points used by the
// planner in verify_attn.cu.
#pragma once

#include "attn_common.cuh"

namespace sv {

// Whether the tensor-core kernel takes this shape (dtype = SPEC_*).
bool tc_supported(const AttnParams &P, int dtype);

// Packed rows per CTA of the tensor-core kernel for this shape.
int tc_rows_per_block(const AttnParams &P);

// Launch the tensor-core split kernel (partials only; the combine runs after).
spec_status_t launch_attn_tc(const AttnParams &P, cudaStream_t s);

}  // namespace sv
