// Tensor-core verify-attention kernel (bf16): entry points used by the
// planner in verify_attn.cu.
#pragma once

#include "attn_common.cuh"

namespace sv {

// Whether the tensor-core kernel takes this shape (dtype = SPEC_*).
bool tc_supported(const AttnParams &P, int dtype);

// Packed rows per CTA of the tensor-core kernel for this shape.
int tc_rows_per_block(const AttnParams &P);

// Workspace bytes of the tensor-core path; *off_ml receives the byte offset
// of the (m, l) partials (the O partials start at offset 0).
size_t tc_workspace_bytes(const AttnParams &P, size_t *off_ml);

// Launch the tensor-core split kernel and its combine kernel.
spec_status_t launch_attn_tc(const AttnParams &P, cudaStream_t s);

}  // namespace sv
