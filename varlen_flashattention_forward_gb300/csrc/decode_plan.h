// decode_plan.h -- host-side planning and launch of one sparse-MLA decode
// call, split so that an entry point can supply the partial-result
// workspace itself.  The plan lives in caller storage (no heap use).
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

#include "../../include/fa_gb300.h"

namespace fa {

constexpr size_t kDecodePlanBytes = 512;

// Checks the arguments of fa_sparse_mla_decode and plans the call into
// `plan` (kDecodePlanBytes of 128-byte-aligned storage): Q tensor map, kernel
// arguments, work split.  *launch = false when there is nothing to run;
// *workspace_bytes = device memory the launch needs for partial results (0:
// none).  Performs the per-device first-call queries; launches nothing.
fa_status decode_plan(const void* q, const void* kv_cache, const int* page_table,
                      const int* topk_idx, int num_tokens, int num_heads, int topk,
                      int num_pages, int max_pages_per_tok, float softmax_scale, void* out,
                      float* lse, void* plan, size_t* workspace_bytes, bool* launch);

// Launches a planned call on `stream`; `workspace` must hold the planned
// workspace_bytes when that is not 0 and must not be used by anything else
// until the launches have completed.
fa_status decode_launch(void* plan, void* workspace, cudaStream_t stream);

}  // namespace fa
