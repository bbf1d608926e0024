// Host-side launchers of the kernels (one translation unit each), called by the
// C-ABI layer in host.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "idx_internal.h"

namespace idxk {

// plan_kernel (1 CTA) then validate_pages_kernel.
cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream);

// Persistent scoring kernel, `grid` CTAs.  mode kModeSelect writes unit
// candidates (topk 512 or 1024); kModeDense writes scores (and logits).
cudaError_t launch_score(const CUtensorMap& tmap_k, const CUtensorMap& tmap_q,
                         const ScoreParams& p, int grid, cudaStream_t stream);

// Shared-memory bytes the scoring kernel needs for a mode/topk.
size_t score_smem_bytes(int mode, int topk);

// One CTA per row: merge unit candidates (FinishParams::scores == null) or
// select from a dense score matrix; then sort, map and write.
cudaError_t launch_finish(const FinishParams& p, cudaStream_t stream);

// Checks 0 <= start <= end <= width for every row of a bare score matrix.
cudaError_t launch_validate_windows(const int32_t* row_start, const int32_t* row_end, int32_t rows,
                                    int64_t width, PlanHeader* hdr, cudaStream_t stream);

}  // namespace idxk
