// Host-side launchers of the kernels (one translation unit each), called by the
// C-ABI layer in host.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "idx_internal.h"

namespace idxk {

// Sets a kernel's dynamic shared-memory limit once per device (the attribute
// persists, and repeating the call is avoided while a stream is captured).
// Host threads may call at once: the per-device flags are atomic, and two
// threads that both see a flag clear both set the same attribute, which is
// harmless.
template <typename Kernel>
inline cudaError_t set_smem_once(Kernel kernel, int bytes, std::atomic<bool> (&done)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return err;
}

// One CTA waiting through the bounded mbarrier wait on a phase that its own
// thread completes (never = false) or that nothing completes (never = true:
// kErrTimeout is recorded in hdr after the wait limit).
cudaError_t launch_wait_probe(PlanHeader* hdr, bool never, cudaStream_t stream);

// plan_kernel (1 CTA): row validation, blocks, units and their schedule.
cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream);

// Persistent scoring kernel, `grid` CTAs.  mode kModeSelect writes unit
// candidates (topk 512 or 1024); kModeDense writes scores (and logits).
cudaError_t launch_score(const CUtensorMap& tmap_k, const CUtensorMap& tmap_q,
                         const ScoreParams& p, int grid, cudaStream_t stream);

// Shared-memory bytes the scoring kernel needs for a mode/topk.
size_t score_smem_bytes(int mode, int topk);

// One CTA per row: merge unit candidates (FinishParams::scores and shard_raw
// null), select from a dense score matrix (scores set) or from the union of
// context-shard lists (shard_raw set); then sort, map and write.
cudaError_t launch_finish(const FinishParams& p, cudaStream_t stream);

// Checks 0 <= start <= end <= width for every row, and 0 <= row_req < num_req
// when row_req is given.
cudaError_t launch_validate_windows(const int32_t* row_start, const int32_t* row_end, int32_t rows,
                                    int64_t width, PlanHeader* hdr, cudaStream_t stream,
                                    const int32_t* row_req = nullptr, int32_t num_req = 0);

// Context-tiled comparison path: windows of one chunk, and the per-chunk
// merge into each row's running TopK (writing the outputs after the last).
cudaError_t launch_clip_windows(const int32_t* row_start, const int32_t* row_end, int32_t rows,
                                int32_t c0, int32_t c1, int32_t topk, int32_t* out_start,
                                int32_t* out_end, cudaStream_t stream);
cudaError_t launch_tile_merge(const TileMergeParams& p, cudaStream_t stream);

}  // namespace idxk
