// Row finishing: exact merge of the per-unit candidates of a row (or exact
// TopK of a materialised fp32 score row), ordering by the total order, the
// short-row contract and the raw -> physical slot mapping.
//
// "[FlyDSL][DSv4] Prototype FP4 MQA streaming TopK" (ROCm/aiter#5282,
// Changes): merge split candidates exactly, then map raw C4 positions through
// the page table; when length <= topk return every logical position in order,
// padded with -1.  The dense variant is the separate TopK of the legacy
// full-logits path (same page, Motivation).
#include <cuda_runtime.h>
#include <stdint.h>

#include "idx_device.cuh"
#include "idx_launch.h"
#include "idx_select.cuh"

namespace idxk {

namespace {

constexpr int kFinThreads = 256;
constexpr int kFinCap = 4096;
constexpr int kFinPer = 4;  // keys per thread per batch
constexpr int kFinBatch = kFinThreads * kFinPer;
constexpr uint32_t kFinBar = 1;

__device__ __forceinline__ int32_t map_phys(const int32_t* row_pt, int32_t raw) {
  if (raw < 0 || row_pt == nullptr) return -1;
  const int64_t v = (int64_t)row_pt[raw >> 6] * kPage + (raw & (kPage - 1));
  return (int32_t)v;
}

template <int TOPK, bool DENSE>
__global__ void __launch_bounds__(kFinThreads) finish_kernel(FinishParams p) {
  __shared__ __align__(16) uint64_t buf[kFinCap];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t bc[4];
  __shared__ uint32_t cnt;
  __shared__ uint64_t tau;
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  if (read_status(p.hdr) != kOk) return;
  const int32_t s0 = p.row_start[r], s1 = p.row_end[r];
  const int64_t len = (int64_t)s1 - s0;
  const int32_t* row_pt =
      p.page_table ? p.page_table + (int64_t)p.row_req[r] * p.max_pages : nullptr;
  int32_t* out_raw = p.out_raw ? p.out_raw + (int64_t)r * TOPK : nullptr;
  int32_t* out_phys = p.out_phys ? p.out_phys + (int64_t)r * TOPK : nullptr;

  if (len <= TOPK) {
    for (int i = tid; i < TOPK; i += kFinThreads) {
      const int32_t raw = i < len ? s0 + i : -1;
      if (out_raw) out_raw[i] = raw;
      if (out_phys) out_phys[i] = map_phys(row_pt, raw);
    }
    return;
  }

  if (tid == 0) {
    cnt = 0;
    tau = 0;
  }
  __syncthreads();
  uint64_t t = 0;
  if constexpr (DENSE) {
    const float* src = p.scores + (int64_t)r * p.score_stride;
    for (int64_t base = s0; base < s1; base += kFinBatch) {
      bool over = false;
#pragma unroll
      for (int e = 0; e < kFinPer; ++e) {
        const int64_t s = base + e * kFinThreads + tid;
        const bool in = s < s1;
        const float v = in ? src[s] : 0.f;
        const uint64_t key = order_key(v, (int32_t)s);
        over |= sel_append(buf, &cnt, kFinCap, kFinCap - kFinBatch, in && key >= t, key);
      }
      if (bar_red_or(kFinBar, kFinThreads, over)) {
        sel_compact<kFinThreads, kFinCap>(buf, &cnt, &tau, hist, bc, TOPK, tid, kFinBar, p.hdr);
        t = *(volatile uint64_t*)&tau;
      }
    }
  } else {
    const BlockInfo bi = p.blocks[p.row_block[r]];
    const int j = r - bi.row0;
    for (int k = 0; k < bi.n_units; ++k) {
      const int64_t slot = bi.slot0 + (int64_t)k * bi.nrows + j;
      const uint32_t n = min(p.cand_cnt[slot], (uint32_t)TOPK);
      const uint64_t* keys = p.cand_keys + slot * TOPK;
      for (uint32_t base = 0; base < n; base += kFinBatch) {
        bool over = false;
#pragma unroll
        for (int e = 0; e < kFinPer; ++e) {
          const uint32_t i = base + e * kFinThreads + tid;
          const bool in = i < n;
          const uint64_t key = in ? keys[i] : 0ull;
          over |= sel_append(buf, &cnt, kFinCap, kFinCap - kFinBatch, in && key >= t, key);
        }
        if (bar_red_or(kFinBar, kFinThreads, over)) {
          sel_compact<kFinThreads, kFinCap>(buf, &cnt, &tau, hist, bc, TOPK, tid, kFinBar, p.hdr);
          t = *(volatile uint64_t*)&tau;
        }
      }
    }
  }
  __syncthreads();
  sel_compact<kFinThreads, kFinCap>(buf, &cnt, &tau, hist, bc, TOPK, tid, kFinBar, p.hdr);
  const uint32_t n = min(*(volatile uint32_t*)&cnt, (uint32_t)TOPK);
  if (n < (uint32_t)TOPK) {
    // a window longer than topk must yield topk candidates
    if (tid == 0) raise_status(p.hdr, kErrInternal, 400);
    for (int i = n + tid; i < TOPK; i += kFinThreads) buf[i] = 0ull;
  }
  __syncthreads();
  // bitonic sort, descending by key (score desc, then index asc)
  for (int size = 2; size <= TOPK; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < TOPK / 2; i += kFinThreads) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const uint64_t a = buf[lo], c = buf[hi];
        const bool desc = (lo & size) == 0;
        if (desc ? (a < c) : (a > c)) {
          buf[lo] = c;
          buf[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int i = tid; i < TOPK; i += kFinThreads) {
    const uint64_t key = buf[i];
    const int32_t raw = key != 0ull ? key_index(key) : -1;
    if (out_raw) out_raw[i] = raw;
    if (out_phys) out_phys[i] = map_phys(row_pt, raw);
  }
}

// Row windows of a bare score matrix: 0 <= start <= end <= width.
__global__ void validate_windows_kernel(const int32_t* row_start, const int32_t* row_end,
                                        int32_t rows, int64_t width, PlanHeader* hdr) {
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows;
       r += (int64_t)gridDim.x * blockDim.x) {
    const int32_t s = row_start[r], e = row_end[r];
    if (s < 0 || e < s || (int64_t)e > width) raise_status(hdr, kErrInvalidMetadata, 410);
  }
}

template <int TOPK, bool DENSE>
cudaError_t launch_t(const FinishParams& p, cudaStream_t stream) {
  finish_kernel<TOPK, DENSE><<<p.rows, kFinThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_finish(const FinishParams& p, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  const bool dense = p.scores != nullptr;
  if (p.topk == 512) return dense ? launch_t<512, true>(p, stream) : launch_t<512, false>(p, stream);
  if (p.topk == 1024)
    return dense ? launch_t<1024, true>(p, stream) : launch_t<1024, false>(p, stream);
  return cudaErrorInvalidValue;
}

namespace {
// Windows of one context chunk [c0, c1): rows longer than topk keep the part
// of their window inside the chunk; shorter rows (closed form) get none.
__global__ void clip_windows_kernel(const int32_t* row_start, const int32_t* row_end, int32_t rows,
                                    int32_t c0, int32_t c1, int32_t topk, int32_t* out_start,
                                    int32_t* out_end) {
  for (int32_t r = blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x) {
    const int32_t s0 = row_start[r], s1 = row_end[r];
    int32_t a = s0 > c0 ? s0 : c0, b = s1 < c1 ? s1 : c1;
    if ((int64_t)s1 - s0 <= topk || a > b) a = b = s0;
    out_start[r] = a;
    out_end[r] = b;
  }
}

// One CTA per row: the row's running TopK (keys in run_keys, count run_cnt,
// threshold run_tau) absorbs the chunk's materialised scores
// (chunk[r * stride + s - c0] for s in the clipped window); after the last
// chunk the keys are sorted and written like the merge of the fused path.
template <int TOPK>
__global__ void __launch_bounds__(kFinThreads) tile_merge_kernel(TileMergeParams p) {
  __shared__ __align__(16) uint64_t buf[kFinCap];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t bc[4];
  __shared__ uint32_t cnt;
  __shared__ uint64_t tau;
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  if (read_status(p.hdr) != kOk) return;
  const int32_t s0 = p.row_start[r], s1 = p.row_end[r];
  const int64_t len = (int64_t)s1 - s0;
  const int32_t* row_pt = p.page_table + (int64_t)p.row_req[r] * p.max_pages;
  if (len <= TOPK) {
    if (!p.last) return;
    for (int i = tid; i < TOPK; i += kFinThreads) {
      const int32_t raw = i < len ? s0 + i : -1;
      if (p.out_raw) p.out_raw[(int64_t)r * TOPK + i] = raw;
      p.out_phys[(int64_t)r * TOPK + i] = map_phys(row_pt, raw);
    }
    return;
  }
  uint64_t* run = p.run_keys + (int64_t)r * TOPK;
  const uint32_t n_run = p.first ? 0u : p.run_cnt[r];
  uint64_t t = p.first ? 0ull : p.run_tau[r];
  for (uint32_t i = tid; i < n_run; i += kFinThreads) buf[i] = run[i];
  if (tid == 0) {
    cnt = n_run;
    tau = t;
  }
  __syncthreads();
  const int32_t a = s0 > p.c0 ? s0 : p.c0, b = s1 < p.c1 ? s1 : p.c1;
  const float* src = p.chunk + (int64_t)r * p.stride - p.c0;
  for (int64_t base = a; base < b; base += kFinBatch) {
    bool over = false;
#pragma unroll
    for (int e = 0; e < kFinPer; ++e) {
      const int64_t s = base + e * kFinThreads + tid;
      const bool in = s < b;
      const float v = in ? src[s] : 0.f;
      const uint64_t key = order_key(v, (int32_t)s);
      over |= sel_append(buf, &cnt, kFinCap, kFinCap - kFinBatch, in && key >= t, key);
    }
    if (bar_red_or(kFinBar, kFinThreads, over)) {
      sel_compact<kFinThreads, kFinCap>(buf, &cnt, &tau, hist, bc, TOPK, tid, kFinBar, p.hdr);
      t = *(volatile uint64_t*)&tau;
    }
  }
  __syncthreads();
  sel_compact<kFinThreads, kFinCap>(buf, &cnt, &tau, hist, bc, TOPK, tid, kFinBar, p.hdr);
  const uint32_t n = min(*(volatile uint32_t*)&cnt, (uint32_t)TOPK);
  if (!p.last) {
    for (uint32_t i = tid; i < n; i += kFinThreads) run[i] = buf[i];
    if (tid == 0) {
      p.run_cnt[r] = n;
      p.run_tau[r] = *(volatile uint64_t*)&tau;
    }
    return;
  }
  if (n < (uint32_t)TOPK) {
    if (tid == 0) raise_status(p.hdr, kErrInternal, 401);
    for (int i = n + tid; i < TOPK; i += kFinThreads) buf[i] = 0ull;
  }
  __syncthreads();
  for (int size = 2; size <= TOPK; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < TOPK / 2; i += kFinThreads) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const uint64_t x = buf[lo], y = buf[hi];
        const bool desc = (lo & size) == 0;
        if (desc ? (x < y) : (x > y)) {
          buf[lo] = y;
          buf[hi] = x;
        }
      }
      __syncthreads();
    }
  }
  for (int i = tid; i < TOPK; i += kFinThreads) {
    const uint64_t key = buf[i];
    const int32_t raw = key != 0ull ? key_index(key) : -1;
    if (p.out_raw) p.out_raw[(int64_t)r * TOPK + i] = raw;
    p.out_phys[(int64_t)r * TOPK + i] = map_phys(row_pt, raw);
  }
}
}  // namespace

cudaError_t launch_clip_windows(const int32_t* row_start, const int32_t* row_end, int32_t rows,
                                int32_t c0, int32_t c1, int32_t topk, int32_t* out_start,
                                int32_t* out_end, cudaStream_t stream) {
  const int grid = rows > 0 ? (rows + 255) / 256 : 1;
  clip_windows_kernel<<<grid, 256, 0, stream>>>(row_start, row_end, rows, c0, c1, topk, out_start,
                                                out_end);
  return cudaGetLastError();
}

cudaError_t launch_tile_merge(const TileMergeParams& p, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  if (p.topk == 512) tile_merge_kernel<512><<<p.rows, kFinThreads, 0, stream>>>(p);
  else if (p.topk == 1024) tile_merge_kernel<1024><<<p.rows, kFinThreads, 0, stream>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

namespace {
__global__ void publish_status_kernel(const PlanHeader* hdr, uint32_t* status_out,
                                      int32_t* out_phys, int32_t* out_raw, int64_t n) {
  const uint32_t st = read_status(hdr);
  if (blockIdx.x == 0 && threadIdx.x == 0) *status_out = st;
  if (st == kOk) return;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    out_phys[i] = -1;
    if (out_raw) out_raw[i] = -1;
  }
}
}  // namespace

cudaError_t launch_publish_status(const PlanHeader* hdr, uint32_t* status_out, int32_t* out_phys,
                                  int32_t* out_raw, int64_t n, cudaStream_t stream) {
  const int64_t want = (n + 255) / 256;
  const int grid = (int)(want < 1 ? 1 : (want > 1024 ? 1024 : want));
  publish_status_kernel<<<grid, 256, 0, stream>>>(hdr, status_out, out_phys, out_raw, n);
  return cudaGetLastError();
}

cudaError_t launch_validate_windows(const int32_t* row_start, const int32_t* row_end, int32_t rows,
                                    int64_t width, PlanHeader* hdr, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  int blocks = (rows + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  validate_windows_kernel<<<blocks, 256, 0, stream>>>(row_start, row_end, rows, width, hdr);
  return cudaGetLastError();
}

}  // namespace idxk
