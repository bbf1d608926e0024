// Planning kernels: row-metadata validation, row blocks, work units, the
// unit schedule, and validation of every page-table entry a window covers --
// all before any K-cache byte is loaded ("[FlyDSL] Add FP4 LiteTopK prefill
// operator", ROCm/aiter#5309, Implementation: fail closed on invalid
// metadata/pages; "[FlyDSL][DSv4] Prototype FP4 MQA streaming TopK",
// ROCm/aiter#5282, Validation: empty windows, nonzero starts, speculative page
// lookahead).
#include <cuda_runtime.h>
#include <stdint.h>

#include "idx_device.cuh"
#include "idx_launch.h"

namespace idxk {

namespace {

constexpr int kRowsPerThread = 8;
constexpr int kPlanThreads = 1024;      // calls of more than kPlanSmallRows rows
// decode-sized calls: 4 warps (their block-wide scans and barriers are cheaper;
// at 1024 rows the extra tiles of the block loops cost more than that saves)
constexpr int kPlanThreadsSmall = 128;
constexpr int kPlanSmallRows = 256;
static_assert(kPlanSmallRows <= kPlanThreadsSmall * kRowsPerThread, "one tile of rows");
constexpr int kLenClasses = 64;  // length classes of the longest-first schedule order

template <typename T, typename Op>
__device__ T block_scan_incl(T v, T* warp_tot, Op op, T identity) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = op(v, u);
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    T w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : identity;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w = op(w, u);
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  if (warp > 0) v = op(v, warp_tot[warp - 1]);
  __syncthreads();
  return v;
}

struct AddI64 {
  __device__ int64_t operator()(int64_t a, int64_t b) const { return a + b; }
};
struct MaxI32 {
  __device__ int32_t operator()(int32_t a, int32_t b) const { return a > b ? a : b; }
};

template <int NT>
__global__ void __launch_bounds__(NT, 1) plan_kernel(PlanParams p) {
  __shared__ int64_t s_tot64[32];
  __shared__ int32_t s_tot32[32];
  __shared__ int64_t s_carry_blocks;
  __shared__ int32_t s_carry_seg;
  const int tid = threadIdx.x;
  PlanHeader* hdr = p.hdr;
  // small calls keep the block table in shared memory as well (phases 3 and
  // 4 read it there instead of from global memory)
  constexpr bool kCache = NT == kPlanThreadsSmall;
  __shared__ BlockInfo s_blk[kCache ? kPlanSmallRows : 1];
  if (p.clear_hdr) {
    // the call's first kernel starts from an empty header (status kOk, no
    // claims); saves a separate clear on the stream
    if (tid == 0) *hdr = PlanHeader{};
    __syncthreads();
  } else if (read_status(hdr) != kOk) {
    return;  // an earlier kernel of the call failed (the same value in every thread)
  }

  // 1. row metadata (the CTA's own verdict decides, not a read of the status)
  bool bad = false;
  for (int r = tid; r < p.rows; r += NT) {
    int32_t req = p.row_req[r], s = p.row_start[r], e = p.row_end[r];
    bool ok = req >= 0 && req < p.num_req && s >= 0 && e >= s &&
              (int64_t)e <= (int64_t)p.max_pages * kPage && (p.check_end_le < 0 || e <= p.check_end_le);
    if (!ok) {
      raise_status(hdr, kErrInvalidMetadata, 100);
      bad = true;
    }
  }
  if (__syncthreads_or(bad)) return;

  // 2. row blocks: a block starts at a request change or every kRowsPerBlock
  //    rows into a run of one request.
  if (tid == 0) {
    s_carry_blocks = 0;
    s_carry_seg = 0;
  }
  __syncthreads();
  for (int64_t base = 0; base < p.rows; base += (int64_t)NT * kRowsPerThread) {
    const int64_t r0 = base + (int64_t)tid * kRowsPerThread;
    // the thread's rows' requests, loaded once: rq[k + 1] is row r0 + k's, rq[0]
    // the previous row's (-1 before row 0 and past the last row)
    int32_t rq[kRowsPerThread + 1];
    rq[0] = (r0 > 0 && r0 <= p.rows) ? p.row_req[r0 - 1] : -1;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) rq[k + 1] = r0 + k < p.rows ? p.row_req[r0 + k] : -1;
    int32_t last_seg = -1;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
      int64_t r = r0 + k;
      if (r < p.rows && (r == 0 || rq[k + 1] != rq[k])) last_seg = (int32_t)r;
    }
    int32_t incl = block_scan_incl<int32_t>(last_seg, s_tot32, MaxI32(), -1);
    int32_t excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if ((tid & 31) == 0) excl = (tid >> 5) > 0 ? s_tot32[(tid >> 5) - 1] : -1;
    int32_t seg = excl >= 0 ? excl : s_carry_seg;
    int64_t nstart = 0;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
      int64_t r = r0 + k;
      if (r >= p.rows) break;
      if (r == 0 || rq[k + 1] != rq[k]) seg = (int32_t)r;
      if (((int32_t)r - seg) % kRowsPerBlock == 0) ++nstart;
    }
    int64_t bincl = block_scan_incl<int64_t>(nstart, s_tot64, AddI64(), 0);
    int64_t b = s_carry_blocks + bincl - nstart;
    seg = excl >= 0 ? excl : s_carry_seg;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
      int64_t r = r0 + k;
      if (r >= p.rows) break;
      if (r == 0 || rq[k + 1] != rq[k]) seg = (int32_t)r;
      if (((int32_t)r - seg) % kRowsPerBlock == 0) {
        BlockInfo bi{};
        bi.row0 = (int32_t)r;
        bi.req = rq[k + 1];
        p.blocks[b] = bi;
        if (kCache) s_blk[b] = bi;
        ++b;
      }
      p.row_block[r] = (int32_t)(b - 1);
    }
    __syncthreads();
    if (tid == NT - 1) {
      s_carry_blocks += bincl;
      int64_t last = base + (int64_t)NT * kRowsPerThread - 1;
      if (last >= p.rows) last = p.rows - 1;
      // segment start of the last row of this tile
      int32_t sg = incl >= 0 ? incl : s_carry_seg;
      (void)last;
      s_carry_seg = sg;
    }
    __syncthreads();
  }
  const int64_t n_blocks = s_carry_blocks;
  __syncthreads();

  // 3. per-block extent and tiles over the scored rows
  int64_t my_tiles = 0;
  for (int64_t b = tid; b < n_blocks; b += NT) {
    BlockInfo bi = kCache ? s_blk[b] : p.blocks[b];
    int32_t next = (b + 1 < n_blocks) ? (kCache ? s_blk[b + 1].row0 : p.blocks[b + 1].row0) : p.rows;
    bi.nrows = next - bi.row0;
    int32_t lo = INT32_MAX, hi = 0;
    for (int j = 0; j < bi.nrows; ++j) {
      int32_t s = p.row_start[bi.row0 + j], e = p.row_end[bi.row0 + j];
      if (e - s > p.score_thr) {
        lo = min(lo, s);
        hi = max(hi, e);
      }
    }
    if (hi > 0 && lo < hi) {
      bi.tile0 = lo / kTile;
      bi.ntiles = (hi + kTile - 1) / kTile - bi.tile0;
    } else {
      bi.tile0 = 0;
      bi.ntiles = 0;
    }
    my_tiles += bi.ntiles;
    p.blocks[b] = bi;
    if (kCache) {  // the fields this phase computes (row0, read by the neighbour, stays)
      s_blk[b].nrows = bi.nrows;
      s_blk[b].tile0 = bi.tile0;
      s_blk[b].ntiles = bi.ntiles;
    }
  }
  int64_t tot_tiles = block_scan_incl<int64_t>(my_tiles, s_tot64, AddI64(), 0);
  if (tid == NT - 1) s_tot64[0] = tot_tiles;
  __syncthreads();
  tot_tiles = s_tot64[0];
  __syncthreads();
  int64_t target = (int64_t)kUnitsPerCta * p.grid;
  int64_t unit_tiles = (tot_tiles + target - 1) / target;
  if (unit_tiles < kMinUnitTiles) unit_tiles = kMinUnitTiles;
  // a block has fewer than 2^31 tiles: 32-bit arithmetic from here on
  const int32_t ut = unit_tiles > INT32_MAX ? INT32_MAX : (int32_t)unit_tiles;

  // 4. units per block and candidate row-slots (blocks handled in tiles of
  //    NT with a running carry)
  __shared__ int64_t s_unit_carry, s_slot_carry;
  __shared__ int32_t s_len_min, s_len_max;  // unit lengths in tiles
  if (tid == 0) {
    s_unit_carry = 0;
    s_slot_carry = 0;
    s_len_min = INT32_MAX;
    s_len_max = 0;
  }
  __syncthreads();
  for (int64_t base = 0; base < n_blocks; base += NT) {
    int64_t b = base + tid;
    int64_t nu = 0, ns = 0;
    BlockInfo bi{};
    if (b < n_blocks) {
      bi = kCache ? s_blk[b] : p.blocks[b];
      nu = bi.ntiles > 0 ? bi.ntiles / ut + (bi.ntiles % ut != 0) : 0;
      ns = nu * bi.nrows;
    }
    int64_t u_incl = block_scan_incl<int64_t>(nu, s_tot64, AddI64(), 0);
    int64_t u_first = s_unit_carry + u_incl - nu;
    int64_t s_incl = block_scan_incl<int64_t>(ns, s_tot64, AddI64(), 0);
    int64_t s_first = s_slot_carry + s_incl - ns;
    if (b < n_blocks) {
      if (u_first + nu > p.max_units || s_first + ns > p.max_row_slots) {
        raise_status(hdr, kErrInternal, 110);
        bad = true;
      } else {
        bi.n_units = (int32_t)nu;
        bi.unit_first = (int32_t)u_first;
        bi.slot0 = s_first;
        p.blocks[b] = bi;
        int32_t lmin = INT32_MAX, lmax = 0;
        // unit k covers tiles tile0 + floor(k * ntiles / nu) .. of the next
        // unit: with ntiles = q * nu + rr that is k * q + floor(k * rr / nu),
        // whose second term grows by 0 or 1 per unit (the remainder k * rr mod
        // nu is carried along, no division per unit)
        const int32_t nu32 = (int32_t)nu;
        const int32_t q = nu32 > 0 ? bi.ntiles / nu32 : 0, rr = nu32 > 0 ? bi.ntiles % nu32 : 0;
        int32_t t_beg = bi.tile0, rem = 0;
        for (int32_t k = 0; k < nu32; ++k) {
          rem += rr;
          const int32_t step = q + (rem >= nu32 ? 1 : 0);
          if (rem >= nu32) rem -= nu32;
          UnitInfo u;
          u.block = (int32_t)b;
          u.k = k;
          u.t_begin = t_beg;
          u.t_end = t_beg + step;
          t_beg = u.t_end;
          p.units[u_first + k] = u;
          lmin = min(lmin, step);
          lmax = max(lmax, step);
        }
        if (nu > 0) {
          atomicMin(&s_len_min, lmin);
          atomicMax(&s_len_max, lmax);
        }
      }
    }
    __syncthreads();
    if (tid == NT - 1) {
      s_unit_carry += u_incl;
      s_slot_carry += s_incl;
    }
    __syncthreads();
  }
  const int64_t n_units = s_unit_carry;
  if (__syncthreads_or(bad)) return;

  // 5. schedule: longest units first (the scorer deals them to its persistent
  //    CTAs band by band, alternating the direction, or its CTAs claim them in
  //    this order).  With no more units than CTAs every unit starts at once and
  //    the order cannot matter.  Units of nearly equal length (longest <= 1.25
  //    x shortest) are not ordered: the alternating deal balances them in any
  //    order, and they are dealt last block first (a request's later rows have
  //    the longer causal windows, so this is close to longest first and keeps
  //    the short ones for the last, partial band).  Otherwise the order is by
  //    kLenClasses length classes of equal width, longest class first (a count
  //    per class, a scan, then each unit to the next free position of its
  //    class): within a class the lengths differ by less than 1/kLenClasses of
  //    the longest unit, and their order is not fixed.
  const bool spread = 4ll * s_len_max > 5ll * s_len_min;
  if (n_units > p.grid && spread) {
    __shared__ uint32_t s_cls[kLenClasses];
    const int32_t width = (s_len_max + kLenClasses) / kLenClasses;  // ceil((max + 1) / classes)
    auto cls_of = [&](int64_t i) -> int {
      const UnitInfo u = p.units[i];
      return kLenClasses - 1 - (u.t_end - u.t_begin) / width;
    };
    for (int c = tid; c < kLenClasses; c += NT) s_cls[c] = 0;
    __syncthreads();
    for (int64_t i = tid; i < n_units; i += NT) atomicAdd(&s_cls[cls_of(i)], 1u);
    __syncthreads();
    if (tid < 32) {  // exclusive scan of the class counts, two per lane
      static_assert(kLenClasses == 64, "two classes per lane");
      const uint32_t a = s_cls[2 * tid], b = s_cls[2 * tid + 1];
      uint32_t x = a + b;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (tid >= o) x += y;
      }
      s_cls[2 * tid] = x - (a + b);
      s_cls[2 * tid + 1] = x - b;
    }
    __syncthreads();
    for (int64_t i = tid; i < n_units; i += NT)
      p.sched[atomicAdd(&s_cls[cls_of(i)], 1u)] = (int32_t)i;
  } else if (n_units > p.grid) {
    for (int64_t i = tid; i < n_units; i += NT) p.sched[i] = (int32_t)(n_units - 1 - i);
  } else {
    for (int64_t i = tid; i < n_units; i += NT) p.sched[i] = (int32_t)i;
  }
  if (tid == 0) {
    hdr->n_blocks = (int32_t)n_blocks;
    hdr->n_units = (int32_t)n_units;
    hdr->unit_tiles = (int32_t)unit_tiles;
    hdr->n_row_slots = s_slot_carry;
  }
}

// Failure-detection diagnostic: one CTA waits through the bounded mbarrier
// wait that every kernel of the library uses.  The phase is completed by the
// CTA's own thread 0 (never == 0), or by nothing (never != 0): the wait then
// gives up after its time limit, records kErrTimeout and the kernel returns.
// Nothing else is in flight, so the context stays usable.
__global__ void __launch_bounds__(64) wait_probe_kernel(PlanHeader* hdr, int never) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (!never && threadIdx.x == 0) mbar_arrive(b);
  if (threadIdx.x < 32) mbar_wait(b, 0, &abort_flag, hdr, 900);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_probe(PlanHeader* hdr, bool never, cudaStream_t stream) {
  wait_probe_kernel<<<1, 64, 0, stream>>>(hdr, never ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream) {
  // (the page-table entries are checked where they are read: by the scorer's
  // producers for the scored rows, by the finishing step's mapping for the rest)
  if (p.rows <= kPlanSmallRows)
    plan_kernel<kPlanThreadsSmall><<<1, kPlanThreadsSmall, 0, stream>>>(p);
  else
    plan_kernel<kPlanThreads><<<1, kPlanThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace idxk
