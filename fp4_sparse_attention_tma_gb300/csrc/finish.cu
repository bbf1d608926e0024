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
constexpr int kFinGridCap = 2048;  // merging CTAs (rows strided over them)

// Physical slot of position raw of a row (page table row_pt), -1 for raw < 0.
// The entry must name a page in [0, num_pages); one that does not maps to -1
// and sets `bad`, which the caller turns into kErrInvalidPage (the call fails
// closed).  This is the page-table check of the rows the scorer does not score
// (their every position is mapped here); the scorer's producers check the
// entries under the scored rows' windows.  (The windows, hence raw / 64 <
// max_pages, were validated by the plan.)
__device__ __forceinline__ int32_t map_phys(const int32_t* row_pt, int32_t raw, int32_t num_pages,
                                            bool& bad) {
  if (raw < 0 || row_pt == nullptr) return -1;
  const int32_t pg = row_pt[raw >> 6];
  const bool ok = pg >= 0 && pg < num_pages;
  bad |= !ok;
  return ok ? (int32_t)((int64_t)pg * kPage + (raw & (kPage - 1))) : -1;
}

// keep the larger (or smaller) of each register and its partner's
__device__ __forceinline__ uint64_t keep_of(uint64_t x, uint64_t o, bool keep_max) {
  return (x > o) == keep_max ? x : o;  // equal keys: either
}

// One bitonic step at distance S (< E) between a thread's own keys t*E + e.
template <int E, int S>
__device__ __forceinline__ void sort_in_thread(uint64_t (&v)[E], int g0, int size) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if ((e & S) != 0) continue;
    const bool desc = ((g0 + e) & size) == 0;
    const uint64_t a = v[e], b = v[e | S];
    const bool sw = (a < b) == desc;  // equal keys (zero padding) may swap
    v[e] = sw ? b : a;
    v[e | S] = sw ? a : b;
  }
}

// Sorts the row's TOPK keys buf[0, TOPK) descending (score desc, then index
// asc: a bitonic network) and writes the row's outputs.  Thread t holds the E
// consecutive keys t*E .. t*E+E-1 in registers: exchanges at distances below E
// stay in the thread, distances below 32*E go between the lanes of a warp,
// and only the larger ones pass through shared memory.  The caller has filled
// buf[0, TOPK) (zero keys pad an underfilled row) before a barrier.
// SCORES: also write the keys' scores to out_score; DUP: raise on dup_hdr when
// two emitted keys are equal (a position listed twice by the shard merge).
template <int TOPK, bool SCORES = false, bool DUP = false>
__device__ __forceinline__ void sort_emit(uint64_t* buf, int tid, const int32_t* row_pt,
                                          int32_t num_pages, PlanHeader* hdr, int32_t* out_raw,
                                          int32_t* out_phys, float* out_score = nullptr) {
  constexpr int E = TOPK / kFinThreads;
  static_assert(E == 2 || E == 4, "keys per thread");
  const int g0 = tid * E;
  uint64_t v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = buf[g0 + e];
#pragma unroll 1
  for (int size = 2; size <= TOPK; size <<= 1) {
#pragma unroll 1
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride < E) {
        if (stride == 1) {
          sort_in_thread<E, 1>(v, g0, size);
        } else if constexpr (E == 4) {
          sort_in_thread<E, 2>(v, g0, size);
        }
      } else {
        // the pair's lower position keeps the larger key in a descending
        // block, the smaller one in an ascending block; all E keys of a
        // thread share both properties at these distances
        const bool keep_max = ((g0 & stride) == 0) == ((g0 & size) == 0);
        if (stride < 32 * E) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const uint64_t o = __shfl_xor_sync(0xffffffffu, v[e], stride / E);
            v[e] = keep_of(v[e], o, keep_max);
          }
        } else {
          __syncthreads();  // earlier readers of buf are done
#pragma unroll
          for (int e = 0; e < E; ++e) buf[g0 + e] = v[e];
          __syncthreads();
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const uint64_t o = buf[(g0 + e) ^ stride];
            v[e] = keep_of(v[e], o, keep_max);
          }
        }
      }
    }
  }
  if (DUP) {
    // the merge of context-shard lists: a position reported twice would show
    // up as two equal (nonzero) neighbours of the sorted keys
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e) buf[g0 + e] = v[e];
    __syncthreads();
    bool dup = false;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = g0 + e;
      dup |= i + 1 < TOPK && v[e] != 0ull && buf[i + 1] == v[e];
    }
    if (dup) raise_status(hdr, kErrInvalidMetadata, 422);
  }
  int32_t raw[E], phys[E];
  bool bad_page = false;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    raw[e] = v[e] != 0ull ? key_index(v[e]) : -1;
    phys[e] = map_phys(row_pt, raw[e], num_pages, bad_page);
    if (SCORES) out_score[g0 + e] = key_score(v[e]);
  }
  // E consecutive outputs per thread; rows start at multiples of 2 KB of a
  // 16-byte aligned base
  if constexpr (E == 4) {
    if (out_raw) *reinterpret_cast<int4*>(out_raw + g0) = make_int4(raw[0], raw[1], raw[2], raw[3]);
    if (out_phys)
      *reinterpret_cast<int4*>(out_phys + g0) = make_int4(phys[0], phys[1], phys[2], phys[3]);
  } else {
    if (out_raw) *reinterpret_cast<int2*>(out_raw + g0) = make_int2(raw[0], raw[1]);
    if (out_phys) *reinterpret_cast<int2*>(out_phys + g0) = make_int2(phys[0], phys[1]);
  }
  if (bad_page) raise_status(hdr, kErrInvalidPage, 440);
}

// A row whose block ran as a single work unit has at most TOPK candidates, all
// of them the row's TopK, so it needs only the sort.  A team of TOPK / 512
// warps per row holds the keys in registers (16 per lane: key
// g = 512 * warp + 16 * lane + e of the sorting network in register e) and
// runs the bitonic network: distances below 16 within a lane, below 512
// between the lanes of a warp, 512 (TOPK = 1024 only) through shared memory
// between the team's two warps.  The teams also handle every short row
// (length <= TOPK: start .. end-1, then -1).  Rows of multi-unit blocks are
// left to merge_rows.
constexpr int kTeamThreads = 256;
constexpr int kTeamE = 16;          // keys per lane
constexpr int kTeamKeys = 32 * kTeamE;

// One bitonic step at distance S < kTeamE: between registers of the same lane.
template <int S>
__device__ __forceinline__ void team_reg_step(uint64_t (&v)[kTeamE], int g0, int size) {
#pragma unroll
  for (int e = 0; e < kTeamE; ++e) {
    if ((e & S) != 0) continue;
    const bool desc = ((g0 + e) & size) == 0;
    const uint64_t a = v[e], b = v[e | S];
    const bool sw = (a < b) == desc;  // equal keys (zero padding) may swap
    v[e] = sw ? b : a;
    v[e | S] = sw ? a : b;
  }
}

// The network over N keys.  The loops over block sizes and distances stay
// rolled (only the per-register work is unrolled) so that the code fits the
// instruction cache.  xbuf: the team's 2 x 512-key exchange area (N = 1024).
template <int N>
__device__ __forceinline__ void team_sort(uint64_t (&v)[kTeamE], int g0, int lane,
                                          uint64_t* xbuf, uint32_t bar_id) {
#pragma unroll 1
  for (int size = 2; size <= N; size <<= 1) {
    int stride = size >> 1;
    if (stride >= kTeamKeys) {  // the two warps' halves: size == N == 1024
      const int w = g0 / kTeamKeys;
#pragma unroll
      for (int e = 0; e < kTeamE; ++e) xbuf[w * kTeamKeys + e * 32 + lane] = v[e];
      bar_sync(bar_id, 64);
      const bool keep_max = w == 0;  // descending block: the lower half keeps the larger
#pragma unroll
      for (int e = 0; e < kTeamE; ++e)
        v[e] = keep_of(v[e], xbuf[(1 - w) * kTeamKeys + e * 32 + lane], keep_max);
      stride >>= 1;
    }
#pragma unroll 1
    for (; stride >= kTeamE; stride >>= 1) {
      // distance >= kTeamE: between lanes; all registers of a lane keep the
      // same side of their pairs
      const bool keep_max = ((g0 & stride) == 0) == ((g0 & size) == 0);
      const int lx = stride / kTeamE;
#pragma unroll
      for (int e = 0; e < kTeamE; ++e)
        v[e] = keep_of(v[e], __shfl_xor_sync(0xffffffffu, v[e], lx), keep_max);
    }
#pragma unroll 1
    for (; stride > 0; stride >>= 1) {
      switch (stride) {
        case 1: team_reg_step<1>(v, g0, size); break;
        case 2: team_reg_step<2>(v, g0, size); break;
        case 4: team_reg_step<4>(v, g0, size); break;
        default: team_reg_step<8>(v, g0, size); break;
      }
    }
  }
}

template <int TOPK>
struct TeamSmem {
  static constexpr int W = TOPK / kTeamKeys;             // warps per row
  static constexpr int kTeams = kTeamThreads / 32 / W;   // rows per CTA
  uint64_t xbuf[W == 2 ? kTeams * TOPK : 1];
  uint32_t team_ok[kTeams];
};

// The rows of CTA `blk` of the team grid (kTeams rows per CTA).  SCORES: a
// context shard's emission (p.out_score set), see FinishParams.
template <int TOPK, bool SCORES>
__device__ __forceinline__ void team_rows(const FinishParams& p, int64_t blk, TeamSmem<TOPK>& ts) {
  constexpr int W = TeamSmem<TOPK>::W;
  constexpr int kTeams = TeamSmem<TOPK>::kTeams;
  uint64_t* xbuf = ts.xbuf;
  uint32_t* team_ok = ts.team_ok;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int team = warp / W, tw = warp % W;
  const uint32_t bar_id = 1u + (uint32_t)team;
  const int64_t r = blk * kTeams + team;
  if (r >= p.rows) return;  // the same for both warps of a team
  // one status read per team, so that its warps take the same path
  if (tw == 0 && lane == 0) team_ok[team] = read_status(p.hdr) == kOk;
  if constexpr (W == 2) bar_sync(bar_id, 64);
  else __syncwarp();
  if (!((volatile uint32_t*)team_ok)[team]) return;
  const int32_t s0 = p.row_start[r], s1 = p.row_end[r];
  const int64_t len = (int64_t)s1 - s0;
  const int32_t* row_pt =
      p.page_table ? p.page_table + (int64_t)p.row_req[r] * p.max_pages : nullptr;
  int32_t* out_raw = p.out_raw ? p.out_raw + r * TOPK : nullptr;
  int32_t* out_phys = p.out_phys ? p.out_phys + r * TOPK : nullptr;
  float* out_score = SCORES ? p.out_score + r * TOPK : nullptr;
  const int t = tw * 32 + lane;  // thread within the team
  // a context shard scores every nonempty clipped window, however short
  if (len <= (SCORES ? 0 : TOPK)) {
    bool bad_page = false;
    for (int i = t; i < TOPK; i += 32 * W) {
      const int32_t raw = i < len ? s0 + i : -1;
      if (out_raw) out_raw[i] = raw;
      if (out_phys) out_phys[i] = map_phys(row_pt, raw, p.num_pages, bad_page);
      if (SCORES) out_score[i] = __uint_as_float(0x7FC00000u);
    }
    if (bad_page) raise_status(p.hdr, kErrInvalidPage, 441);
    return;
  }
  const BlockInfo bi = p.blocks[p.row_block[r]];
  if (bi.n_units != 1) return;
  const int64_t slot = bi.slot0 + (r - bi.row0);
  if (!IDX_IN_RANGE(slot >= 0 && slot < p.hdr->n_row_slots, p.hdr, 430)) return;
  const uint32_t n = min(p.cand_cnt[slot], (uint32_t)TOPK);
  const uint64_t* keys = p.cand_keys + slot * TOPK;
  uint64_t v[kTeamE];
#pragma unroll
  for (int e = 0; e < kTeamE; ++e) {
    // any placement of the inputs suits the network: read coalesced; an
    // underfilled row (never expected) is padded with the empty key 0, which
    // maps to -1
    const uint32_t i = (uint32_t)(tw * kTeamKeys + e * 32 + lane);
    v[e] = i < n ? keys[i] : 0ull;
  }
  const int g0 = tw * kTeamKeys + lane * kTeamE;
  team_sort<TOPK>(v, g0, lane, xbuf + (W == 2 ? team * TOPK : 0), bar_id);
  // the lane now holds ranks g0 .. g0 + 15; rows start at multiples of 2 KB
  // of a 16-byte aligned base
  bool bad_page = false;
#pragma unroll
  for (int e = 0; e < kTeamE; e += 4) {
    int32_t raw[4], phys[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      raw[k] = v[e + k] != 0ull ? key_index(v[e + k]) : -1;
      phys[k] = map_phys(row_pt, raw[k], p.num_pages, bad_page);
    }
    if (out_raw)
      *reinterpret_cast<int4*>(out_raw + g0 + e) = make_int4(raw[0], raw[1], raw[2], raw[3]);
    if (out_phys)
      *reinterpret_cast<int4*>(out_phys + g0 + e) = make_int4(phys[0], phys[1], phys[2], phys[3]);
    if (SCORES)
      *reinterpret_cast<float4*>(out_score + g0 + e) =
          make_float4(key_score(v[e]), key_score(v[e + 1]), key_score(v[e + 2]), key_score(v[e + 3]));
  }
  if (bad_page) raise_status(p.hdr, kErrInvalidPage, 442);
}

// Shared memory of a finishing CTA.
struct FinSmem {
  uint64_t buf[kFinCap];
  uint32_t hist[256];
  uint32_t uoff[kFinThreads];           // keys of the row's units before each unit
  uint32_t ucnt[kFinThreads];           // keys of each unit (at most TOPK)
  uint32_t wsum[kFinThreads / 32];
  uint32_t bc[4];
  uint32_t cnt;
  uint32_t ok;
  uint64_t tau;
};

// Where finish_row takes a row's candidates from.
enum FinSrc : int { kSrcUnits = 0, kSrcDense = 1, kSrcShards = 2 };

// One row, by the whole CTA (every early return is uniform over the CTA).
// SCORES: a context shard's emission (p.out_score set), see FinishParams.
template <int TOPK, int SRC, bool SCORES>
__device__ __forceinline__ void finish_row(const FinishParams& p, int64_t r, FinSmem& sm) {
  constexpr bool DENSE = SRC != kSrcUnits;  // the closed form of short rows is ours
  uint64_t* buf = sm.buf;
  uint32_t* hist = sm.hist;
  uint32_t* bc = sm.bc;
  uint32_t& cnt = sm.cnt;
  uint64_t& tau = sm.tau;
  const int tid = threadIdx.x;
  const int32_t s0 = p.row_start[r], s1 = p.row_end[r];
  const int64_t len = (int64_t)s1 - s0;
  const int32_t* row_pt =
      p.page_table ? p.page_table + (int64_t)p.row_req[r] * p.max_pages : nullptr;
  int32_t* out_raw = p.out_raw ? p.out_raw + (int64_t)r * TOPK : nullptr;
  int32_t* out_phys = p.out_phys ? p.out_phys + (int64_t)r * TOPK : nullptr;
  float* out_score = SCORES ? p.out_score + (int64_t)r * TOPK : nullptr;

  if (len <= (SCORES ? 0 : TOPK)) {
    if constexpr (DENSE) {
      bool bad_page = false;
      for (int i = tid; i < TOPK; i += kFinThreads) {
        const int32_t raw = i < len ? s0 + i : -1;
        if (out_raw) out_raw[i] = raw;
        if (out_phys) out_phys[i] = map_phys(row_pt, raw, p.num_pages, bad_page);
      }
      if (bad_page) raise_status(p.hdr, kErrInvalidPage, 443);
    }
    return;  // the merge's short rows are team_rows'
  }
  if constexpr (!DENSE) {
    if (p.blocks[p.row_block[r]].n_units == 1) return;  // team_rows'
  }

  if (tid == 0) {
    cnt = 0;
    tau = 0;
  }
  __syncthreads();
  uint64_t t = 0;
  if constexpr (SRC == kSrcShards) {
    // the union of the row's context-shard lists; every listed position must
    // lie in the row's window
    bool bad = false;
    for (int k = 0; k < p.n_shards; ++k) {
      const int64_t off = ((int64_t)k * p.rows + r) * TOPK;
      for (int base = 0; base < TOPK; base += kFinBatch) {
        bool over = false;
#pragma unroll
        for (int e = 0; e < kFinPer; ++e) {
          const int i = base + e * kFinThreads + tid;
          const int32_t raw = i < TOPK ? p.shard_raw[off + i] : -1;
          const bool in = raw >= 0;
          bad |= raw < -1 || (in && (raw < s0 || raw >= s1));
          const uint64_t key = in ? order_key(p.shard_score[off + i], raw) : 0ull;
          over |= sel_append(buf, &cnt, kFinCap, kFinCap - kFinBatch, in && key >= t, key);
        }
        if (bar_red_or(kFinBar, kFinThreads, over)) {
          sel_compact<kFinThreads, kFinCap>(buf, &cnt, &tau, hist, bc, TOPK, tid, kFinBar, p.hdr,
                                            nullptr, 0, 0, kErrInvalidMetadata);
          t = *(volatile uint64_t*)&tau;
        }
      }
    }
    if (bad) raise_status(p.hdr, kErrInvalidMetadata, 420);
  } else if constexpr (DENSE) {
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
    const int j = (int)(r - bi.row0);
    // The row's units in groups of kGroup: each thread loads all its keys of a
    // group before it stores any (one memory round trip per group instead of
    // one per key), unit u's keys to consecutive slots after those of the
    // group's earlier units.  Before a group that does not fit the buffer's
    // free space the buffer is reduced to the TOPK largest keys.
    bool gathered = false;
    if (bi.n_units <= kFinThreads) {
      uint32_t c = 0;
      if (tid < bi.n_units &&
          IDX_IN_RANGE(bi.slot0 + (int64_t)tid * bi.nrows + j < p.hdr->n_row_slots, p.hdr, 431))
        c = min(p.cand_cnt[bi.slot0 + (int64_t)tid * bi.nrows + j], (uint32_t)TOPK);
      const int lane = tid & 31, w = tid >> 5;
      uint32_t x = c;  // inclusive scan of the counts: lanes, then warps
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) sm.wsum[w] = x;
      __syncthreads();
      uint32_t before = 0, total = 0;
#pragma unroll
      for (int k = 0; k < kFinThreads / 32; ++k) {
        const uint32_t ws = sm.wsum[k];
        before += k < w ? ws : 0u;
        total += ws;
      }
      sm.uoff[tid] = before + x - c;
      sm.ucnt[tid] = c;
      __syncthreads();
      constexpr int kE = TOPK / kFinThreads;        // keys of one unit per thread
      constexpr int kGroup = (kFinCap - TOPK) / TOPK;  // fits after a reduction to TOPK
      static_assert(kGroup >= 1, "buffer capacity");
      for (int u0 = 0; u0 < bi.n_units; u0 += kGroup) {
        const int u1 = min(u0 + kGroup, bi.n_units);
        const uint32_t gsize = (u1 < bi.n_units ? sm.uoff[u1] : total) - sm.uoff[u0];
        uint32_t base = *(volatile uint32_t*)&cnt;
        if (base + gsize > (uint32_t)kFinCap) {  // the same decision in every thread
          sel_compact<kFinThreads, kFinCap>(buf, &cnt, &tau, hist, bc, TOPK, tid, kFinBar, p.hdr);
          base = *(volatile uint32_t*)&cnt;
        }
        uint64_t v[kGroup * kE];
#pragma unroll
        for (int q = 0; q < kGroup * kE; ++q) {
          const int u = u0 + q / kE;
          const uint32_t i = (uint32_t)(tid + (q % kE) * kFinThreads);
          const bool in = u < u1 && i < sm.ucnt[u];
          v[q] = in ? p.cand_keys[(bi.slot0 + (int64_t)u * bi.nrows + j) * TOPK + i] : 0ull;
        }
#pragma unroll
        for (int q = 0; q < kGroup * kE; ++q) {
          const int u = u0 + q / kE;
          const uint32_t i = (uint32_t)(tid + (q % kE) * kFinThreads);
          if (u < u1 && i < sm.ucnt[u]) {
            const uint32_t pos = base + (sm.uoff[u] - sm.uoff[u0]) + i;
            if (IDX_IN_RANGE(pos < (uint32_t)kFinCap, p.hdr, 433)) buf[pos] = v[q];
          }
        }
        __syncthreads();
        if (tid == 0) cnt = base + gsize;
        __syncthreads();
      }
      gathered = true;
    }
    // a row of more than kFinThreads units (a window of over two million
    // positions even at the smallest unit size): unit by unit through the
    // selector
    for (int k = 0; !gathered && k < bi.n_units; ++k) {
      const int64_t slot = bi.slot0 + (int64_t)k * bi.nrows + j;
      if (!IDX_IN_RANGE(slot < p.hdr->n_row_slots, p.hdr, 432)) break;
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
  sel_compact<kFinThreads, kFinCap>(buf, &cnt, &tau, hist, bc, TOPK, tid, kFinBar, p.hdr, nullptr,
                                    0, 0, SRC == kSrcShards ? kErrInvalidMetadata : kErrInternal);
  const uint32_t n = min(*(volatile uint32_t*)&cnt, (uint32_t)TOPK);
  if (n < (uint32_t)TOPK) {
    // a window of len positions yields min(len, topk) candidates (len > topk
    // except for the clipped windows of a context shard)
    if (tid == 0 && (!SCORES || n < (uint64_t)len))
      raise_status(p.hdr, SRC == kSrcShards ? kErrInvalidMetadata : kErrInternal,
                   SRC == kSrcShards ? 421 : 400);
    for (int i = n + tid; i < TOPK; i += kFinThreads) buf[i] = 0ull;
  }
  __syncthreads();
  sort_emit<TOPK, SCORES, SRC == kSrcShards>(buf, tid, row_pt, p.num_pages, p.hdr, out_raw,
                                            out_phys, out_score);
}

// Rows r = blk, blk + nblk, ...; the status is read once per row by one
// thread so that the CTA's threads agree on it.
template <int TOPK, int SRC, bool SCORES>
__device__ __forceinline__ void merge_rows(const FinishParams& p, int64_t blk, int64_t nblk,
                                           FinSmem& sm) {
  for (int64_t r = blk; r < p.rows; r += nblk) {
    if (threadIdx.x == 0) sm.ok = read_status(p.hdr) == kOk;
    __syncthreads();
    if (!sm.ok) return;
    finish_row<TOPK, SRC, SCORES>(p, r, sm);
    __syncthreads();  // the row's shared state is free again
  }
}

// Exact TopK of the rows of a materialised score matrix (the dense path), or
// of the union of a row's context-shard lists.
template <int TOPK, int SRC>
__global__ void __launch_bounds__(kFinThreads) finish_kernel(FinishParams p) {
  __shared__ __align__(16) FinSmem sm;
  merge_rows<TOPK, SRC, false>(p, blockIdx.x, gridDim.x, sm);
}

// The fused path's finishing step in one launch: CTAs [0, team_blocks) sort
// the single-unit and short rows (team_rows), the others merge the rows of
// multi-unit blocks; the two sets of rows are disjoint, so both run at once.
template <int TOPK>
union FinishShared {
  TeamSmem<TOPK> team;
  FinSmem merge;
};

// The CTA that finishes last (every CTA's writes are fenced before it counts
// itself on the header) publishes the call's status and, on an error, fills
// the outputs with -1.
__device__ __forceinline__ void publish_if_last(const FinishParams& p) {
  __shared__ uint32_t s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&p.hdr->fin_done, 1u) == gridDim.x - 1u;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const uint32_t st = read_status(p.hdr);
  if (threadIdx.x == 0) *p.status_out = st;
  if (st == kOk) return;
  const int64_t n = (int64_t)p.rows * p.topk;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    if (p.out_phys) p.out_phys[i] = -1;
    if (p.out_raw) p.out_raw[i] = -1;
  }
}

template <int TOPK, bool SCORES>
__global__ void __launch_bounds__(kFinThreads) finish_fused_kernel(FinishParams p, int team_blocks) {
  static_assert(kTeamThreads == kFinThreads, "one block shape for both paths");
  __shared__ __align__(16) FinishShared<TOPK> sh;
  if ((int)blockIdx.x < team_blocks) {
    team_rows<TOPK, SCORES>(p, blockIdx.x, sh.team);
  } else {
    merge_rows<TOPK, kSrcUnits, SCORES>(p, (int64_t)blockIdx.x - team_blocks,
                                        (int64_t)gridDim.x - team_blocks, sh.merge);
  }
  if (p.status_out) publish_if_last(p);
}

// Row windows: 0 <= start <= end <= width, and (row_req non-null) a request
// in [0, num_req).
__global__ void validate_windows_kernel(const int32_t* row_start, const int32_t* row_end,
                                        int32_t rows, int64_t width, const int32_t* row_req,
                                        int32_t num_req, PlanHeader* hdr) {
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows;
       r += (int64_t)gridDim.x * blockDim.x) {
    const int32_t s = row_start[r], e = row_end[r];
    bool bad = s < 0 || e < s || (int64_t)e > width;
    if (row_req) bad |= row_req[r] < 0 || row_req[r] >= num_req;
    if (bad) raise_status(hdr, kErrInvalidMetadata, 410);
  }
}

template <int TOPK, int SRC>
cudaError_t launch_t(const FinishParams& p, cudaStream_t stream) {
  const int merge_grid = p.rows < kFinGridCap ? p.rows : kFinGridCap;
  if (SRC != kSrcUnits) {
    finish_kernel<TOPK, SRC><<<merge_grid, kFinThreads, 0, stream>>>(p);
  } else {
    constexpr int kTeams = TeamSmem<TOPK>::kTeams;
    const int team_grid = (p.rows + kTeams - 1) / kTeams;
    if (p.out_score)
      finish_fused_kernel<TOPK, true><<<team_grid + merge_grid, kFinThreads, 0, stream>>>(p, team_grid);
    else
      finish_fused_kernel<TOPK, false><<<team_grid + merge_grid, kFinThreads, 0, stream>>>(p, team_grid);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_finish(const FinishParams& p, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  const int src = p.shard_raw ? kSrcShards : (p.scores ? kSrcDense : kSrcUnits);
  if (p.topk == 512) {
    if (src == kSrcShards) return launch_t<512, kSrcShards>(p, stream);
    return src == kSrcDense ? launch_t<512, kSrcDense>(p, stream) : launch_t<512, kSrcUnits>(p, stream);
  }
  if (p.topk == 1024) {
    if (src == kSrcShards) return launch_t<1024, kSrcShards>(p, stream);
    return src == kSrcDense ? launch_t<1024, kSrcDense>(p, stream)
                            : launch_t<1024, kSrcUnits>(p, stream);
  }
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
  __shared__ uint32_t ok;  // one status read, so that the CTA's threads agree
  if (tid == 0) ok = read_status(p.hdr) == kOk;
  __syncthreads();
  if (!ok) return;
  const int32_t s0 = p.row_start[r], s1 = p.row_end[r];
  const int64_t len = (int64_t)s1 - s0;
  const int32_t* row_pt = p.page_table + (int64_t)p.row_req[r] * p.max_pages;
  if (len <= TOPK) {
    if (!p.last) return;
    bool bad_page = false;
    for (int i = tid; i < TOPK; i += kFinThreads) {
      const int32_t raw = i < len ? s0 + i : -1;
      if (p.out_raw) p.out_raw[(int64_t)r * TOPK + i] = raw;
      p.out_phys[(int64_t)r * TOPK + i] = map_phys(row_pt, raw, p.num_pages, bad_page);
    }
    if (bad_page) raise_status(p.hdr, kErrInvalidPage, 444);
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
  sort_emit<TOPK>(buf, tid, row_pt, p.num_pages, p.hdr,
                  p.out_raw ? p.out_raw + (int64_t)r * TOPK : nullptr, p.out_phys + (int64_t)r * TOPK);
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

cudaError_t launch_validate_windows(const int32_t* row_start, const int32_t* row_end, int32_t rows,
                                    int64_t width, PlanHeader* hdr, cudaStream_t stream,
                                    const int32_t* row_req, int32_t num_req) {
  if (rows <= 0) return cudaSuccess;
  int blocks = (rows + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  validate_windows_kernel<<<blocks, 256, 0, stream>>>(row_start, row_end, rows, width, row_req,
                                                      num_req, hdr);
  return cudaGetLastError();
}

}  // namespace idxk
