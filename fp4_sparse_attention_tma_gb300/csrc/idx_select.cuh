// Bounded streaming exact TopK in shared memory, used by the fused scorer's
// epilogue, the candidate merge and the dense-matrix TopK.
//
// A row keeps a buffer of 64-bit order keys (see order_key) that are >= its
// threshold tau.  Threads append passing keys with warp-aggregated atomics;
// when the count gets close to the capacity, the group runs a radix select
// (8-bit windows, most significant first, the first one starting at the
// highest bit in which the keys differ, with early exit) that finds a
// threshold T with exactly topk keys >= T, compacts the buffer to those keys
// and raises tau to T.  Because the composite key includes the logical index,
// keys of one row are distinct and the selection is exact.  This follows the
// design stated in "[FlyDSL][DSv4] Prototype FP4 MQA streaming TopK"
// (ROCm/aiter#5282, Changes): scores stream through a bounded on-chip pool; a
// four-byte score radix plus a four-byte logical-index radix implements the
// total order.
#pragma once

#include "idx_device.cuh"

namespace idxk {

// Appends `key` when `pass`; returns true (on lane 0 only) when the count after
// this warp's append exceeds `limit`.  buf has room for cap entries.
__device__ __forceinline__ bool sel_append(uint64_t* buf, uint32_t* cnt, uint32_t cap,
                                           uint32_t limit, bool pass, uint64_t key) {
  const int lane = threadIdx.x & 31;
  const uint32_t m = __ballot_sync(0xffffffffu, pass);
  bool over = false;
  if (m) {
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(cnt, (uint32_t)__popc(m));
    base = __shfl_sync(0xffffffffu, base, 0);
    const uint32_t pos = base + (uint32_t)__popc(m & ((1u << lane) - 1u));
    if (pass && pos < cap) buf[pos] = key;
    over = (lane == 0) && (base + (uint32_t)__popc(m) > limit);
  }
  return over;
}

// Key storage seen by sel_compact: buf[0, *cnt_s) holds keys kept so far;
// with NREG > 0, region r additionally holds reg_cnt[r] keys at
// buf[reg_base + r * reg_stride ...] (reg_base >= the number of keys that are
// kept, so regions are never overwritten by the result).
template <int NREG>
struct SelSegments {
  uint32_t kept;
  uint32_t cnt[NREG > 0 ? NREG : 1];
  uint32_t reg_base, reg_stride;
  // physical index of the i-th key in the order kept, region 0, region 1, ...
  __device__ __forceinline__ uint32_t phys(uint32_t i) const {
    if (NREG == 0 || i < kept) return i;
    uint32_t j = i - kept;
#pragma unroll
    for (int r = 0; r < NREG; ++r) {
      if (j < cnt[r]) return reg_base + (uint32_t)r * reg_stride + j;
      j -= cnt[r];
    }
    return 0;  // not reached for i < total
  }
};

// Collective over NT threads (tid in [0, NT), named barrier bar_id, NT a
// multiple of 32 and at most 256).  Reduces the row's keys -- buf[0, *cnt_s)
// plus, with NREG > 0, the NREG append regions whose counts are in reg_cnt
// (shared memory) -- to the K largest, stored in buf[0, min(n, K)); *cnt_s and,
// when keys were dropped, *tau_s (the K-th largest key's radix prefix, a lower
// bound of every kept key) are updated.  All keys are distinct; keys that are
// not (a list that names a position twice) leave the kept count off, which is
// reported as err_code.  CAP is the buffer's capacity.
template <int NT, int CAP, int NREG = 0>
__device__ __noinline__ void sel_compact(uint64_t* buf, uint32_t* cnt_s, uint64_t* tau_s,
                                         uint32_t* hist, uint32_t* bc, uint32_t K, int tid,
                                         uint32_t bar_id, PlanHeader* hdr,
                                         const uint32_t* reg_cnt = nullptr, uint32_t reg_base = 0,
                                         uint32_t reg_stride = 0, uint32_t err_code = kErrInternal) {
  SelSegments<NREG> sg;
  sg.kept = *(volatile uint32_t*)cnt_s;
  uint32_t n = sg.kept;
#pragma unroll
  for (int r = 0; r < NREG; ++r) {
    sg.cnt[r] = ((volatile const uint32_t*)reg_cnt)[r];
    n += sg.cnt[r];
  }
  sg.reg_base = reg_base;
  sg.reg_stride = reg_stride;
  if (NREG == 0 && n <= K) return;
  const int lane = tid & 31, wid = tid >> 5;
  uint64_t prefix = 0ull;  // keep every key >= prefix
  if (n > K) {
    // Bytes that every key shares need no histogram pass: find the highest bit
    // in which the keys differ (they are distinct, so one exists).
    uint64_t kand = ~0ull, kor = 0ull;
    for (uint32_t i = tid; i < n; i += NT) {
      const uint64_t k = buf[sg.phys(i)];
      kand &= k;
      kor |= k;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      kand &= __shfl_xor_sync(0xffffffffu, kand, o);
      kor |= __shfl_xor_sync(0xffffffffu, kor, o);
    }
    volatile uint64_t* red = reinterpret_cast<volatile uint64_t*>(hist);  // 2 x NT/32 words
    if (lane == 0) {
      red[2 * wid] = kand;
      red[2 * wid + 1] = kor;
    }
    bar_sync(bar_id, NT);
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
      kand &= red[2 * w];
      kor |= red[2 * w + 1];
    }
    bar_sync(bar_id, NT);  // the words are read before the histogram is cleared
    const int top = 63 - __clzll((long long)(kand ^ kor));
    // the first 8-bit window starts at the highest differing bit, so that it
    // splits the keys 256 ways instead of the 2 or 3 ways a byte-aligned window
    // gives keys of nearly equal scores (fewer passes, and the histogram's
    // shared-memory atomics spread over many bins)
    int shift = top >= 7 ? top - 7 : 0;
    uint64_t pmask = shift >= 56 ? 0ull : (~0ull << (shift + 8));
    prefix = kand & pmask;
    uint32_t need = K;
    for (; shift > -8; shift -= 8) {
      if (shift < 0) shift = 0;  // the last window overlaps bits already resolved
      for (int b2 = tid; b2 < 256; b2 += NT) hist[b2] = 0;
      bar_sync(bar_id, NT);
      for (uint32_t i = tid; i < n; i += NT) {
        const uint64_t k = buf[sg.phys(i)];
        if ((k & pmask) == prefix) atomicAdd(&hist[(uint32_t)(k >> shift) & 255u], 1u);
      }
      bar_sync(bar_id, NT);
      if (tid < 32) {
        uint32_t c[8], sum = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          c[e] = hist[255 - 8 * tid - e];
          sum += c[e];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += v;
        }
        uint32_t above = incl - sum;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (above < need && above + c[e] >= need) {
            bc[0] = 255u - 8u * tid - e;
            bc[1] = above;
            bc[2] = c[e];
          }
          above += c[e];
        }
      }
      bar_sync(bar_id, NT);
      const uint32_t d = bc[0], ab = bc[1], cd = bc[2];
      need -= ab;
      prefix |= (uint64_t)d << shift;
      pmask |= (uint64_t)0xffu << shift;
      if (cd == need || shift == 0) break;
    }
  }
  // Keep the keys >= prefix, written in order of the scan to buf[0, ...):
  // chunk by chunk, every chunk read before any slot of it can be overwritten
  // (a kept key never moves to a higher index than it is read from, and the
  // regions lie above every written slot).
  constexpr int CH = 8;
  if (tid == 0) bc[3] = 0;
  bar_sync(bar_id, NT);
  for (uint32_t base = 0; base < n; base += NT * CH) {
    uint64_t v[CH];
#pragma unroll
    for (int e = 0; e < CH; ++e) {
      const uint32_t i = base + (uint32_t)(tid + e * NT);
      v[e] = i < n ? buf[sg.phys(i)] : 0ull;
    }
    bar_sync(bar_id, NT);
#pragma unroll
    for (int e = 0; e < CH; ++e) {
      const bool keep = v[e] != 0ull && v[e] >= prefix;
      const uint32_t m = __ballot_sync(0xffffffffu, keep);
      if (m) {
        uint32_t pos0 = 0;
        if (lane == 0) pos0 = atomicAdd(&bc[3], (uint32_t)__popc(m));
        pos0 = __shfl_sync(0xffffffffu, pos0, 0);
        const uint32_t pos = pos0 + (uint32_t)__popc(m & ((1u << lane) - 1u));
        if (keep && pos < (uint32_t)CAP) buf[pos] = v[e];
      }
    }
    bar_sync(bar_id, NT);
  }
  if (tid == 0) {
    const uint32_t expect = n > K ? K : n;
    if (bc[3] != expect) raise_status(hdr, err_code, 200);
    *cnt_s = expect;
    if (n > K) *tau_s = prefix;
  }
  bar_sync(bar_id, NT);
}

}  // namespace idxk
