// Fused FP4 paged-MQA scorer for sm_103a (one persistent CTA per SM).
//
// Per work unit (a block of up to 3 rows of one request x a run of 128-slot K
// tiles; see idx_internal.h) the CTA
//   * stages each K tile (2 pages of 64 slots x 64 B of E2M1 codes, plus their
//     UE8M0 scales) with TMA, the page looked up in the page table, and the
//     query block (3 rows x 64 heads x 64 B + scales + weights) once per unit;
//   * runs the contraction logit[s, (r,h)] = sum_d k[s,d] q[r,h,d] on the
//     tcgen05 block-scaled FP4 MMA (kind::mxf4, scale vector 32, M = 128 slots,
//     N = 3 rows x 64 heads = 192, K = 64 per instruction, two per tile) into a
//     double-buffered TMEM accumulator;
//   * drains TMEM in three epilogue warpgroups, one per row, each holding its
//     row's 64 weights in registers: score[r, s] = sum_h w[r,h] * max(logit, 0)
//     in fp32, then either streams the (score, slot) keys through the bounded
//     shared-memory TopK (select mode) or writes the fp32 scores (dense mode).
// This realises the fused scorer + CTA-local exact TopK of "[FlyDSL] Add FP4
// LiteTopK prefill operator" (ROCm/aiter#5309, Implementation) and
// "[FlyDSL][DSv4] Prototype FP4 MQA streaming TopK" (ROCm/aiter#5282, Changes
// and Scope), re-designed around TMA, tcgen05 and TMEM.
//
// Warp roles (512 threads): warps 0 and 3 TMA producers (alternate K tiles;
// each also rearranges its tiles' scale factors into the TMEM copy layout),
// warps 1 and 2 MMA issuers (one accumulator buffer each; warp 1 also owns the
// TMEM allocation), warps 4..15 epilogue (warpgroup g = row g of the block;
// warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31, i.e. slots of the tile).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "idx_device.cuh"
#include "idx_launch.h"
#include "idx_select.cuh"

namespace idxk {

namespace {

constexpr int kThreads = 512;
constexpr int kStages = 6;       // K-tile ring (TMA latency x tile rate)
constexpr int kEpiWarp0 = 4;
constexpr int kProducer2 = 3;  // second TMA producer warp
static_assert(kStages % 2 == 0, "producers own the stages of one parity each");
static_assert(kAccStages == 2, "one MMA issuer warp per accumulator buffer");
constexpr int kEpiThreads = 128;  // one warpgroup

constexpr uint32_t kPageBytes = kPage * kDimBytes;                 // 4096
constexpr uint32_t kABytes = kTile * kDimBytes;                    // 8192
constexpr uint32_t kRowBBytes = kHeads * kDimBytes;                // 4096 (one query row)
constexpr uint32_t kBBytes = kRowsPerBlock * kRowBBytes;           // 12288
constexpr uint32_t kRowSfBytes = kHeads * kNumSF;                  // 256
constexpr uint32_t kSfbAtoms = (kRowsPerBlock * kHeads + 127) / 128;  // 2 atoms of 128 rows
constexpr uint32_t kSfbAtomBytes = kSfbAtoms * 512;                // 1024
constexpr uint32_t kBlockWBytes = kRowsPerBlock * kHeads * 4;      // 768

constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kABytes;
constexpr uint32_t kOffSfaAtom = kOffB + 2 * kBBytes;               // [kStages] K-tile scale atoms
constexpr uint32_t kOffSfbRaw = kOffSfaAtom + kStages * 512;        // [2 q buffers], padded to atoms
constexpr uint32_t kOffSfbAtom = kOffSfbRaw + 2 * kSfbAtomBytes;    // [2 issuers][2 q buffers]
constexpr uint32_t kOffW = kOffSfbAtom + 2 * 2 * kSfbAtomBytes;
constexpr uint32_t kOffBar = kOffW + 2 * kBlockWBytes;
constexpr uint32_t kOffMisc = kOffBar + 512;
constexpr uint32_t kOffHist = kOffMisc + 256;
constexpr uint32_t kOffCand = kOffHist + kChunks * 256 * 4;
static_assert(kOffB % 1024 == 0 && kOffA % 1024 == 0 && kRowBBytes % 1024 == 0,
              "operand buffers must be 1 KB aligned");
static_assert(kOffSfaAtom % 128 == 0 && kOffSfbAtom % 128 == 0 && kOffCand % 16 == 0,
              "alignment");

// misc region
constexpr uint32_t kMiscTmem = 0, kMiscAbort = 4, kMiscTau = 32,
                   kMiscBc = 64,    // [3 rows][8 words] selection scratch
                   kMiscWc = 160,   // [3 rows][4 warps] region counts
                   kMiscUnit = 224; // [2 q buffers] claimed schedule position (dynamic mode)

// barriers (8 bytes each)
constexpr int kBarFull = 0;                                  // [kStages]
constexpr int kBarEmpty = kBarFull + kStages;                // [kStages]
constexpr int kBarAccFull = kBarEmpty + kStages;             // [kAccStages]
constexpr int kBarAccEmpty = kBarAccFull + kAccStages;       // [kAccStages]
constexpr int kBarQFull = kBarAccEmpty + kAccStages;         // [2]
constexpr int kBarQEmpty = kBarQFull + 2;                    // [2]
constexpr int kBarEpiDone = kBarQEmpty + 2;                  // [2]
constexpr int kBarMmaFinal = kBarEpiDone + 2;                // [kAccStages]
static_assert((kBarMmaFinal + kAccStages) * 8 <= 512, "barrier region");


// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = kRowsPerBlock * kHeads;  // 192: one accumulator buffer
constexpr uint32_t kColAcc = 0;                      // + kAccCols * stage + 64 * row
constexpr uint32_t kColSfa = kAccStages * kAccCols;  // 384: + 4 * K stage
constexpr uint32_t kColSfb = kColSfa + 4 * kStages;  // + 4 * kSfbAtoms * (2 * issuer + q buffer)
static_assert(kColSfb + 2 * 2 * 4 * kSfbAtoms <= kTmemCols, "TMEM budget");

constexpr uint32_t kIdescK0 = idesc_mxf4(128, kAccCols, 0);
constexpr uint32_t kIdescK1 = idesc_mxf4(128, kAccCols, 2);

// Per-row candidate buffer of order keys, split into one region per epilogue
// warp of the row (warp_region keys each).  A warp appends its passing keys to
// its own region, counting in a register (no shared-memory atomics).  Every
// kCheckTiles tiles the warps of the block's scored rows vote (named barrier
// kBarVote); when a region of any row has fewer than kCheckTiles * 32 entries
// free, each row's group finds the threshold that keeps exactly topk keys over
// its four regions and each warp compacts its own region in place.  A region never has to hold more than topk survivors plus
// one check window of appends.
constexpr int kCheckTiles = 12;
// At topk 512 a unit of at most kShortUnitTiles tiles compacts as soon as a
// region holds more than kShortTrig keys (at the first vote when the row's
// window covers the first 12 tiles: 4 x 384 keys for 512), so that its
// threshold rises early and its later tiles append few keys.  Longer units and
// topk 1024 keep the late trigger (an early one measured slower there).
constexpr int kShortUnitTiles = 96;
constexpr uint32_t kShortTrig = 383;
constexpr uint32_t kBarVote = 4;  // named barrier of the compaction vote (1..3: row groups)
// The candidate buffers take all shared memory the pipeline leaves free.
constexpr uint32_t kMaxSmem = 227u * 1024u;
constexpr uint32_t kCandCap = (kMaxSmem - 1024u - kOffCand) / (kRowsPerBlock * 8u) / 128u * 128u;
__host__ __device__ constexpr uint32_t cand_cap(int topk) { return topk > 0 ? kCandCap : 0u; }
__host__ __device__ constexpr uint32_t warp_region(int topk) { return cand_cap(topk) / 4u; }
static_assert(warp_region(1024) >= 1024 + kCheckTiles * 32 && warp_region(1024) % 32 == 0,
              "a region must hold topk survivors plus one check window");

__host__ __device__ constexpr size_t smem_bytes_for(int mode, int topk) {
  return 1024 + kOffCand +
         (mode == kModeSelect ? (size_t)kRowsPerBlock * cand_cap(topk) * sizeof(uint64_t) : 0);
}

static_assert(smem_bytes_for(kModeSelect, 1024) <= kMaxSmem, "shared memory budget");

// Bounded wait for the teardown: ignores the abort flag.  A phase that does
// not complete within 0.2 s means the barrier accounting went wrong (or an
// earlier wait already failed): it is recorded as kErrTimeout, not passed over.
__device__ void mbar_drain(uint32_t bar, uint32_t parity, PlanHeader* hdr, uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > 200000000ull) {  // 0.2 s
      raise_status(hdr, kErrTimeout, site);
      break;
    }
  }
}

// score = sum over heads of w * max(logit, 0) in fp32.
//
// Each head pair is folded into one of four packed (f32x2) accumulators by a
// single paired FMA; four accumulators keep the dependency chains short.  The
// rectification is split between two pipes: accumulators 0 and 1 take
// max(x, 0) (ALU pipe), accumulators 2 and 3 take |x| + x = 2 max(x, 0) (an
// add with an absolute-value operand, FMA pipe) and so hold doubled sums,
// which the final sum halves.  Both forms are exact for every logit of the
// accepted value domain (|x| < 2^93), and scaling by 2 commutes with fp32
// rounding away from the subnormal range, so the score equals the plain
// sum_h w * max(x, 0) with the same association.  The fused and the dense
// paths share this code, so their scores are bit-identical.

// One head pair: acc += (relu(x0), relu(x1)) * (w0, w1), packed (first
// product: acc = ...).  Written in PTX so that the pair is formed in place
// from the TMEM-load registers.
template <bool kInit>
__device__ __forceinline__ void pair_max(uint64_t& acc, uint32_t x0, uint32_t x1, uint64_t w) {
  if (kInit)
    asm("{\n\t.reg .f32 a, b;\n\t.reg .b64 v;\n\t"
        "max.f32 a, %1, 0f00000000;\n\t"
        "max.f32 b, %2, 0f00000000;\n\t"
        "mov.b64 v, {a, b};\n\t"
        "mul.rn.f32x2 %0, v, %3;\n\t}"
        : "=l"(acc)
        : "f"(__uint_as_float(x0)), "f"(__uint_as_float(x1)), "l"(w));
  else
    asm("{\n\t.reg .f32 a, b;\n\t.reg .b64 v;\n\t"
        "max.f32 a, %1, 0f00000000;\n\t"
        "max.f32 b, %2, 0f00000000;\n\t"
        "mov.b64 v, {a, b};\n\t"
        "fma.rn.f32x2 %0, v, %3, %0;\n\t}"
        : "+l"(acc)
        : "f"(__uint_as_float(x0)), "f"(__uint_as_float(x1)), "l"(w));
}

// One head pair into a doubled accumulator: acc += (|x0| + x0, |x1| + x1) * (w0, w1).
template <bool kInit>
__device__ __forceinline__ void pair_abs(uint64_t& acc, uint32_t x0, uint32_t x1, uint64_t w) {
  if (kInit)
    asm("{\n\t.reg .f32 a, b, c, d;\n\t.reg .b64 v;\n\t"
        "abs.f32 a, %1;\n\t"
        "abs.f32 b, %2;\n\t"
        "add.rn.f32 c, a, %1;\n\t"
        "add.rn.f32 d, b, %2;\n\t"
        "mov.b64 v, {c, d};\n\t"
        "mul.rn.f32x2 %0, v, %3;\n\t}"
        : "=l"(acc)
        : "f"(__uint_as_float(x0)), "f"(__uint_as_float(x1)), "l"(w));
  else
    asm("{\n\t.reg .f32 a, b, c, d;\n\t.reg .b64 v;\n\t"
        "abs.f32 a, %1;\n\t"
        "abs.f32 b, %2;\n\t"
        "add.rn.f32 c, a, %1;\n\t"
        "add.rn.f32 d, b, %2;\n\t"
        "mov.b64 v, {c, d};\n\t"
        "fma.rn.f32x2 %0, v, %3, %0;\n\t}"
        : "+l"(acc)
        : "f"(__uint_as_float(x0)), "f"(__uint_as_float(x1)), "l"(w));
}

// Heads 2*P0 .. 2*P0+15 from one 16-column TMEM load; head pair p goes to
// accumulator p % 4.  P0 == 0 starts the four accumulators with plain
// products instead of adding to zero: the sums differ at most in the sign of
// an all-zero total, which head_sum_final normalises.
template <int P0>
__device__ __forceinline__ void head_sum_part(const uint32_t (&x)[16], const uint64_t (&w2)[32],
                                              uint64_t (&acc)[4]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // head pair (2p, 2p+1), p = P0 + i
    const bool init = P0 == 0 && i < 4;
    if ((i & 3) < 2) {
      if (init) pair_max<true>(acc[i & 3], x[2 * i], x[2 * i + 1], w2[P0 + i]);
      else pair_max<false>(acc[i & 3], x[2 * i], x[2 * i + 1], w2[P0 + i]);
    } else {
      if (init) pair_abs<true>(acc[i & 3], x[2 * i], x[2 * i + 1], w2[P0 + i]);
      else pair_abs<false>(acc[i & 3], x[2 * i], x[2 * i + 1], w2[P0 + i]);
    }
  }
}

__device__ __forceinline__ float2 unpack2(uint64_t v) {
  return make_float2(__uint_as_float((uint32_t)v), __uint_as_float((uint32_t)(v >> 32)));
}

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint64_t half2(uint64_t a) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(0x3F0000003F000000ull));
  return d;
}

// The four packed partial sums folded lane-wise ((acc0 + acc1) + (acc2 + acc3)),
// the doubled pair halved, then the two lanes added.
__device__ __forceinline__ float head_sum_final(const uint64_t (&acc)[4]) {
  const float2 t = unpack2(add2(add2(acc[0], acc[1]), half2(add2(acc[2], acc[3]))));
  // + 0 turns an all-zero total of -0 into +0, the value a sum started at +0 has
  return (t.x + t.y) + 0.0f;
}

// The select step of one slot: the 64-bit order key (32-bit score key in the
// high word, ~position in the low word) is appended to the warp's region at
// wreg_s (shared address) when pass_in is set and the key is at least tau;
// *wcnt counts the region's keys.  One ballot, a predicated store and the
// count update, no branch.  The score key here is sb ^ (sign(sb) ? ~0 :
// 0x80000000): the order key of a finite score (every accepted call's scores
// are finite; the NaN rule of score_key needs no test here).
__device__ __forceinline__ void append_if(uint32_t& wcnt, uint32_t wreg_s, float sc, uint32_t lo,
                                          uint64_t tau, uint32_t pass_in, uint32_t lt_mask) {
  asm volatile(
      "{\n\t.reg .b64 key;\n\t.reg .pred p, q;\n\t.reg .b32 sb, sh, k, m, off, c, a;\n\t"
      "mov.b32 sb, %2;\n\t"
      "shr.s32 sh, sb, 31;\n\t"
      "or.b32 sh, sh, 0x80000000;\n\t"
      "xor.b32 k, sb, sh;\n\t"
      "mov.b64 key, {%3, k};\n\t"
      "setp.ne.u32 q, %5, 0;\n\t"
      "setp.ge.and.u64 p, key, %4, q;\n\t"
      "vote.sync.ballot.b32 m, p, 0xffffffff;\n\t"
      "and.b32 off, m, %6;\n\t"
      "popc.b32 off, off;\n\t"
      "add.u32 off, off, %0;\n\t"
      "shl.b32 off, off, 3;\n\t"
      "add.u32 a, off, %1;\n\t"
      "@p st.shared.b64 [a], key;\n\t"
      "popc.b32 c, m;\n\t"
      "add.u32 %0, %0, c;\n\t}"
      : "+r"(wcnt)
      : "r"(wreg_s), "f"(sc), "r"(lo), "l"(tau), "r"(pass_in), "r"(lt_mask)
      : "memory");
}

// Collective over a row's four epilogue warps (named barrier bar_id, 128
// threads): keeps the row's TOPK largest keys over the four regions (region w
// at buf + w * warp_region(TOPK), holding wc_s[w] keys) and compacts each region
// in place.  Returns the calling warp's new count; *tau_s receives the kept
// keys' radix prefix (a lower bound of every kept key) when keys were dropped.
// The caller has stored its count in wc_s[qd] before a barrier.
template <int TOPK>
__device__ __noinline__ uint32_t sel_compact_regions(uint64_t* buf, const uint32_t* wc_s,
                                                     uint64_t* tau_s, uint32_t* hist,
                                                     uint32_t* bc, uint32_t my_cnt, int qd,
                                                     int lane, uint32_t bar_id, PlanHeader* hdr) {
  constexpr uint32_t kQ = warp_region(TOPK);
  uint64_t* reg = buf + (uint32_t)qd * kQ;
  if (!IDX_IN_RANGE(my_cnt <= kQ, hdr, 340)) my_cnt = kQ;
  uint32_t n = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) n += ((volatile const uint32_t*)wc_s)[w];
  if (n <= (uint32_t)TOPK) return my_cnt;
  // highest bit in which the (distinct) keys differ
  uint64_t kand = ~0ull, kor = 0ull;
  for (uint32_t i = lane; i < my_cnt; i += 32) {
    const uint64_t k = reg[i];
    kand &= k;
    kor |= k;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    kand &= __shfl_xor_sync(0xffffffffu, kand, o);
    kor |= __shfl_xor_sync(0xffffffffu, kor, o);
  }
  volatile uint64_t* red = reinterpret_cast<volatile uint64_t*>(hist);
  if (lane == 0) {
    red[2 * qd] = kand;
    red[2 * qd + 1] = kor;
  }
  bar_sync(bar_id, kEpiThreads);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    kand &= red[2 * w];
    kor |= red[2 * w + 1];
  }
  bar_sync(bar_id, kEpiThreads);
  const int top = 63 - __clzll((long long)(kand ^ kor));
  // the first 8-bit window starts at the highest differing bit, so that it
  // splits the keys 256 ways instead of the 2 or 3 ways a byte-aligned window
  // gives keys of nearly equal scores (fewer passes, and the histogram's
  // shared-memory atomics spread over many bins)
  int shift = top >= 7 ? top - 7 : 0;
  uint64_t pmask = shift >= 56 ? 0ull : (~0ull << (shift + 8));
  uint64_t prefix = kand & pmask;
  uint32_t need = (uint32_t)TOPK;
  const int tg = qd * 32 + lane;
  for (; shift > -8; shift -= 8) {
    if (shift < 0) shift = 0;  // the last window overlaps bits already resolved
    for (int b2 = tg; b2 < 256; b2 += kEpiThreads) hist[b2] = 0;
    bar_sync(bar_id, kEpiThreads);
    for (uint32_t i = lane; i < my_cnt; i += 32) {
      const uint64_t k = reg[i];
      if ((k & pmask) == prefix) atomicAdd(&hist[(uint32_t)(k >> shift) & 255u], 1u);
    }
    bar_sync(bar_id, kEpiThreads);
    if (qd == 0) {
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        c[e] = hist[255 - 8 * lane - e];
        sum += c[e];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      uint32_t above = incl - sum;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (above < need && above + c[e] >= need) {
          bc[0] = 255u - 8u * lane - e;
          bc[1] = above;
          bc[2] = c[e];
        }
        above += c[e];
      }
    }
    bar_sync(bar_id, kEpiThreads);
    const uint32_t d = bc[0], ab = bc[1], cd = bc[2];
    need -= ab;
    prefix |= (uint64_t)d << shift;
    pmask |= (uint64_t)0xffu << shift;
    if (cd == need || shift == 0) break;
  }
  // in place: a kept key moves to an index no higher than the one it was read
  // from, and a chunk is read before any of its slots is written
  uint32_t kept = 0;
  for (uint32_t base = 0; base < my_cnt; base += 32) {
    const uint32_t i = base + (uint32_t)lane;
    const uint64_t v = i < my_cnt ? reg[i] : 0ull;
    const bool keep = i < my_cnt && v >= prefix;
    const uint32_t m = __ballot_sync(0xffffffffu, keep);
    const uint32_t at = kept + (uint32_t)__popc(m & ((1u << lane) - 1u));
    if (keep && IDX_IN_RANGE(at < kQ, hdr, 341)) reg[at] = v;
    kept += (uint32_t)__popc(m);
    __syncwarp();
  }
  // every region has been read for the histogram before any warp compacts
  // (the last barrier above); check the total
  if (lane == 0) bc[4 + qd] = kept;
  bar_sync(bar_id, kEpiThreads);
  if (qd == 0 && lane == 0) {
    if (bc[4] + bc[5] + bc[6] + bc[7] != (uint32_t)TOPK) raise_status(hdr, kErrInternal, 201);
    *tau_s = prefix;
  }
  bar_sync(bar_id, kEpiThreads);
  return kept;
}

struct UnitView {
  UnitInfo u;
  BlockInfo b;
};

// Schedule position of this CTA's i-th unit.  The planner orders the units
// longest first (or nearly so); band i (positions i*G .. i*G+G-1) is dealt in
// ascending CTA order when i is even and descending when odd, so a CTA that
// drew a longer unit of one band draws a shorter one of the next.
__device__ __forceinline__ int cta_unit(int i) {
  const int c = (i & 1) ? (int)(gridDim.x - 1u - blockIdx.x) : (int)blockIdx.x;
  return i * (int)gridDim.x + c;
}

__device__ __forceinline__ UnitView load_unit(const ScoreParams& p, int ui) {
  UnitView v;
  v.u = p.units[p.sched[ui]];
  v.b = p.blocks[v.u.block];
  return v;
}

// DYN: the CTAs claim schedule positions from a global counter (longest unit
// first) instead of taking the fixed deal of cta_unit; warp 0 claims and
// publishes each position in shared memory before the unit's query block
// arrives, and the other roles read it behind that barrier.  Chosen on the host
// for calls with several requests, whose units differ in length.
template <int MODE, int TOPK, bool DYN>
__global__ void __launch_bounds__(kThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                 const ScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  PlanHeader* hdr = p.hdr;
  // after an earlier error no unit is run; all threads take the same decision
  if (__syncthreads_or(read_status(hdr) != kOk)) return;
  const int n_units = hdr->n_units;

  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + kMiscAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc + kMiscTmem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int c = 0; c < kAccStages; ++c) {
      mbar_init(bar(kBarAccFull + c), 1);
      mbar_init(bar(kBarAccEmpty + c), kRowsPerBlock * kEpiThreads);
      mbar_init(bar(kBarMmaFinal + c), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarQFull + b), 1);
      mbar_init(bar(kBarQEmpty + b), kAccStages);  // one commit per MMA issuer
      mbar_init(bar(kBarEpiDone + b), (kThreads / 32) - kEpiWarp0);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto wait = [&](uint32_t b, uint32_t par, uint32_t site) -> bool {
    return mbar_wait(b, par, abort_flag, hdr, site);
  };
  volatile int32_t* unit_slot = reinterpret_cast<volatile int32_t*>(smem + kOffMisc + kMiscUnit);
  // dynamic mode: the schedule position of the CTA's unit i, published by warp
  // 0 before the query buffer's barrier completes (-1: no unit is left)
  auto claimed_unit = [&](int i) -> int {
    const uint32_t qpar = (uint32_t)(i >> 1) & 1u;
    if (!wait(bar(kBarQFull + (i & 1)), qpar, 330)) return -2;
    return unit_slot[i & 1];
  };

  if (warp == 0 || warp == kProducer2) {
    // ----------------------------------------------------- TMA producers ----
    // Two warps share the K ring: tile n of the CTA's sequence (stage
    // n % kStages) is handled by warp 0 when n is even and by the second
    // producer when n is odd.  Per tile the warp rearranges the two pages'
    // UE8M0 scales into the TMEM copy layout itself (operand row r of the
    // 128-row atom -> 32-bit word 4*(r%32) + r/32; lane i holds rows i, 32+i,
    // 64+i, 96+i), read one own tile ahead with plain loads, and issues the
    // two 4 KB page copies.  Warp 0 also loads each unit's query block.
    const uint32_t pw = warp == 0 ? 0u : 1u;
    if (lane == 0 && pw == 0) {
      prefetch_tmap(&tmap_k);
      prefetch_tmap(&tmap_q);
    }
    const uint32_t* kscale = reinterpret_cast<const uint32_t*>(p.k_scale);  // per page: 64 slot words
    uint32_t n_issued = 0;  // K tiles of the CTA's sequence so far (both producers)
    uint32_t q_issued[2] = {0, 0};
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int qb = i & 1;
      const uint32_t qpar = (uint32_t)(i >> 1) & 1u;
      int ui;
      if constexpr (DYN) {
        if (pw == 0) {
          // the query buffer is free again (units i - 2 done) before its
          // position slot is rewritten
          if (i >= 2) {
            ok = wait(bar(kBarQEmpty + qb), qpar ^ 1u, 300) &&
                 wait(bar(kBarEpiDone + qb), qpar ^ 1u, 301);
            if (!ok) break;
          }
          int c = 0;
          if (lane == 0) {
            // the first unit of CTA b is schedule position b (no round trip to
            // the counter when the call starts); the later ones are claimed
            // from position gridDim.x on
            c = i == 0 ? (int)blockIdx.x : (int)gridDim.x + (int)atomicAdd(&hdr->claim, 1u);
            if (c >= n_units) c = -1;
            unit_slot[qb] = c;
          }
          ui = __shfl_sync(0xffffffffu, c, 0);
          if (ui < 0) {
            if (lane == 0) mbar_arrive(bar(kBarQFull + qb));  // releases the other roles
            ++q_issued[qb];  // that arrival completed a phase of the buffer's barrier too
            break;
          }
        } else {
          ui = claimed_unit(i);
          if (ui < 0) {
            ok = ui == -1;
            break;
          }
        }
      } else {
        ui = cta_unit(i);
        if (ui >= n_units) break;
      }
      const UnitView uv = load_unit(p, ui);
      int32_t rs = 0, re = 0;
      bool act = false;
      if (lane < uv.b.nrows) {
        rs = p.row_start[uv.b.row0 + lane];
        re = p.row_end[uv.b.row0 + lane];
        act = (re - rs) > p.score_thr;
      }
      const uint32_t act_mask = __ballot_sync(0xffffffffu, act);
      if (pw == 0) {
        if (!DYN && i >= 2) {
          ok = wait(bar(kBarQEmpty + qb), qpar ^ 1u, 300) &&
               wait(bar(kBarEpiDone + qb), qpar ^ 1u, 301);
          if (!ok) break;
        }
        if (lane == 0) {
          uint32_t bytes = 2u * (uint32_t)uv.b.nrows * kRowSfBytes;
          for (int c = 0; c < kChunks; ++c)
            if ((act_mask >> c) & 1u) bytes += kRowBBytes;
          const uint32_t qf = bar(kBarQFull + qb);
          mbar_arrive_expect_tx(qf, bytes);
          for (int c = 0; c < kChunks; ++c)
            if ((act_mask >> c) & 1u)
              tma_load_2d(sbase + kOffB + qb * kBBytes + c * kRowBBytes, &tmap_q, 0,
                          (uv.b.row0 + c) * kHeads, qf);
          bulk_load(sbase + kOffSfbRaw + qb * kSfbAtomBytes,
                    p.q_scale + (int64_t)uv.b.row0 * kRowSfBytes, uv.b.nrows * kRowSfBytes, qf);
          bulk_load(sbase + kOffW + qb * kBlockWBytes, p.weights + (int64_t)uv.b.row0 * kHeads,
                    uv.b.nrows * kHeads * 4u, qf);
        }
        ++q_issued[qb];
      }
      const int32_t* row_pt = p.page_table + (int64_t)uv.b.req * p.max_pages;
      // row windows of the block, broadcast to every lane
      int32_t ws[kRowsPerBlock], we[kRowsPerBlock];
#pragma unroll
      for (int j = 0; j < kRowsPerBlock; ++j) {
        const bool aj = __shfl_sync(0xffffffffu, act, j);
        ws[j] = aj ? __shfl_sync(0xffffffffu, rs, j) : 0;
        we[j] = aj ? __shfl_sync(0xffffffffu, re, j) : 0;
      }
      // page-table entries of 32 consecutive logical pages, one per lane, read
      // only for pages that some row's window touches; the window always
      // covers the current tile and the warp's next one (two tiles later)
      int32_t pt_base = -64, pt_val = -1;
      uint32_t pt_need = 0;
      auto pages_of = [&](int tt, int32_t& pg0, int32_t& pg1, bool& need0, bool& need1) {
        const int32_t lp0 = 2 * tt, lp1 = 2 * tt + 1;
        need0 = (pt_need >> (lp0 - pt_base)) & 1u;
        need1 = (pt_need >> (lp1 - pt_base)) & 1u;
        const int32_t e0v = __shfl_sync(0xffffffffu, pt_val, lp0 - pt_base);
        const int32_t e1v = __shfl_sync(0xffffffffu, pt_val, lp1 - pt_base);
        pg0 = need0 ? e0v : -1;
        pg1 = need1 ? e1v : -1;
      };
      auto load_scales = [&](int32_t pg0, int32_t pg1, uint32_t (&w)[4]) {
        const bool v0 = pg0 >= 0 && pg0 < p.num_pages, v1 = pg1 >= 0 && pg1 < p.num_pages;
        if (p.k_scale_mma) {
          // already in copy order: slots lane and 32 + lane are one 8-byte word
          const uint2 a = v0 ? *reinterpret_cast<const uint2*>(
                                   kscale + (int64_t)pg0 * p.k_scale_stride + 2 * lane)
                             : make_uint2(0u, 0u);
          const uint2 b = v1 ? *reinterpret_cast<const uint2*>(
                                   kscale + (int64_t)pg1 * p.k_scale_stride + 2 * lane)
                             : make_uint2(0u, 0u);
          w[0] = a.x;
          w[1] = a.y;
          w[2] = b.x;
          w[3] = b.y;
        } else {
          w[0] = v0 ? kscale[(int64_t)pg0 * p.k_scale_stride + lane] : 0u;
          w[1] = v0 ? kscale[(int64_t)pg0 * p.k_scale_stride + 32 + lane] : 0u;
          w[2] = v1 ? kscale[(int64_t)pg1 * p.k_scale_stride + lane] : 0u;
          w[3] = v1 ? kscale[(int64_t)pg1 * p.k_scale_stride + 32 + lane] : 0u;
        }
      };
      uint32_t wnext[4] = {0u, 0u, 0u, 0u};
      bool have_next = false;
      uint32_t sf_over = 0;  // K scale bytes of this unit's pages outside the domain
      for (int t = uv.u.t_begin; t < uv.u.t_end; ++t) {
        const uint32_t n = n_issued++;
        if ((n & 1u) != pw) continue;
        const uint32_t st = n % kStages, sp = (n / kStages) & 1u;
        if (2 * t + 5 >= pt_base + 32) {
          pt_base = 2 * t;
          const int32_t lp = pt_base + lane;
          bool need = false;
#pragma unroll
          for (int j = 0; j < kRowsPerBlock; ++j)
            need |= ws[j] < (lp + 1) * kPage && we[j] > lp * kPage;
          need &= lp < p.max_pages;
          pt_need = __ballot_sync(0xffffffffu, need);
          pt_val = need ? row_pt[lp] : -1;
        }
        int32_t pg0, pg1;
        bool need0, need1;
        pages_of(t, pg0, pg1, need0, need1);
        uint32_t wcur[4];
        if (have_next) {
#pragma unroll
          for (int k = 0; k < 4; ++k) wcur[k] = wnext[k];
        } else {
          load_scales(pg0, pg1, wcur);
        }
        sf_over |= scale_bytes_over(wcur[0]) | scale_bytes_over(wcur[1]) |
                   scale_bytes_over(wcur[2]) | scale_bytes_over(wcur[3]);
        have_next = t + 2 < uv.u.t_end;
        if (have_next) {
          int32_t ng0, ng1;
          bool nn0, nn1;
          pages_of(t + 2, ng0, ng1, nn0, nn1);
          load_scales(ng0, ng1, wnext);
        }
        if (!wait(bar(kBarEmpty + st), sp ^ 1u, 302)) {
          ok = false;
          break;
        }
        // the stage's previous scale atom was read by the MMA that released it
        *reinterpret_cast<uint4*>(smem + kOffSfaAtom + st * 512u + 16u * lane) =
            make_uint4(wcur[0], wcur[1], wcur[2], wcur[3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const uint32_t fb = bar(kBarFull + st);
          const bool v0 = need0 && pg0 >= 0 && pg0 < p.num_pages;
          const bool v1 = need1 && pg1 >= 0 && pg1 < p.num_pages;
          // this is the page-table check of the scored rows' windows (the
          // finishing step checks the entries it maps for the other rows)
          if ((need0 && !v0) || (need1 && !v1)) raise_status(hdr, kErrInvalidPage, 303);
          const uint32_t bytes = ((uint32_t)v0 + (uint32_t)v1) * kPageBytes;
          if (bytes) {
            mbar_arrive_expect_tx(fb, bytes);
            const uint32_t a = sbase + kOffA + st * kABytes;
            if (v0) tma_load_3d(a, &tmap_k, 0, 0, pg0, fb);
            if (v1) tma_load_3d(a + kPageBytes, &tmap_k, 0, 0, pg1, fb);
          } else {
            mbar_arrive(fb);
          }
        }
      }
      if (__any_sync(0xffffffffu, sf_over != 0u) && lane == 0)
        raise_status(hdr, kErrInvalidValue, 304);
    }
    if (lane == 0) {
      // wait for this warp's copies in flight (its stages have parity pw)
      for (uint32_t s2 = pw; s2 < (uint32_t)kStages; s2 += 2) {
        const uint32_t uses = n_issued > s2 ? (n_issued - s2 + kStages - 1) / kStages : 0;
        if (uses) mbar_drain(bar(kBarFull + s2), (uses - 1u) & 1u, hdr, 305);
      }
      if (pw == 0)
        for (int b2 = 0; b2 < 2; ++b2)
          if (q_issued[b2]) mbar_drain(bar(kBarQFull + b2), (q_issued[b2] - 1u) & 1u, hdr, 306);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------ MMA issuers ----
    // Warp 1 + j issues the tiles n with n % 2 == j, all into accumulator
    // buffer j: a thread that issues MMAs stalls on its own shared-memory
    // accesses until they retire, so two issuers hide each other's waits.
    // Per unit the whole warp rearranges the query block's scales into its own
    // atom buffer; lane 0 copies them to TMEM and issues the tile MMAs.
    const uint32_t j = (uint32_t)warp - 1u;
    uint32_t n_seen = 0, own = 0;
    const uint64_t a_desc0 = desc_kmajor_sw64(sbase + kOffA);
    const uint64_t b_desc0 = desc_kmajor_sw64(sbase + kOffB);
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int qb = i & 1;
      const uint32_t qpar = (uint32_t)(i >> 1) & 1u;
      int ui;
      if constexpr (DYN) {
        ui = claimed_unit(i);
        if (ui < 0) break;
      } else {
        ui = cta_unit(i);
        if (ui >= n_units) break;
        if (!wait(bar(kBarQFull + qb), qpar, 310)) break;
      }
      const UnitInfo u = p.units[p.sched[ui]];
      // both issuers' copies from this atom buffer two units ago have completed
      if (i >= 2 && !wait(bar(kBarQEmpty + qb), qpar ^ 1u, 311)) break;
      const uint32_t atom_off = kOffSfbAtom + (2u * j + (uint32_t)qb) * kSfbAtomBytes;
      {
        const uint32_t* raw = reinterpret_cast<const uint32_t*>(smem + kOffSfbRaw + qb * kSfbAtomBytes);
        uint32_t* atom = reinterpret_cast<uint32_t*>(smem + atom_off);
#pragma unroll
        for (int k = 0; k < (int)kSfbAtoms * 4; ++k) {
          const int a = k >> 2, jj = k & 3;  // atom, 32-row group
          atom[a * 128 + 4 * lane + jj] = raw[a * 128 + 32 * jj + lane];
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t sfb = tmem + kColSfb + 4u * kSfbAtoms * (2u * j + (uint32_t)qb);
        for (uint32_t a = 0; a < kSfbAtoms; ++a)
          tc_cp_sf(sfb + 4u * a, desc_sf_block(sbase + atom_off + 512u * a));
        const uint64_t bd = b_desc0 + ((qb * kBBytes) >> 4);
        const uint32_t d = tmem + kColAcc + kAccCols * j;
        for (int t = u.t_begin; t < u.t_end; ++t) {
          const uint32_t n = n_seen++;
          if ((n & 1u) != j) continue;
          const uint32_t st = n % kStages, sp = (n / kStages) & 1u;
          // K tile and its scale atom landed
          if (!wait(bar(kBarFull + st), sp, 312)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa = tmem + kColSfa + 4u * st;
          tc_cp_sf(sfa, desc_sf_block(sbase + kOffSfaAtom + st * 512u));
          if (!wait(bar(kBarAccEmpty + j), (own & 1u) ^ 1u, 313)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // all rows of the block in one N = 192 instruction per K step; the
          // second K = 64 step advances both operands by 32 bytes
          const uint64_t ad = a_desc0 + ((st * kABytes) >> 4);
          tc_mma_mxf4(d, ad, bd, kIdescK0, sfa, sfb, 0u);
          tc_mma_mxf4(d, ad + 2, bd + 2, kIdescK1, sfa, sfb, 1u);
          tc_commit(bar(kBarAccFull + j));
          tc_commit(bar(kBarEmpty + st));
          ++own;
        }
        tc_commit(bar(kBarQEmpty + qb));
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0) {
      tc_commit(bar(kBarMmaFinal + j));
      mbar_drain(bar(kBarMmaFinal + j), 0, hdr, 314);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // --------------------------------------------------------- epilogue ----
    const int g = (warp - kEpiWarp0) >> 2;  // row of the block handled by this warpgroup
    const int qd = warp & 3;                 // TMEM lane quarter
    const int tg = qd * 32 + lane;           // slot within tile == thread in group
    const uint32_t bar_id = 1u + (uint32_t)g;
    constexpr uint32_t kCap = cand_cap(TOPK);
    uint64_t* tau_s = reinterpret_cast<uint64_t*>(smem + kOffMisc + kMiscTau) + g;
    uint32_t* bc = reinterpret_cast<uint32_t*>(smem + kOffMisc + kMiscBc) + 8 * g;
    uint32_t* wc_s = reinterpret_cast<uint32_t*>(smem + kOffMisc + kMiscWc) + 4 * g;
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kOffHist) + 256 * g;
    uint64_t* cand = reinterpret_cast<uint64_t*>(smem + kOffCand) + (size_t)g * kCap;
    uint32_t acc_use = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int qb = i & 1;
      const uint32_t qpar = (uint32_t)(i >> 1) & 1u;
      int ui;
      if constexpr (DYN) {
        ui = claimed_unit(i);
        if (ui < 0) {
          ok = ui == -1;
          break;
        }
      } else {
        ui = cta_unit(i);
        if (ui >= n_units) break;
      }
      const UnitView uv = load_unit(p, ui);
      const bool valid = g < uv.b.nrows;
      const int64_t row = uv.b.row0 + g;
      const int32_t s0 = valid ? p.row_start[row] : 0;
      const int32_t e0 = valid ? p.row_end[row] : 0;
      const bool act = valid && (e0 - s0) > p.score_thr;
      if (!act) {
        // this row is not scored, but every warpgroup releases each
        // accumulator buffer, so walk the unit's tiles
        for (int t = uv.u.t_begin; t < uv.u.t_end; ++t) {
          const uint32_t b = acc_use & 1u;
          if (!wait(bar(kBarAccFull + b), (acc_use >> 1) & 1u, 322)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mbar_arrive(bar(kBarAccEmpty + b));
          ++acc_use;
        }
        if (MODE == kModeSelect && valid && tg == 0) {
          const int64_t slot_idx = uv.b.slot0 + (int64_t)uv.u.k * uv.b.nrows + g;
          if (IDX_IN_RANGE(slot_idx >= 0 && slot_idx < hdr->n_row_slots, hdr, 343))
            p.cand_cnt[slot_idx] = 0;
        }
      } else {
        if (!DYN && !wait(bar(kBarQFull + qb), qpar, 320)) {
          ok = false;
        } else {
          uint64_t w2[32];  // the row's weights as packed pairs (heads 2p, 2p+1)
          const ulonglong2* wsrc =
              reinterpret_cast<const ulonglong2*>(smem + kOffW + qb * kBlockWBytes) + g * (kHeads / 4);
          auto load_w2 = [&]() {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const ulonglong2 v = wsrc[k];
              w2[2 * k] = v.x;
              w2[2 * k + 1] = v.y;
            }
          };
          load_w2();
          if (tg < kHeads) {
            // the row's query scales (one word per head) and weights must lie
            // in the accepted value domain
            const uint32_t qsf = reinterpret_cast<const uint32_t*>(
                smem + kOffSfbRaw + qb * kSfbAtomBytes + g * kRowSfBytes)[tg];
            const uint32_t wb = reinterpret_cast<const uint32_t*>(
                smem + kOffW + qb * kBlockWBytes + g * kHeads * 4)[tg];
            if (scale_bytes_over(qsf) != 0u || weight_out_of_domain(wb))
              raise_status(hdr, kErrInvalidValue, 323);
          }
          uint64_t tau = 0;    // threshold key: appended keys are >= tau
          uint32_t wcnt = 0;   // keys in this warp's append region
          uint64_t* wreg = cand + (uint32_t)qd * warp_region(TOPK);
          const uint32_t wreg_s = smem_u32(wreg);
          const uint32_t lt_mask = (1u << lane) - 1u;
          if constexpr (MODE == kModeSelect) {
            if (tg == 0) *tau_s = 0ull;
            bar_sync(bar_id, kEpiThreads);
          }
          const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16) + kColAcc + 64u * g;
          int check_in = kCheckTiles;  // tiles until the next over-limit check
          const uint32_t trig = (TOPK == 512 && uv.u.t_end - uv.u.t_begin <= kShortUnitTiles)
                                    ? kShortTrig
                                    : warp_region(TOPK) - kCheckTiles * 32u;
          // scored rows of the block: their warps take part in the votes (every
          // epilogue warp computes the same count from the same row windows)
          uint32_t n_act = 0;
          for (int j = 0; j < uv.b.nrows; ++j)
            n_act += (p.row_end[uv.b.row0 + j] - p.row_start[uv.b.row0 + j]) > p.score_thr;
          // A tile's score is reduced at the end of the tile; its select step
          // runs one tile late, at the end of the next tile, after that tile's
          // accumulator buffer has been released: nothing between the wait for
          // a buffer and its release delays the next MMA into it.  The first
          // call of a unit is a no-op (pwin false).
          float psc = 0.f;
          int32_t pslot = 0;
          bool pwin = false;
          auto tail = [&]() {
            if constexpr (MODE == kModeDense) {
              if (pwin && IDX_IN_RANGE((int64_t)pslot - p.dense_col0 >= 0 &&
                                           (int64_t)pslot - p.dense_col0 < p.dense_stride,
                                       hdr, 345))
                p.dense_out[row * p.dense_stride + (pslot - p.dense_col0)] = psc;
            } else {
              append_if(wcnt, wreg_s, psc, ~(uint32_t)pslot, tau, (uint32_t)pwin, lt_mask);
              // the region never holds more than its capacity
              if (!IDX_IN_RANGE(wcnt <= warp_region(TOPK), hdr, 342)) wcnt = warp_region(TOPK);
            }
          };
          for (int t = uv.u.t_begin; t < uv.u.t_end; ++t) {
            const uint32_t b = acc_use & 1u;
            const uint32_t ph = (acc_use >> 1) & 1u;
            if (!wait(bar(kBarAccFull + b), ph, 321)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t tb = lane_base + kAccCols * b;
            const int32_t slot = t * kTile + tg;
            const bool in_win = (uint32_t)(slot - s0) < (uint32_t)(e0 - s0);
            uint64_t acc[4];  // four packed partial sums
            // four 16-column TMEM loads, each issued before the previous
            // chunk is reduced (a wait covers every load issued before it)
            uint32_t xa[16], xb[16];
            auto dump = [&](const uint32_t(&x)[16], int h0) {
              if constexpr (MODE == kModeDense) {
                if (p.logits_out && in_win) {
                  float* lo = p.logits_out + (row * kHeads + h0) * p.logits_stride + slot;
#pragma unroll
                  for (int h = 0; h < 16; ++h) lo[(int64_t)h * p.logits_stride] = __uint_as_float(x[h]);
                }
              }
            };
            tmem_ld16(tb, xa);
            if constexpr (MODE == kModeDense) tail();  // (its registers fit better here)
            tmem_wait_ld16(xa);
            tmem_ld16(tb + 16u, xb);
            dump(xa, 0);
            head_sum_part<0>(xa, w2, acc);
            tmem_wait_ld16(xb);
            tmem_ld16(tb + 32u, xa);
            dump(xb, 16);
            head_sum_part<8>(xb, w2, acc);
            tmem_wait_ld16(xa);
            tmem_ld16(tb + 48u, xb);
            dump(xa, 32);
            head_sum_part<16>(xa, w2, acc);
            tmem_wait_ld16(xb);
            tc_fence_before();
            mbar_arrive(bar(kBarAccEmpty + b));
            ++acc_use;
            dump(xb, 48);
            head_sum_part<24>(xb, w2, acc);
            if constexpr (MODE == kModeSelect) tail();  // previous tile
            psc = head_sum_final(acc);
            pslot = slot;
            pwin = in_win;
            if constexpr (MODE == kModeSelect) {
              // every kCheckTiles tails the warps vote on compaction (no TMEM
              // load is in flight here)
              if (--check_in == 0) {
                check_in = kCheckTiles;
                const bool over = wcnt > trig;
                if (lane == 0) wc_s[qd] = wcnt;  // visible to the group after the vote
                // one vote for the whole block: when any row needs it, every
                // scored row compacts at the same tile, so that their pauses
                // (each holds the accumulator handshake of all 12 warps) overlap
                if (bar_red_or(kBarVote, n_act * kEpiThreads, over)) {
                  wcnt = sel_compact_regions<TOPK>(cand, wc_s, tau_s, hist, bc, wcnt, qd, lane,
                                                   bar_id, hdr);
                  tau = *(volatile uint64_t*)tau_s;
                  load_w2();  // the weights are not kept live across the compaction
                }
              }
            }
          }
          if (ok) tail();  // last tile of the unit
          if constexpr (MODE == kModeSelect) {
            if (ok) {
              const int64_t slot_idx = uv.b.slot0 + (int64_t)uv.u.k * uv.b.nrows + g;
              if (lane == 0) wc_s[qd] = wcnt;
              bar_sync(bar_id, kEpiThreads);
              wcnt = sel_compact_regions<TOPK>(cand, wc_s, tau_s, hist, bc, wcnt, qd, lane, bar_id,
                                               hdr);
              // the regions' survivors, region by region, to the unit's list
              if (lane == 0) wc_s[qd] = wcnt;
              bar_sync(bar_id, kEpiThreads);
              uint32_t pre = 0, n = 0;
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const uint32_t c = ((volatile uint32_t*)wc_s)[w];
                pre += w < qd ? c : 0u;
                n += c;
              }
              const bool slot_ok = IDX_IN_RANGE(
                  slot_idx >= 0 && slot_idx < hdr->n_row_slots && pre + wcnt <= (uint32_t)TOPK, hdr,
                  344);
              uint64_t* dst = p.cand_keys + slot_idx * TOPK + pre;
              for (uint32_t e = lane; slot_ok && e < wcnt; e += 32) dst[e] = wreg[e];
              if (tg == 0 && slot_ok) p.cand_cnt[slot_idx] = n;
              bar_sync(bar_id, kEpiThreads);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarEpiDone + qb));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int MODE, int TOPK, bool DYN>
cudaError_t launch_score_t(const CUtensorMap& tk, const CUtensorMap& tq, const ScoreParams& p,
                           int grid, cudaStream_t stream) {
  const size_t smem = smem_bytes_for(MODE, TOPK);
  static std::atomic<bool> done[64] = {};
  cudaError_t err = set_smem_once(score_kernel<MODE, TOPK, DYN>, (int)smem, done);
  if (err != cudaSuccess) return err;
  score_kernel<MODE, TOPK, DYN><<<grid, kThreads, smem, stream>>>(tk, tq, p);
  return cudaGetLastError();
}

}  // namespace

size_t score_smem_bytes(int mode, int topk) { return smem_bytes_for(mode, topk); }

cudaError_t launch_score(const CUtensorMap& tmap_k, const CUtensorMap& tmap_q, const ScoreParams& p,
                         int grid, cudaStream_t stream) {
  if (p.mode == kModeDense)
    return launch_score_t<kModeDense, 0, false>(tmap_k, tmap_q, p, grid, stream);
  if (p.topk == 512)
    return p.dyn ? launch_score_t<kModeSelect, 512, true>(tmap_k, tmap_q, p, grid, stream)
                 : launch_score_t<kModeSelect, 512, false>(tmap_k, tmap_q, p, grid, stream);
  if (p.topk == 1024)
    return p.dyn ? launch_score_t<kModeSelect, 1024, true>(tmap_k, tmap_q, p, grid, stream)
                 : launch_score_t<kModeSelect, 1024, false>(tmap_k, tmap_q, p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace idxk
