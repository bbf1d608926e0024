// Fused FP4 paged-MQA scorer for sm_103a (one persistent CTA per SM).
//
// Per work unit (a block of up to 6 rows of one request x a run of 128-slot K
// tiles; see idx_internal.h) the CTA
//   * stages each K tile (2 pages of 64 slots x 64 B of E2M1 codes, plus their
//     UE8M0 scales) with TMA, the page looked up in the page table, and the
//     query block (6 rows x 64 heads x 64 B + scales + weights) once per unit;
//   * runs the contraction logit[s, (r,h)] = sum_d k[s,d] q[r,h,d] on the
//     tcgen05 block-scaled FP4 MMA (kind::mxf4, scale vector 32, M = 128 slots,
//     N = 2 rows x 64 heads, K = 64 per instruction) into TMEM accumulators;
//   * drains TMEM in three epilogue warpgroups (one per accumulator, two rows
//     each): score[r, s] = sum_h w[r,h] * max(logit, 0) in fp32, then either
//     streams the (score, slot) keys through the bounded shared-memory TopK
//     (select mode) or writes the fp32 scores (dense / debug mode).
// This realises the fused scorer + CTA-local exact TopK of "[FlyDSL] Add FP4
// LiteTopK prefill operator" (ROCm/aiter#5309, Implementation) and
// "[FlyDSL][DSv4] Prototype FP4 MQA streaming TopK" (ROCm/aiter#5282, Changes
// and Scope), re-designed around TMA, tcgen05 and TMEM.
//
// Warp roles (512 threads): warp 0 TMA producer, warp 1 TMEM allocator + MMA
// issuer (+ rearranges scale factors into the TMEM copy layout), warps 4..15
// epilogue (warpgroup g = accumulator g; warp w reads TMEM lanes 32*(w%4)...).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "idx_device.cuh"
#include "idx_launch.h"
#include "idx_select.cuh"

namespace idxk {

namespace {

constexpr int kThreads = 512;
constexpr int kStages = 4;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiThreads = 128;  // one warpgroup

constexpr uint32_t kPageBytes = kPage * kDimBytes;                        // 4096
constexpr uint32_t kPageSfBytes = kPage * kNumSF;                         // 256
constexpr uint32_t kABytes = kTile * kDimBytes;                           // 8192
constexpr uint32_t kChunkBBytes = kRowsPerChunk * kHeads * kDimBytes;     // 8192
constexpr uint32_t kBBytes = kChunks * kChunkBBytes;                      // 24576
constexpr uint32_t kRowSfBytes = kHeads * kNumSF;                         // 256
constexpr uint32_t kBlockSfBytes = kRowsPerBlock * kRowSfBytes;           // 1536
constexpr uint32_t kBlockWBytes = kRowsPerBlock * kHeads * 4;             // 1536

constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kABytes;
constexpr uint32_t kOffSfaRaw = kOffB + 2 * kBBytes;
constexpr uint32_t kOffSfaAtom = kOffSfaRaw + kStages * 512;
constexpr uint32_t kOffSfbRaw = kOffSfaAtom + kStages * 512;
constexpr uint32_t kOffSfbAtom = kOffSfbRaw + 2 * kBlockSfBytes;
constexpr uint32_t kOffW = kOffSfbAtom + 2 * kBlockSfBytes;
constexpr uint32_t kOffBar = kOffW + 2 * kBlockWBytes;
constexpr uint32_t kOffMisc = kOffBar + 256;
constexpr uint32_t kOffHist = kOffMisc + 256;
constexpr uint32_t kOffCand = kOffHist + kChunks * 256 * 4;
static_assert(kOffB % 1024 == 0 && kOffA % 1024 == 0, "operand buffers must be 1 KB aligned");
static_assert(kOffCand % 16 == 0, "candidate buffer alignment");

// misc region
constexpr uint32_t kMiscTmem = 0, kMiscAbort = 4, kMiscCnt = 8, kMiscTau = 32, kMiscBc = 80;

// barriers (8 bytes each)
constexpr int kBarFull = 0, kBarEmpty = 4, kBarAccFull = 8, kBarAccEmpty = 11, kBarQFull = 14,
              kBarQEmpty = 16, kBarEpiDone = 18, kBarMmaFinal = 20;

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColAcc = 0;      // + 128 * chunk
constexpr uint32_t kColSfa = 384;    // + 4 * stage
constexpr uint32_t kColSfb = 400;    // + 12 * q-buffer + 4 * chunk

constexpr uint32_t kIdescK0 = idesc_mxf4(128, kRowsPerChunk * kHeads, 0);
constexpr uint32_t kIdescK1 = idesc_mxf4(128, kRowsPerChunk * kHeads, 2);

__host__ __device__ constexpr uint32_t cand_cap(int topk) { return topk > 0 ? 2u * (uint32_t)topk : 0u; }

__host__ __device__ constexpr size_t smem_bytes_for(int mode, int topk) {
  return 1024 + kOffCand +
         (mode == kModeSelect ? (size_t)kRowsPerBlock * cand_cap(topk) * sizeof(uint64_t) : 0);
}

// Bounded wait for the teardown: ignores the abort flag.
__device__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > 200000000ull) break;  // 0.2 s
  }
}

// score = sum over heads of w * max(logit, 0); heads split over two packed
// fp32 accumulators (even/odd pairs), summed at the end.  The fused and the
// dense paths share this function, so their scores are bit-identical.
__device__ __forceinline__ float head_sum(const uint32_t (&xa)[32], const uint32_t (&xb)[32],
                                          const float* w) {
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int h = 0; h < 32; h += 4) {
    const float4 wv = *reinterpret_cast<const float4*>(w + h);
    const float2 a = make_float2(fmaxf(__uint_as_float(xa[h]), 0.f), fmaxf(__uint_as_float(xa[h + 1]), 0.f));
    const float2 b = make_float2(fmaxf(__uint_as_float(xa[h + 2]), 0.f), fmaxf(__uint_as_float(xa[h + 3]), 0.f));
    acc0 = __ffma2_rn(a, make_float2(wv.x, wv.y), acc0);
    acc1 = __ffma2_rn(b, make_float2(wv.z, wv.w), acc1);
  }
#pragma unroll
  for (int h = 0; h < 32; h += 4) {
    const float4 wv = *reinterpret_cast<const float4*>(w + 32 + h);
    const float2 a = make_float2(fmaxf(__uint_as_float(xb[h]), 0.f), fmaxf(__uint_as_float(xb[h + 1]), 0.f));
    const float2 b = make_float2(fmaxf(__uint_as_float(xb[h + 2]), 0.f), fmaxf(__uint_as_float(xb[h + 3]), 0.f));
    acc0 = __ffma2_rn(a, make_float2(wv.x, wv.y), acc0);
    acc1 = __ffma2_rn(b, make_float2(wv.z, wv.w), acc1);
  }
  return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

struct UnitView {
  UnitInfo u;
  BlockInfo b;
};

__device__ __forceinline__ UnitView load_unit(const ScoreParams& p, int ui) {
  UnitView v;
  v.u = p.units[p.sched[ui]];
  v.b = p.blocks[v.u.block];
  return v;
}

template <int MODE, int TOPK>
__global__ void __launch_bounds__(kThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                 const ScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  PlanHeader* hdr = p.hdr;
  if (read_status(hdr) != kOk) return;
  const int n_units = hdr->n_units;

  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + kMiscAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc + kMiscTmem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int c = 0; c < kChunks; ++c) {
      mbar_init(bar(kBarAccFull + c), 1);
      mbar_init(bar(kBarAccEmpty + c), 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarQFull + b), 1);
      mbar_init(bar(kBarQEmpty + b), 1);
      mbar_init(bar(kBarEpiDone + b), (kThreads / 32) - kEpiWarp0);
    }
    mbar_init(bar(kBarMmaFinal), 1);
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

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer ----
    if (lane == 0) {
      prefetch_tmap(&tmap_k);
      prefetch_tmap(&tmap_q);
    }
    uint32_t stage = 0, sphase = 0;
    uint32_t k_issued[kStages] = {0, 0, 0, 0};
    uint32_t q_issued[2] = {0, 0};
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int ui = blockIdx.x + i * gridDim.x;
      if (ui >= n_units) break;
      const UnitView uv = load_unit(p, ui);
      const int qb = i & 1;
      const uint32_t qpar = (uint32_t)(i >> 1) & 1u;
      int32_t rs = 0, re = 0;
      bool act = false;
      if (lane < uv.b.nrows) {
        rs = p.row_start[uv.b.row0 + lane];
        re = p.row_end[uv.b.row0 + lane];
        act = (re - rs) > p.score_thr;
      }
      const uint32_t act_mask = __ballot_sync(0xffffffffu, act);
      if (i >= 2) {
        ok = mbar_wait(bar(kBarQEmpty + qb), qpar ^ 1u, abort_flag, hdr, 300) &&
             mbar_wait(bar(kBarEpiDone + qb), qpar ^ 1u, abort_flag, hdr, 301);
        if (!ok) break;
      }
      if (lane == 0) {
        uint32_t bytes = 2u * (uint32_t)uv.b.nrows * kRowSfBytes;
        for (int c = 0; c < kChunks; ++c)
          if ((act_mask >> (2 * c)) & 3u) bytes += kChunkBBytes;
        const uint32_t qf = bar(kBarQFull + qb);
        mbar_arrive_expect_tx(qf, bytes);
        for (int c = 0; c < kChunks; ++c)
          if ((act_mask >> (2 * c)) & 3u)
            tma_load_2d(sbase + kOffB + qb * kBBytes + c * kChunkBBytes, &tmap_q, 0,
                        (uv.b.row0 + kRowsPerChunk * c) * kHeads, qf);
        bulk_load(sbase + kOffSfbRaw + qb * kBlockSfBytes,
                  p.q_scale + (int64_t)uv.b.row0 * kRowSfBytes, uv.b.nrows * kRowSfBytes, qf);
        bulk_load(sbase + kOffW + qb * kBlockWBytes, p.weights + (int64_t)uv.b.row0 * kHeads,
                  uv.b.nrows * kHeads * 4u, qf);
      }
      ++q_issued[qb];
      const int32_t* row_pt = p.page_table + (int64_t)uv.b.req * p.max_pages;
      for (int t = uv.u.t_begin; t < uv.u.t_end; ++t) {
        if (!mbar_wait(bar(kBarEmpty + stage), sphase ^ 1u, abort_flag, hdr, 302)) {
          ok = false;
          break;
        }
        const int32_t lp0 = 2 * t, lp1 = 2 * t + 1;
        const bool need0 = __any_sync(0xffffffffu, act && rs < (lp0 + 1) * kPage && re > lp0 * kPage);
        const bool need1 = __any_sync(0xffffffffu, act && rs < (lp1 + 1) * kPage && re > lp1 * kPage);
        if (lane == 0) {
          const uint32_t fb = bar(kBarFull + stage);
          const int32_t pg0 = need0 ? row_pt[lp0] : -1;
          const int32_t pg1 = need1 ? row_pt[lp1] : -1;
          const bool v0 = need0 && pg0 >= 0 && pg0 < p.num_pages;
          const bool v1 = need1 && pg1 >= 0 && pg1 < p.num_pages;
          if ((need0 && !v0) || (need1 && !v1)) raise_status(hdr, kErrInvalidPage, 303);
          const uint32_t bytes = ((uint32_t)v0 + (uint32_t)v1) * (kPageBytes + kPageSfBytes);
          if (bytes) {
            mbar_arrive_expect_tx(fb, bytes);
            const uint32_t a = sbase + kOffA + stage * kABytes;
            const uint32_t sf = sbase + kOffSfaRaw + stage * 512u;
            if (v0) {
              tma_load_2d(a, &tmap_k, 0, pg0 * kPage, fb);
              bulk_load(sf, p.k_scale + (int64_t)pg0 * kPageSfBytes, kPageSfBytes, fb);
            }
            if (v1) {
              tma_load_2d(a + kPageBytes, &tmap_k, 0, pg1 * kPage, fb);
              bulk_load(sf + kPageSfBytes, p.k_scale + (int64_t)pg1 * kPageSfBytes, kPageSfBytes, fb);
            }
          } else {
            mbar_arrive(fb);
          }
        }
        ++k_issued[stage];
        if (++stage == kStages) {
          stage = 0;
          sphase ^= 1u;
        }
      }
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (k_issued[s]) mbar_drain(bar(kBarFull + s), (k_issued[s] - 1u) & 1u);
      for (int b = 0; b < 2; ++b)
        if (q_issued[b]) mbar_drain(bar(kBarQFull + b), (q_issued[b] - 1u) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer ----
    uint32_t stage = 0, sphase = 0;
    uint32_t acc_use[kChunks] = {0, 0, 0};
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int ui = blockIdx.x + i * gridDim.x;
      if (ui >= n_units) break;
      const UnitView uv = load_unit(p, ui);
      const int qb = i & 1;
      const uint32_t qpar = (uint32_t)(i >> 1) & 1u;
      bool act = false;
      if (lane < uv.b.nrows) {
        const int32_t rs = p.row_start[uv.b.row0 + lane], re = p.row_end[uv.b.row0 + lane];
        act = (re - rs) > p.score_thr;
      }
      const uint32_t act_mask = __ballot_sync(0xffffffffu, act);
      uint32_t cmask = 0;
      for (int c = 0; c < kChunks; ++c)
        if ((act_mask >> (2 * c)) & 3u) cmask |= 1u << c;
      if (!mbar_wait(bar(kBarQFull + qb), qpar, abort_flag, hdr, 310)) break;
      if (i >= 2 && !mbar_wait(bar(kBarQEmpty + qb), qpar ^ 1u, abort_flag, hdr, 311)) break;
      {
        // query scales [row][head][4] -> per chunk of 128 (row, head) rows, the
        // 32x16-byte TMEM copy layout: row n -> word 4*(n%32) + n/32
        const uint32_t* raw = reinterpret_cast<const uint32_t*>(smem + kOffSfbRaw + qb * kBlockSfBytes);
        uint32_t* atom = reinterpret_cast<uint32_t*>(smem + kOffSfbAtom + qb * kBlockSfBytes);
        for (int idx = lane; idx < kChunks * 128; idx += 32) {
          const int c = idx >> 7, n = idx & 127;
          atom[c * 128 + 4 * (n & 31) + (n >> 5)] = raw[idx];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          for (int c = 0; c < kChunks; ++c)
            if ((cmask >> c) & 1u)
              tc_cp_sf(tmem + kColSfb + 12u * qb + 4u * c,
                       desc_sf_block(sbase + kOffSfbAtom + qb * kBlockSfBytes + 512u * c));
        }
        __syncwarp();
      }
      for (int t = uv.u.t_begin; t < uv.u.t_end && ok; ++t) {
        if (!mbar_wait(bar(kBarFull + stage), sphase, abort_flag, hdr, 312)) {
          ok = false;
          break;
        }
        {
          const uint32_t* raw = reinterpret_cast<const uint32_t*>(smem + kOffSfaRaw + stage * 512u);
          uint32_t* atom = reinterpret_cast<uint32_t*>(smem + kOffSfaAtom + stage * 512u);
          for (int idx = lane; idx < 128; idx += 32) atom[4 * (idx & 31) + (idx >> 5)] = raw[idx];
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tc_fence_after();
            tc_cp_sf(tmem + kColSfa + 4u * stage, desc_sf_block(sbase + kOffSfaAtom + stage * 512u));
          }
          __syncwarp();
        }
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          if (!((cmask >> c) & 1u)) continue;
          if (!mbar_wait(bar(kBarAccEmpty + c), (acc_use[c] & 1u) ^ 1u, abort_flag, hdr, 313)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            tc_fence_after();
            const uint64_t ad = desc_kmajor_sw64(sbase + kOffA + stage * kABytes);
            const uint64_t bd = desc_kmajor_sw64(sbase + kOffB + qb * kBBytes + c * kChunkBBytes);
            const uint32_t d = tmem + kColAcc + 128u * c;
            const uint32_t sfa = tmem + kColSfa + 4u * stage;
            const uint32_t sfb = tmem + kColSfb + 12u * qb + 4u * c;
            tc_mma_mxf4(d, ad, bd, kIdescK0, sfa, sfb, 0u);
            // second K=64 step: operands advance 32 bytes along K
            tc_mma_mxf4(d, ad + 2, bd + 2, kIdescK1, sfa, sfb, 1u);
            tc_commit(bar(kBarAccFull + c));
          }
          __syncwarp();
          ++acc_use[c];
        }
        if (!ok) break;
        if (lane == 0) tc_commit(bar(kBarEmpty + stage));
        __syncwarp();
        if (++stage == kStages) {
          stage = 0;
          sphase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(bar(kBarQEmpty + qb));
      __syncwarp();
    }
    if (lane == 0) {
      tc_commit(bar(kBarMmaFinal));
      mbar_drain(bar(kBarMmaFinal), 0);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // --------------------------------------------------------- epilogue ----
    const int g = (warp - kEpiWarp0) >> 2;  // accumulator / warpgroup
    const int qd = warp & 3;                 // TMEM lane quarter
    const int tg = qd * 32 + lane;           // slot within tile == thread in group
    const uint32_t bar_id = 1u + (uint32_t)g;
    constexpr uint32_t kCap = cand_cap(TOPK);
    uint32_t* cnt_s = reinterpret_cast<uint32_t*>(smem + kOffMisc + kMiscCnt);
    uint64_t* tau_s = reinterpret_cast<uint64_t*>(smem + kOffMisc + kMiscTau);
    uint32_t* bc = reinterpret_cast<uint32_t*>(smem + kOffMisc + kMiscBc) + 4 * g;
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kOffHist) + 256 * g;
    uint64_t* cand = reinterpret_cast<uint64_t*>(smem + kOffCand);
    uint32_t acc_use = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int ui = blockIdx.x + i * gridDim.x;
      if (ui >= n_units) break;
      const UnitView uv = load_unit(p, ui);
      const int qb = i & 1;
      const uint32_t qpar = (uint32_t)(i >> 1) & 1u;
      int32_t s_j[2], e_j[2];
      bool act_j[2], valid_j[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int rj = kRowsPerChunk * g + j;
        valid_j[j] = rj < uv.b.nrows;
        s_j[j] = valid_j[j] ? p.row_start[uv.b.row0 + rj] : 0;
        e_j[j] = valid_j[j] ? p.row_end[uv.b.row0 + rj] : 0;
        act_j[j] = valid_j[j] && (e_j[j] - s_j[j]) > p.score_thr;
      }
      if (act_j[0] || act_j[1]) {
        if (!mbar_wait(bar(kBarQFull + qb), qpar, abort_flag, hdr, 320)) {
          ok = false;
        } else {
          const float* wrow = reinterpret_cast<const float*>(smem + kOffW + qb * kBlockWBytes);
          uint64_t tau[2] = {0ull, 0ull};
          if constexpr (MODE == kModeSelect) {
            if (tg < 2) {
              cnt_s[kRowsPerChunk * g + tg] = 0;
              tau_s[kRowsPerChunk * g + tg] = 0ull;
            }
            bar_sync(bar_id, kEpiThreads);
          }
          for (int t = uv.u.t_begin; t < uv.u.t_end; ++t) {
            if (!mbar_wait(bar(kBarAccFull + g), acc_use & 1u, abort_flag, hdr, 321)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const int32_t slot = t * kTile + tg;
            const uint32_t tbase = tmem + ((uint32_t)(qd * 32) << 16) + kColAcc + 128u * g;
            bool over = false;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              if (!act_j[j]) continue;
              const int rj = kRowsPerChunk * g + j;
              uint32_t xa[32], xb[32];
              tmem_ld32(tbase + 64u * j, xa);
              tmem_ld32(tbase + 64u * j + 32u, xb);
              tmem_wait_ld();
              if (j == 1 || !act_j[1]) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarAccEmpty + g));
              }
              const float sc = head_sum(xa, xb, wrow + rj * kHeads);
              const bool in_win = slot >= s_j[j] && slot < e_j[j];
              if constexpr (MODE == kModeDense) {
                const int64_t row = uv.b.row0 + rj;
                if (in_win) {
                  p.dense_out[row * p.dense_stride + slot] = sc;
                  if (p.logits_out) {
                    float* lo = p.logits_out + row * kHeads * p.logits_stride + slot;
#pragma unroll
                    for (int h = 0; h < 32; ++h) lo[(int64_t)h * p.logits_stride] = __uint_as_float(xa[h]);
#pragma unroll
                    for (int h = 0; h < 32; ++h)
                      lo[(int64_t)(32 + h) * p.logits_stride] = __uint_as_float(xb[h]);
                  }
                }
              } else {
                const uint64_t key = order_key(sc, slot);
                const bool pass = in_win && key >= tau[j];
                over |= sel_append(cand + (size_t)rj * kCap, cnt_s + rj, kCap, kCap - kEpiThreads,
                                   pass, key);
              }
            }
            ++acc_use;
            if constexpr (MODE == kModeSelect) {
              if (bar_red_or(bar_id, kEpiThreads, over)) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                  if (!act_j[j]) continue;
                  const int rj = kRowsPerChunk * g + j;
                  if (*(volatile uint32_t*)(cnt_s + rj) > kCap - kEpiThreads)
                    sel_compact<kEpiThreads, kCap>(cand + (size_t)rj * kCap, cnt_s + rj, tau_s + rj,
                                                   hist, bc, (uint32_t)TOPK, tg, bar_id, hdr);
                  tau[j] = *(volatile uint64_t*)(tau_s + rj);
                }
              }
            }
          }
          if constexpr (MODE == kModeSelect) {
           if (ok) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int rj = kRowsPerChunk * g + j;
              if (!valid_j[j]) continue;
              const int64_t slot_idx = uv.b.slot0 + (int64_t)uv.u.k * uv.b.nrows + rj;
              if (!act_j[j]) {
                if (tg == 0) p.cand_cnt[slot_idx] = 0;
                continue;
              }
              sel_compact<kEpiThreads, kCap>(cand + (size_t)rj * kCap, cnt_s + rj, tau_s + rj, hist,
                                             bc, (uint32_t)TOPK, tg, bar_id, hdr);
              const uint32_t n = min(*(volatile uint32_t*)(cnt_s + rj), (uint32_t)TOPK);
              uint64_t* dst = p.cand_keys + slot_idx * TOPK;
              const uint64_t* src = cand + (size_t)rj * kCap;
              for (uint32_t e = tg; e < n; e += kEpiThreads) dst[e] = src[e];
              if (tg == 0) p.cand_cnt[slot_idx] = n;
            }
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

template <int MODE, int TOPK>
cudaError_t launch_score_t(const CUtensorMap& tk, const CUtensorMap& tq, const ScoreParams& p,
                           int grid, cudaStream_t stream) {
  const size_t smem = smem_bytes_for(MODE, TOPK);
  cudaError_t err = cudaFuncSetAttribute(score_kernel<MODE, TOPK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  score_kernel<MODE, TOPK><<<grid, kThreads, smem, stream>>>(tk, tq, p);
  return cudaGetLastError();
}

}  // namespace

size_t score_smem_bytes(int mode, int topk) { return smem_bytes_for(mode, topk); }

cudaError_t launch_score(const CUtensorMap& tmap_k, const CUtensorMap& tmap_q, const ScoreParams& p,
                         int grid, cudaStream_t stream) {
  if (p.mode == kModeDense) return launch_score_t<kModeDense, 0>(tmap_k, tmap_q, p, grid, stream);
  if (p.topk == 512) return launch_score_t<kModeSelect, 512>(tmap_k, tmap_q, p, grid, stream);
  if (p.topk == 1024) return launch_score_t<kModeSelect, 1024>(tmap_k, tmap_q, p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace idxk
