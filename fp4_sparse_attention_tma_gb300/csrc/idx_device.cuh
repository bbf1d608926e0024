// Device helpers for the sm_103a kernels: inline PTX for mbarriers, TMA,
// tcgen05 (TMEM allocation, block-scaled FP4 MMA, TMEM loads, SMEM->TMEM scale
// copies), the 64-bit order key of the selection, and bounded waits that turn a
// would-be hang into an error status.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "idx_internal.h"

namespace idxk {

// ---------------------------------------------------------------- status ----

__device__ __forceinline__ void raise_status(PlanHeader* hdr, uint32_t code, uint32_t site) {
  if (atomicCAS(&hdr->status, (uint32_t)kOk, code) == kOk) {
    atomicExch(&hdr->err_site, site);
  }
}

__device__ __forceinline__ uint32_t read_status(const PlanHeader* hdr) {
  return *(volatile const uint32_t*)&hdr->status;
}

// Software range checks of the debug build (compiled with -DIDX_DEBUG_BOUNDS;
// it stands in for a memory checker): IDX_IN_RANGE(cond, hdr, site) is false,
// and records kErrInternal with `site`, when an index is outside its buffer, so
// that the caller skips the access and the call fails closed.  In the release
// build it is the constant true and costs nothing.
#ifdef IDX_DEBUG_BOUNDS
__device__ __forceinline__ bool idx_in_range(bool ok, PlanHeader* hdr, uint32_t site) {
  if (!ok) raise_status(hdr, kErrInternal, site);
  return ok;
}
#define IDX_IN_RANGE(cond, hdr, site) ::idxk::idx_in_range((cond), (hdr), (site))
#else
#define IDX_IN_RANGE(cond, hdr, site) true
#endif

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A bounded wait gives up after this long and reports kErrTimeout.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// ----------------------------------------------------------- value domain ----
// Nonzero when some byte of `w` exceeds kMaxScaleByte (167 = 0xA7): a byte b is
// >= 168 exactly when its top bit is set and (b & 0x7F) + 88 carries into bit 7
// (no carry crosses bytes, since (b & 0x7F) + 88 <= 0xD7).
__device__ __forceinline__ uint32_t scale_bytes_over(uint32_t w) {
  static_assert(kMaxScaleByte == 167, "the byte test below is written for 167");
  return ((w & 0x7F7F7F7Fu) + 0x58585858u) & w & 0x80808080u;
}

// True when the fp32 weight with bits `b` is NaN, infinite or above 2^24 in magnitude.
__device__ __forceinline__ bool weight_out_of_domain(uint32_t b) {
  return (b & 0x7FFFFFFFu) > kMaxAbsWeightBits;
}

// ------------------------------------------------------------- order key ----
// Total order of (score, logical index): score descending with NaN below every
// number and +0 above -0, then index ascending.  The 32-bit score key is
// monotone in that order; the low word holds ~index so that the lower index
// gets the larger composite key.  Key 0 never occurs for an index < 2^31, so it
// serves as an empty sentinel.
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t b = __float_as_uint(x);
  if (x != x) return 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ uint64_t order_key(float score, int32_t idx) {
  return ((uint64_t)score_key(score) << 32) | (uint64_t)(~(uint32_t)idx);
}

__device__ __forceinline__ int32_t key_index(uint64_t key) {
  return (int32_t)(~(uint32_t)(key & 0xffffffffu));
}

// The score of a key (the inverse of score_key on its high word); the empty
// key 0 gives NaN.
__device__ __forceinline__ float key_score(uint64_t key) {
  const uint32_t k = (uint32_t)(key >> 32);
  const uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return key == 0ull ? __uint_as_float(0x7FC00000u) : __uint_as_float(b);
}

// ------------------------------------------------------------- smem / PTX ----

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of parity `parity` of `bar` to complete.  Gives up when
// *abort becomes nonzero or after kWaitLimitNs, setting *abort and the status.
static __device__ __noinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                               PlanHeader* hdr, uint32_t site) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (*abort) return false;
      uint64_t now = global_timer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kWaitLimitNs) {
        *abort = 1;
        raise_status(hdr, kErrTimeout, site);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          PlanHeader* hdr, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_bounded(bar, parity, abort, hdr, site);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA: 2D tiled tensor load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// TMA: 3D tiled tensor load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, int32_t z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Bulk (non-tensor) copy global -> shared; both addresses 16-byte aligned,
// size a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"((uint64_t)src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// Named barrier over `count` threads with an OR-reduction of `pred`.
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t count, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t count) {
  asm volatile("barrier.cta.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ----------------------------------------------------------------- tcgen05 ---

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Copy a 32-row x 16-byte scale-factor block from shared memory into TMEM,
// replicated into all four 32-lane groups.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T with UE8M0 block-32 scales, FP4 E2M1 operands.
__device__ __forceinline__ void tc_mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.  The registers are valid only
// after tmem_wait_ld16 on the same array.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Waits for every outstanding tcgen05.ld of this thread; naming the
// destination registers keeps the compiler from using them earlier.
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Shared-memory matrix descriptor (tcgen05 layout): K-major operand stored as
// 64-byte rows with the 64-byte swizzle that TMA applies; 8-row groups are
// 512 bytes apart.  Buffers are 1024-byte aligned, so the base offset is 0.
__device__ __forceinline__ uint64_t desc_kmajor_sw64(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16)  // leading offset (unused)
         | ((uint64_t)(512 >> 4) << 32)                                // 8-row group stride
         | ((uint64_t)1 << 46)                                         // descriptor version
         | ((uint64_t)4 << 61);                                        // 64-byte swizzle
}

// Descriptor of a 32-row x 16-byte block (no swizzle; 8-row groups 128 B apart)
// for the scale-factor copy into TMEM.
__device__ __forceinline__ uint64_t desc_sf_block(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor: kind::mxf4, E2M1 x E2M1, UE8M0 scales, K-major A/B,
// shape M x N; sf_id selects which two scale bytes (k-blocks) of each TMEM
// scale word this K=64 step uses (0 -> bytes 0,1; 2 -> bytes 2,3).
__host__ __device__ constexpr uint32_t idesc_mxf4(uint32_t M, uint32_t N, uint32_t sf_id) {
  return (sf_id << 4)            // B scale-factor id
         | (1u << 7)             // A format: E2M1
         | (1u << 10)            // B format: E2M1
         | ((N >> 3) << 17)      // N / 8
         | (1u << 23)            // scale format: UE8M0
         | ((M >> 4) << 24)      // M / 16
         | (sf_id << 29);        // A scale-factor id
}

}  // namespace idxk
