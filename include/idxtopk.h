/*
 * idxtopk.h -- C ABI of the GB300 (sm_103a) FP4 paged-MQA indexer prefill with
 * fused exact TopK.
 *
 * The operation (defined by "[FlyDSL] Add FP4 LiteTopK prefill operator",
 * ROCm/aiter#5309, Summary and Implementation, and "[FlyDSL][DSv4] Prototype
 * FP4 MQA streaming TopK", ROCm/aiter#5282, Changes and Scope):
 *
 *   for every query row r of request req = row_req[r] and window
 *   [start, end) = [row_start[r], row_end[r]) of logical C4 positions:
 *     logit[r,h,s] = sum_{d<128} q[r,h,d] * k[s,d]        (FP4 E2M1, UE8M0/32)
 *     score[r,s]   = sum_{h<64} w[r,h] * max(logit[r,h,s], 0)    (fp32)
 *     raw[r]       = the topk positions s in [start, end) ranked by score
 *                    descending, then position ascending; NaN ranks below
 *                    every number and +0 above -0 (aiter#5282 Changes).  When
 *                    end - start <= topk the row returns start..end-1 in
 *                    order, padded with -1 (short-row contract, aiter#5282
 *                    Changes).  The dense [rows, context] score matrix is
 *                    never materialised (aiter#5309 Summary).
 *     phys[r]      = page_table[req][raw / 64] * 64 + raw % 64; -1 stays -1
 *                    (aiter#5282 Changes: raw C4 positions mapped through the
 *                    page table; sglang#38101 Changes: physical slots and
 *                    optional raw indices written in place).
 *
 * Conventions for every entry point:
 *  - Tensors are passed as idx_tensor_t descriptors of DEVICE memory that the
 *    caller owns (idx_topk_fp4_prefill_host alone takes host memory); the
 *    library keeps no pointer after it returns.  All tensors
 *    of a call must live on one device; the call makes that device current for
 *    its duration and restores the caller's current device before returning
 *    (aiter#5309 Implementation: caller device/stream ownership).
 *  - Work is enqueued on the caller's `stream` only (never the legacy default
 *    stream); the call returns after that stream has reached the end of the
 *    call's work, because the status is read back to the host.  Scratch is
 *    allocated stream-ordered on that stream from a library-owned pool and is
 *    bounded by rows, topk and the SM count -- never by the context length
 *    (aiter#5282 Changes, last paragraph).
 *  - Every tensor must be C-contiguous with a 16-byte-aligned base address.
 *  - Offsets are computed in 64 bits (aiter#5309 Implementation).
 *  - Fail closed (aiter#5309 Implementation): any error returns a nonzero
 *    code, and, when the output descriptors themselves are valid, the outputs
 *    are filled with -1 -- except while the stream is being captured into a
 *    CUDA graph, where nothing is enqueued and IDX_ERR_UNSUPPORTED is returned
 *    (aiter#5282 Scope: graph capture is rejected explicitly).
 */
#ifndef IDXTOPK_H_
#define IDXTOPK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* idx_stream_t;

typedef enum {
  IDX_OK = 0,
  IDX_ERR_INVALID_ARGUMENT = 1, /* null/misaligned/non-contiguous tensor, wrong dtype/rank/shape,
                                   tensors on different devices */
  IDX_ERR_UNSUPPORTED = 2,      /* topk not in {512, 1024}; H != 64, D != 128, page != 64;
                                   stream capture active; device is not sm_103 */
  IDX_ERR_INVALID_METADATA = 3, /* row_req out of [0, num_req), start < 0, end < start,
                                   end > max_pages * 64 */
  IDX_ERR_INVALID_PAGE = 4,     /* a page-table entry covering some row's window is outside
                                   [0, num_pages) */
  IDX_ERR_OVERFLOW = 5,         /* num_pages * 64 or max_pages * 64 exceeds INT32_MAX, or a
                                   size product overflows 64 bits */
  IDX_ERR_CUDA = 6,             /* a CUDA runtime/driver call failed */
  IDX_ERR_INTERNAL = 7,         /* selector failure: a scored row produced fewer than topk
                                   candidates, or a plan bound was exceeded */
  IDX_ERR_TIMEOUT = 8,          /* a bounded device-side wait expired (the kernel returned
                                   instead of hanging) */
  IDX_ERR_SCRATCH_LIMIT = 9,    /* idx_topk_fp4_prefill_noalloc only: the call needs more
                                   scratch than IDX_NOALLOC_SCRATCH_BYTES */
  IDX_ERR_INVALID_VALUE = 10    /* an input value outside the accepted domain (see
                                   IDX_MAX_SCALE_BYTE and IDX_MAX_ABS_WEIGHT): a scale byte
                                   above 167 in the query block of a scored row or in a K page
                                   that a window covers, or a weight of a scored row that is not
                                   finite or exceeds 2^24 in magnitude */
} idx_status_t;

/*
 * Accepted value domain (aiter#5309 Implementation: the operator fails closed
 * rather than produce nonfinite scores).  Every UE8M0 scale byte the scorer
 * reads -- the query block of each row it scores, and every K page under a
 * scored window -- must be at most IDX_MAX_SCALE_BYTE (scale exponent at most
 * +40; the NaN byte 255 is above it), and every weight of a scored row must be
 * finite with magnitude at most IDX_MAX_ABS_WEIGHT.  A per-head logit is then
 * below 2^93 in magnitude (at most 4 blocks x 32 products of E2M1 magnitudes
 * <= 6, i.e. < 2^13, times 2^(40+40)) and a score below 64 * 2^24 * 2^93 =
 * 2^123, so every score is finite.  A call that reads a value outside the
 * domain returns IDX_ERR_INVALID_VALUE with -1 outputs.  Bytes the scorer never
 * reads (pages outside every window, query blocks and weights of rows of
 * length <= topk) are not checked.
 */
#define IDX_MAX_SCALE_BYTE 167
#define IDX_MAX_ABS_WEIGHT 16777216.0f

typedef enum { IDX_U8 = 1, IDX_I32 = 2, IDX_F32 = 3 } idx_dtype_t;

/* Descriptor of one device tensor.  shape/stride are in elements; only the
 * first ndim entries are read. */
typedef struct {
  void* data;
  int32_t dtype; /* idx_dtype_t */
  int32_t ndim;
  int64_t shape[4];
  int64_t stride[4];
} idx_tensor_t;

/*
 * Fused FP4 paged-MQA scoring + exact TopK + page mapping (the hot path).
 *
 *   q_fp4        u8  [R, 64, 64]   FP4 E2M1 codes of the 64x128 query block of each row,
 *                                  two per byte, even element of D in the low nibble
 *   q_scale      u8  [R, 64, 4]    UE8M0 scale per 32 elements of D (2^(byte-127))
 *   k_cache_fp4  u8  [NP, 64, 64]  C4 K cache, page size 64, same encoding
 *   k_scale      u8  [NP, 64, 4]   UE8M0 scales of the K cache
 *   weights      f32 [R, 64]       per-head weights
 *   page_table   i32 [NR, MP]      physical page of logical page p of request i
 *   row_req      i32 [R]           request of each row
 *   row_start    i32 [R]           window start (logical C4 position, inclusive)
 *   row_end      i32 [R]           window end (exclusive)
 *   topk         512 or 1024
 *   out_phys_slot i32 [R, topk]    physical C4 slot (page * 64 + offset) or -1
 *   out_raw_idx   i32 [R, topk]    logical C4 position or -1; may be NULL
 *
 * Rows whose window is longer than topk are ordered by (score desc, position asc).
 * Scale bytes and weights must lie in the accepted domain above (else
 * IDX_ERR_INVALID_VALUE).  The operation is the one
 * defined at the top of this file (aiter#5309 Summary and Implementation;
 * aiter#5282 Changes and Scope).
 */
int idx_topk_fp4_prefill(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                         const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                         const idx_tensor_t* weights, const idx_tensor_t* page_table,
                         const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                         const idx_tensor_t* row_end, int32_t topk,
                         const idx_tensor_t* out_phys_slot, const idx_tensor_t* out_raw_idx,
                         idx_stream_t stream);

/*
 * idx_topk_fp4_prefill for a page-interleaved K cache (a consumer layout named
 * as follow-up work in "[FlyDSL][DSv4] Prototype FP4 MQA streaming TopK",
 * ROCm/aiter#5282, Scope): each physical page holds its codes and then its
 * scales, so one page is one contiguous 4352-byte record.
 *   k_pages u8 [NP, 4352]   bytes [0, 4096): 64 slots x 64 B of E2M1 codes
 *                           (as k_cache_fp4[page]); bytes [4096, 4352): 64
 *                           slots x 4 UE8M0 scales (as k_scale[page]).
 * Every other argument, the results and the error behaviour are those of
 * idx_topk_fp4_prefill; the outputs are identical for the same data.
 */
int idx_topk_fp4_prefill_paged(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                               const idx_tensor_t* k_pages, const idx_tensor_t* weights,
                               const idx_tensor_t* page_table, const idx_tensor_t* row_req,
                               const idx_tensor_t* row_start, const idx_tensor_t* row_end,
                               int32_t topk, const idx_tensor_t* out_phys_slot,
                               const idx_tensor_t* out_raw_idx, idx_stream_t stream);

/*
 * idx_topk_fp4_prefill with the K cache's scales pre-arranged in the order in
 * which the block-scaled MMA's scale copy reads them (the pre-shuffled scale
 * input named as follow-up work in "[FlyDSL][DSv4] Prototype FP4 MQA streaming
 * TopK", ROCm/aiter#5282, Scope; here the layout of sm_103a's 32x128b scale
 * copy into tensor memory instead of the AMD matrix-core layout):
 *   k_scale_mma u8 [NP, 256]  byte 8*j + 4*h + b of page p = scale b (D
 *                             elements 32b .. 32b+31) of slot 32*h + j of page
 *                             p, for j < 32, h < 2, b < 4; i.e. the page's
 *                             slot words reordered j, 32+j, j+1, 33+j, ...
 * A cache writer that stores its scales this way spares the scorer the
 * rearrangement; each producer lane then reads one 8-byte word per page.
 * Every other argument, the value domain, the results and the errors are those
 * of idx_topk_fp4_prefill; the outputs are identical for the same data.
 */
int idx_topk_fp4_prefill_mma_scales(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                                    const idx_tensor_t* k_cache_fp4,
                                    const idx_tensor_t* k_scale_mma, const idx_tensor_t* weights,
                                    const idx_tensor_t* page_table, const idx_tensor_t* row_req,
                                    const idx_tensor_t* row_start, const idx_tensor_t* row_end,
                                    int32_t topk, const idx_tensor_t* out_phys_slot,
                                    const idx_tensor_t* out_raw_idx, idx_stream_t stream);

/*
 * idx_topk_fp4_prefill on tensors in host memory (no counterpart on the
 * pages: it serves callers whose query block, K cache and metadata sit
 * in host memory, and it is the end-to-end form of the operation, host copies
 * included).
 *   device  the GPU to run on (0 .. count-1); stream must belong to it or be NULL.
 * Every descriptor points to host memory: pinned memory (cudaHostAlloc or
 * cudaHostRegister) makes the copies asynchronous DMA; pageable memory also
 * works, at host-copy speed.  Shapes, dtypes and results are those of
 * idx_topk_fp4_prefill; host buffers need no particular alignment.  The call
 * takes one block of device memory from the library's stream-ordered pool,
 * copies each input into it (one cudaMemcpyAsync per tensor on `stream`), runs
 * the fused path there, copies the outputs back, returns the block to the pool
 * and returns once `stream` has completed.  It keeps no pointer.  Error codes
 * are those of idx_topk_fp4_prefill; a descriptor that points to device memory
 * or a device index out of range is IDX_ERR_INVALID_ARGUMENT.  On any error
 * after the output descriptors are validated, the host outputs are filled
 * with -1.
 */
int idx_topk_fp4_prefill_host(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                              const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                              const idx_tensor_t* weights, const idx_tensor_t* page_table,
                              const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                              const idx_tensor_t* row_end, int32_t topk,
                              const idx_tensor_t* out_phys_slot, const idx_tensor_t* out_raw_idx,
                              int32_t device, idx_stream_t stream);

/*
 * Stream-ordered variant of idx_topk_fp4_prefill for decode loops and CUDA
 * graphs: the same operation and outputs, with no allocation and no host
 * synchronisation, so a call may be captured into a graph and replayed.  The
 * pages keep decode and graph capture on their previous path and name it as
 * follow-up work ("[FlyDSL][DSv4] Prototype FP4 MQA streaming TopK",
 * ROCm/aiter#5282, Scope); this entry point is that follow-up.
 *   workspace        device memory on the tensors' device, 256-byte aligned,
 *                    at least idx_topk_fp4_scratch_bytes(rows, topk) bytes;
 *                    caller-owned, must not be used by another call that runs
 *                    at the same time.
 *   status           one device uint32 (4-byte aligned) on the same device;
 *                    after the call's work completes on `stream` it holds
 *                    IDX_OK or the device-detected error (invalid metadata,
 *                    invalid page, internal, timeout), and on such an error
 *                    every output entry is -1.
 * Returns IDX_OK when the work was enqueued on `stream` (whether or not the
 * stream is being captured).  Argument errors found on the host (descriptors,
 * shapes, topk, device, workspace size or alignment) return their code with
 * nothing enqueued, the outputs and *status untouched; IDX_ERR_CUDA means a
 * launch failed and *status is not written.  While `stream` is being
 * captured, pointer and stream-device queries are not allowed, so the call
 * uses the current device and does not check that the stream and the tensors
 * belong to it; make one call outside the capture first (it checks them and
 * performs the library's per-device setup).  Graph
 * replays reuse the pointers and sizes seen at capture (a new shape needs a
 * new capture).
 */
int idx_topk_fp4_prefill_async(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                               const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                               const idx_tensor_t* weights, const idx_tensor_t* page_table,
                               const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                               const idx_tensor_t* row_end, int32_t topk,
                               const idx_tensor_t* out_phys_slot, const idx_tensor_t* out_raw_idx,
                               void* workspace, uint64_t workspace_bytes, uint32_t* status,
                               idx_stream_t stream);

/*
 * Allocation-free variant of idx_topk_fp4_prefill (no counterpart on the
 * pages; it exists for callers that must not allocate device memory
 * during a call: a serving process that has handed all free HBM to its own
 * caches and allocator, so a new reservation would fail or evict; or a caller
 * that cannot afford the device synchronisation and driver work that growing
 * a memory pool may cost inside a latency-bound loop).
 *
 * Arguments, layouts, results, ownership and error behaviour are those of
 * idx_topk_fp4_prefill, with one difference: the scratch comes from a fixed
 * buffer of IDX_NOALLOC_SCRATCH_BYTES per device that is part of the
 * library's device image, so the call makes no cudaMalloc/cudaFree, pool or
 * event allocation.  Its size need is idx_topk_fp4_scratch_bytes(rows, topk):
 * (rows + 3 * SMs) * topk * 8 bytes plus a few KB; a call that needs more
 * returns IDX_ERR_SCRATCH_LIMIT (outputs filled with -1) without running.
 * At 152 SMs that admits up to about 5,640 rows at topk 1024 and 11,630 at 512.
 *
 *  - The buffer is reserved on a device when the library's device code is
 *    loaded there: under CUDA's default lazy module loading that happens at
 *    the first call of this function on the device (which also looks up the
 *    buffer's address, with the device made current); under eager loading
 *    (CUDA_MODULE_LOADING=EAGER) it happens when the process creates its
 *    context on the device, whether or not this function is ever called.
 *    Make the first call before any stream capture begins, and before the
 *    caller hands the device's remaining memory to its own allocator (the
 *    reservation can fail with IDX_ERR_CUDA when no memory is left).
 *  - A device index of 64 or more is rejected with IDX_ERR_INVALID_ARGUMENT
 *    before anything is enqueued.
 *  - All calls on one device share the one buffer.  The call returns only
 *    after its work on `stream` has completed, and a per-device lock held for
 *    the whole call makes concurrent calls from several host threads run one
 *    after another, so calls never overlap on the buffer (other streams of
 *    the same process included; each process has its own buffer).
 */
#define IDX_NOALLOC_SCRATCH_BYTES (48u * 1024u * 1024u)
int idx_topk_fp4_prefill_noalloc(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                                 const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                                 const idx_tensor_t* weights, const idx_tensor_t* page_table,
                                 const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                                 const idx_tensor_t* row_end, int32_t topk,
                                 const idx_tensor_t* out_phys_slot,
                                 const idx_tensor_t* out_raw_idx, idx_stream_t stream);

/* The supported topk values, {512, 1024} (aiter#5309 Implementation: explicit
 * supported-K contract).  *ks points to static storage.  Always IDX_OK unless
 * an argument is NULL (IDX_ERR_INVALID_ARGUMENT). */
int idx_topk_supported_k(const int32_t** ks, int32_t* n);

/* Static, human-readable name of a status code (the fail-closed status
 * contract of aiter#5309 Implementation). */
const char* idx_topk_status_string(int code);

/* Scratch bytes that idx_topk_fp4_prefill allocates for `rows` rows and
 * `topk`, on `device` (its SM count bounds the work units).  Independent of
 * the context length (aiter#5282 Changes, last paragraph; sglang#38101 Memory
 * geometry).  Returns IDX_ERR_UNSUPPORTED for an unsupported topk,
 * IDX_ERR_CUDA if the device cannot be queried. */
int idx_topk_fp4_scratch_bytes(int32_t rows, int32_t topk, int32_t device, uint64_t* bytes);

/* Diagnostic of the device-side failure detection (no counterpart on the
 * pages).  One CTA on `device` waits, through the same bounded mbarrier wait
 * every kernel of the library uses, on a phase that its own thread completes
 * (never_completes == 0) or that nothing completes (never_completes != 0).
 * Returns the status the kernel recorded: IDX_OK, or IDX_ERR_TIMEOUT once the
 * wait has given up after its 2 s limit -- the kernel then returns with
 * nothing in flight and the CUDA context stays usable.  Synchronises
 * `stream`; IDX_ERR_UNSUPPORTED while the stream is being captured;
 * IDX_ERR_INVALID_ARGUMENT for a bad device index or a stream of another
 * device. */
int idx_debug_bounded_wait(int32_t device, int32_t never_completes, idx_stream_t stream);

/* Peak bytes ever reserved by the library's scratch pool on `device` in this
 * process (the pool's reserved-memory high-water mark).  Measurement support
 * with no counterpart on the pages; it evidences the context-independent
 * scratch bound of aiter#5282 Changes. */
int idx_topk_scratch_high_water(int32_t device, uint64_t* bytes);

/* Measurement support (no counterpart on the pages): when enabled, each call
 * of the calling thread records CUDA events on its stream around the kernel
 * phases; idx_topk_last_timings then returns, in milliseconds, {planning,
 * scoring kernel, finishing kernel, whole kernel sequence} of
 * that thread's last completed call.  Process-wide switch; default off. */
int idx_topk_set_timing(int32_t enable);
int idx_topk_last_timings(float* ms4);

/*
 * Context-parallel pieces ("[AMD][DSv4] Add experimental AITER FP4 streaming
 * TopK", sglang#38101, Changes: context-parallel paths; "[FlyDSL][DSv4]
 * Prototype FP4 MQA streaming TopK", ROCm/aiter#5282, Changes: merge split
 * candidates exactly).  A context partition [c_0, c_1), [c_1, c_2), ... of the
 * logical C4 positions is scored one shard at a time (each call may run where
 * that shard's K pages live); the shards' lists, gathered into one
 * [S, R, topk] pair of tensors by the caller, are merged exactly.  The merged
 * outputs equal those of idx_topk_fp4_prefill on the same data, bit for bit.
 *
 * idx_topk_fp4_prefill_shard: every row whose whole window [start, end) is
 * longer than topk is scored against the part of it inside [ctx_begin,
 * ctx_end) only -- however short that part -- and emits that part's exact
 * TopK, ordered by (score desc, position asc):
 *   out_score    f32 [R, topk]  the scores (as the fused path computes them),
 *                               NaN after the part's last position
 *   out_raw_idx  i32 [R, topk]  logical C4 positions, -1 after the last one
 * Rows whose whole window is at most topk long emit only -1 / NaN (the merge
 * gives them the closed form).  Inputs, value domain and errors as
 * idx_topk_fp4_prefill; ctx_begin < 0 or ctx_end < ctx_begin is
 * IDX_ERR_INVALID_ARGUMENT.  Only the page entries and K pages under the
 * clipped windows are read and checked.  On error out_raw_idx is -1 and
 * out_score NaN.
 */
int idx_topk_fp4_prefill_shard(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                               const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                               const idx_tensor_t* weights, const idx_tensor_t* page_table,
                               const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                               const idx_tensor_t* row_end, int32_t ctx_begin, int32_t ctx_end,
                               int32_t topk, const idx_tensor_t* out_score,
                               const idx_tensor_t* out_raw_idx, idx_stream_t stream);

/*
 * idx_topk_merge_shards: the exact TopK of each row over the union of its S
 * shard lists (aiter#5282 Changes: exact merge of split candidates), then the
 * short-row contract and the page mapping of idx_topk_fp4_prefill.
 *   shard_score  f32 [S, R, topk]  shard s's out_score (S >= 1)
 *   shard_raw    i32 [S, R, topk]  shard s's out_raw_idx (-1 = empty entry)
 *   page_table, row_req, row_start, row_end  as for idx_topk_fp4_prefill
 *   out_phys_slot, out_raw_idx (nullable)   as for idx_topk_fp4_prefill
 * The shards must cover every window and be disjoint.  A listed position
 * outside its row's window, a position listed twice among the emitted TopK, or
 * a row whose lists hold fewer than topk positions although its window is
 * longer than topk returns IDX_ERR_INVALID_METADATA (as do bad row metadata);
 * a negative page-table entry read by the mapping returns IDX_ERR_INVALID_PAGE
 * (the K cache is not an argument, so entries are not compared with its page
 * count here: the shard calls checked every entry under their windows);
 * unsupported topk IDX_ERR_UNSUPPORTED; outputs -1 on every error.  Scratch:
 * one status word.
 */
int idx_topk_merge_shards(const idx_tensor_t* shard_score, const idx_tensor_t* shard_raw,
                          const idx_tensor_t* page_table, const idx_tensor_t* row_req,
                          const idx_tensor_t* row_start, const idx_tensor_t* row_end,
                          int32_t topk, const idx_tensor_t* out_phys_slot,
                          const idx_tensor_t* out_raw_idx, idx_stream_t stream);

/*
 * Context-tiled comparison path (an ablation of the fused design: "[FlyDSL]
 * [DSv4] Prototype FP4 MQA streaming TopK", ROCm/aiter#5282, Changes, names a
 * bounded context-tiled fallback).  The same operation and outputs as
 * idx_topk_fp4_prefill, computed by scoring `context_tile` logical positions
 * at a time into a materialised fp32 buffer [rows, context_tile] and folding
 * each chunk into every row's running TopK.  Scratch is bounded by rows *
 * (context_tile * 4 + topk * 8) bytes plus the plan, not by the context.
 *   context_tile  positions per chunk, a multiple of 128 and >= 1024.
 * Errors and ownership as idx_topk_fp4_prefill (a bad context_tile returns
 * IDX_ERR_INVALID_ARGUMENT).
 */
int idx_tiled_topk_fp4_prefill(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                               const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                               const idx_tensor_t* weights, const idx_tensor_t* page_table,
                               const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                               const idx_tensor_t* row_end, int32_t topk, int32_t context_tile,
                               const idx_tensor_t* out_phys_slot, const idx_tensor_t* out_raw_idx,
                               idx_stream_t stream);

/*
 * Debug / dense scorer: the same scoring kernel as the fused path, writing the
 * fp32 scores instead of selecting (no counterpart on the pages; it exposes
 * the scores and per-head logits that the parity tests compare).
 *   out_scores f32 [R, S]      score[r, s] written for every s in [start_r, end_r)
 *                              of every row with a non-empty window; other entries are
 *                              left untouched.  S >= max(row_end) is required and
 *                              checked on the device (IDX_ERR_INVALID_METADATA).
 *   out_logits f32 [R, 64, S2] optional (may be NULL): per-head logits
 *                              logit[r, h, s] for the same (r, s).
 * Other arguments as for idx_topk_fp4_prefill (no topk, no outputs).
 */
int idx_fp4_debug_scores(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                         const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                         const idx_tensor_t* weights, const idx_tensor_t* page_table,
                         const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                         const idx_tensor_t* row_end, const idx_tensor_t* out_scores,
                         const idx_tensor_t* out_logits, idx_stream_t stream);

/*
 * Exact TopK of a materialised fp32 score matrix under the same total order and
 * short-row contract (aiter#5282 Changes: the order key, NaN below every
 * number, +0 above -0, ties to the lower position; the selection half of the
 * dense comparison path, and the entry that pins that ordering on crafted
 * matrices).
 *   scores      f32 [R, S]   row r's candidates are scores[r, start_r .. end_r)
 *   row_start, row_end i32 [R]
 *   out_raw_idx i32 [R, topk]   positions (absolute within the row) or -1
 * Requires end_r <= S (checked on the device, IDX_ERR_INVALID_METADATA).
 */
int idx_topk_select_scores(const idx_tensor_t* scores, const idx_tensor_t* row_start,
                           const idx_tensor_t* row_end, int32_t topk,
                           const idx_tensor_t* out_raw_idx, idx_stream_t stream);

/*
 * Dense comparison path: materialises fp32 scores [R, score_stride] (rows with
 * window longer than topk), then runs the separate TopK and the page mapping
 * (aiter#5309 Validation: the dense-scores-then-TopK baseline the pages time
 * the fused operator against).
 * Same arguments and outputs as idx_topk_fp4_prefill plus:
 *   score_workspace f32 [R, S_ws], S_ws >= max(row_end), caller-owned; may be
 *                   NULL, in which case R * MP * 64 * 4 bytes are allocated
 *                   stream-ordered for the call.
 */
int idx_dense_topk_fp4_prefill(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                               const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                               const idx_tensor_t* weights, const idx_tensor_t* page_table,
                               const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                               const idx_tensor_t* row_end, int32_t topk,
                               const idx_tensor_t* out_phys_slot,
                               const idx_tensor_t* out_raw_idx,
                               const idx_tensor_t* score_workspace, idx_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* IDXTOPK_H_ */
