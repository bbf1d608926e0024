// Internal definitions shared by the host library and the sm_103a kernels.
//
// Work decomposition of the fused scorer: rows are grouped into row blocks of
// up to kRowsPerBlock consecutive rows of one request, so that each staged K
// tile is reused by every row of the block; the union window of a block is cut
// into work units (contiguous runs of K tiles).  Each unit emits, per row, at
// most topk candidates (64-bit order keys) into bounded scratch; the merge
// kernel unions a row's candidates and selects the exact TopK.  This is the
// split/merge structure of "[FlyDSL][DSv4] Prototype FP4 MQA streaming TopK"
// (ROCm/aiter#5282, Changes: per-CTA candidate emission, exact merge of split
// candidates), laid out for 152 SMs with one persistent CTA per SM.
#pragma once

#include <cstddef>
#include <cstdint>

namespace idxk {

constexpr int kHeads = 64;          // H
constexpr int kDim = 128;           // D (FP4 elements)
constexpr int kDimBytes = 64;       // D / 2
constexpr int kNumSF = 4;           // D / 32 UE8M0 scales per row
constexpr int kPage = 64;           // slots per KV page
constexpr int kTile = 128;          // slots per K tile = MMA M
constexpr int kRowsPerBlock = 3;    // query rows sharing one K tile (one per epilogue warpgroup)
constexpr int kRowsPerChunk = 1;    // query rows per TMA box of the query block (64 head rows)
constexpr int kChunks = kRowsPerBlock / kRowsPerChunk;
constexpr int kAccStages = 2;       // TMEM accumulator buffers (double buffer, N = 3 x 64 each)
// Work-unit sizing: the planner cuts a block's tiles into units of about
// max(total tiles / SMs, kMinUnitTiles) tiles.  About one unit per persistent
// CTA keeps the per-unit costs (query-block load, threshold warm-up, final
// selection and candidate write) and the merge of a row's units small; the
// longest-first, alternating deal of the units keeps the CTAs balanced.
constexpr int kMinUnitTiles = 64;   // shortest work unit (tiles), except whole short blocks
constexpr int kUnitsPerCta = 1;     // target work units per persistent CTA

// Status codes (mirror idx_status_t of the public header).
enum : uint32_t {
  kOk = 0,
  kErrInvalidArgument = 1,
  kErrUnsupported = 2,
  kErrInvalidMetadata = 3,
  kErrInvalidPage = 4,
  kErrOverflow = 5,
  kErrCuda = 6,
  kErrInternal = 7,
  kErrTimeout = 8,
  kErrInvalidValue = 10,
};

// Accepted value domain (the header's IDX_MAX_SCALE_BYTE / IDX_MAX_ABS_WEIGHT):
// UE8M0 bytes <= 167 and finite weights of magnitude <= 2^24 keep every logit
// below 2^93 and every score finite.
constexpr uint32_t kMaxScaleByte = 167;
constexpr uint32_t kMaxAbsWeightBits = 0x4B800000u;  // 2^24 as fp32

struct BlockInfo {
  int32_t row0;       // first row
  int32_t nrows;      // rows in the block (1..kRowsPerBlock)
  int32_t req;        // request of every row of the block
  int32_t n_units;    // work units of this block (0 when no row is scored)
  int32_t tile0;      // first K tile (absolute: slots [tile0*128, ...))
  int32_t ntiles;     // tiles covering the union window of the scored rows
  int32_t unit_first; // index of the block's first unit in the unit table
  int32_t pad;
  int64_t slot0;      // first candidate row-slot: unit k, row j -> slot0 + k*nrows + j
};

struct UnitInfo {
  int32_t block;
  int32_t t_begin;    // absolute tile index range [t_begin, t_end)
  int32_t t_end;
  int32_t k;          // index of the unit within its block
};

struct PlanHeader {
  uint32_t status;      // first error wins (atomicCAS from kOk)
  int32_t n_blocks;
  int32_t n_units;
  int32_t unit_tiles;   // chunk length the planner chose
  int64_t n_row_slots;  // candidate row-slots in use
  uint32_t err_site;    // where the first error was raised (diagnostics)
  uint32_t claim;       // next schedule position of the dynamically scheduled scorer
  uint32_t fin_done;    // CTAs of the finishing kernel that are done (status publishing)
  uint32_t pad[7];
};

// Byte offsets of the scratch regions of one call.
struct ScratchLayout {
  size_t header, row_block, blocks, units, sched, cand_cnt, cand_keys, total;
  int64_t max_blocks, max_units, max_row_slots;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bounds: blocks <= rows; units <= blocks + kUnitsPerCta * G (ceil per block);
// candidate row-slots <= rows + kRowsPerBlock * kUnitsPerCta * G.  None depends
// on the context length.
inline ScratchLayout scratch_layout(int64_t rows, int64_t topk, int64_t grid, bool with_cands) {
  ScratchLayout L{};
  L.max_blocks = rows > 0 ? rows : 1;
  L.max_units = L.max_blocks + kUnitsPerCta * grid;
  L.max_row_slots = rows + (int64_t)kRowsPerBlock * kUnitsPerCta * grid;
  size_t off = 0;
  L.header = off;    off = align_up(off + sizeof(PlanHeader), 256);
  L.row_block = off; off = align_up(off + sizeof(int32_t) * (size_t)L.max_blocks, 256);
  L.blocks = off;    off = align_up(off + sizeof(BlockInfo) * (size_t)L.max_blocks, 256);
  L.units = off;     off = align_up(off + sizeof(UnitInfo) * (size_t)L.max_units, 256);
  L.sched = off;     off = align_up(off + sizeof(int32_t) * (size_t)L.max_units, 256);
  if (with_cands) {
    L.cand_cnt = off;  off = align_up(off + sizeof(uint32_t) * (size_t)L.max_row_slots, 256);
    L.cand_keys = off; off = align_up(off + sizeof(uint64_t) * (size_t)L.max_row_slots * (size_t)topk, 256);
  } else {
    L.cand_cnt = L.cand_keys = off;
  }
  L.total = off;
  return L;
}

// Parameters of the planning kernels.
struct PlanParams {
  const int32_t* row_req;
  const int32_t* row_start;
  const int32_t* row_end;
  const int32_t* page_table;
  int32_t rows, num_req, max_pages, num_pages;
  int32_t score_thr;     // rows with end - start > score_thr are scored
  int32_t grid;          // persistent CTAs of the scorer
  int32_t check_end_le;  // >= 0: every end must be <= this (score matrix width); -1: none
  int32_t clear_hdr;     // 1: the planner zeroes the header first (no kernel of the call
                         // touches it before the planner); 0: the caller cleared it
  int64_t max_units, max_row_slots;
  PlanHeader* hdr;
  int32_t* row_block;    // row -> block
  BlockInfo* blocks;
  UnitInfo* units;
  int32_t* sched;
};

enum ScoreMode : int32_t { kModeSelect = 0, kModeDense = 1 };

// Parameters of the scoring kernel (tensor maps are separate launch arguments).
struct ScoreParams {
  const uint8_t* q_scale;
  const uint8_t* k_scale;    // page p's 64 scale words start at word p * k_scale_stride
  int64_t k_scale_stride;    // 32-bit words between consecutive pages' scales
  int32_t k_scale_mma;       // 0: word s = slot s's 4 scales; 1: the MMA's scale-copy
                             // order, word 2j + h = slot 32h + j's 4 scales
  int32_t pad0;
  const float* weights;
  const int32_t* page_table;
  const int32_t* row_start;
  const int32_t* row_end;
  int32_t rows, max_pages, num_pages, topk;
  int32_t mode, score_thr;
  int32_t dyn;               // 1: the CTAs claim work units from hdr->claim (several requests)
  int32_t pad1;
  PlanHeader* hdr;
  const BlockInfo* blocks;
  const UnitInfo* units;
  const int32_t* sched;
  uint32_t* cand_cnt;
  uint64_t* cand_keys;
  float* dense_out;        // [rows, dense_stride]; column = slot - dense_col0
  int64_t dense_stride;
  int64_t dense_col0;
  float* logits_out;       // [rows, 64, logits_stride] or null
  int64_t logits_stride;
};

// Parameters of the context-tiled comparison path's per-chunk merge.
struct TileMergeParams {
  const int32_t* row_req;
  const int32_t* row_start;   // the full windows
  const int32_t* row_end;
  const int32_t* page_table;
  int32_t rows, max_pages, topk, c0, c1, first, last;
  int32_t num_pages;          // pages of the K cache: a mapped entry must lie in [0, num_pages)
  int64_t stride;             // floats per row of the chunk buffer
  const float* chunk;         // [rows, stride], column = slot - c0
  uint64_t* run_keys;         // [rows, topk] running candidates
  uint32_t* run_cnt;          // [rows]
  uint64_t* run_tau;          // [rows] running threshold
  PlanHeader* hdr;
  int32_t* out_phys;
  int32_t* out_raw;           // nullable
};

// Parameters of the row finishing kernels (merge of unit candidates, or TopK of
// a dense score matrix), followed by sort and page mapping.
struct FinishParams {
  const int32_t* row_req;
  const int32_t* row_start;
  const int32_t* row_end;
  const int32_t* page_table;  // null: no physical mapping
  int32_t rows, max_pages, topk;
  int32_t num_pages;          // a mapped page-table entry must lie in [0, num_pages)
  PlanHeader* hdr;            // status word (and plan for the merge)
  const int32_t* row_block;
  const BlockInfo* blocks;
  const uint32_t* cand_cnt;
  const uint64_t* cand_keys;
  const float* scores;        // dense source [rows, score_stride] (null for the merge)
  int64_t score_stride;
  int32_t* out_phys;          // [rows, topk] or null
  int32_t* out_raw;           // [rows, topk] or null
  // context shard (out_score non-null): every nonempty (clipped) window was
  // scored whatever its length; each row emits its sorted TopK positions with
  // their scores, padded with -1 / NaN, and no physical slots
  float* out_score;           // [rows, topk] or null
  // merge of context-shard lists: n_shards lists of [rows, topk] (score, position)
  int32_t n_shards;
  int32_t pad2;
  const float* shard_score;   // [n_shards, rows, topk]
  const int32_t* shard_raw;   // [n_shards, rows, topk], -1 = empty entry
  // stream-ordered call (non-null): the finishing kernel's last CTA copies the
  // call's status here and, on an error, fills out_phys / out_raw with -1
  uint32_t* status_out;
};

}  // namespace idxk
