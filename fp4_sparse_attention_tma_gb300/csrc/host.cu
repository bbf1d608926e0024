// C ABI of the library (declared in include/idxtopk.h): argument validation,
// device guard, graph-capture rejection, stream-ordered bounded scratch, TMA
// descriptors, the kernel sequence, status read-back and fail-closed output
// fill.  Follows the operator contract of "[FlyDSL] Add FP4 LiteTopK prefill
// operator" (ROCm/aiter#5309, Implementation) and "[FlyDSL][DSv4] Prototype FP4
// MQA streaming TopK" (ROCm/aiter#5282, Changes and Scope).
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "idx_internal.h"
#include "idx_launch.h"
#include "idxtopk.h"

using namespace idxk;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool init = false;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  cudaMemPool_t pool = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Optional per-kernel timing of the last call (CUDA events on the caller's
// stream around each launch): plan, scorer, finish, whole call.
std::atomic<bool> g_timing{false};
thread_local float g_last_ms[4] = {0.f, 0.f, 0.f, 0.f};

struct CallTimer {
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
  bool on = false;
  CallTimer() {
    if (!g_timing) return;
    on = true;
    for (auto& e : ev)
      if (cudaEventCreate(&e) != cudaSuccess) on = false;
  }
  ~CallTimer() {
    for (auto& e : ev)
      if (e) cudaEventDestroy(e);
  }
  void mark(int i, cudaStream_t s) {
    if (on) cudaEventRecord(ev[i], s);
  }
  // call after the stream has been synchronised
  void collect(cudaEvent_t end) {
    if (!on) return;
    float t[4] = {0.f, 0.f, 0.f, 0.f};
    cudaEvent_t pts[5] = {ev[0], ev[1], ev[2], ev[3], end};
    for (int i = 0; i < 3; ++i) cudaEventElapsedTime(&t[i], pts[i], pts[i + 1]);
    cudaEventElapsedTime(&t[3], pts[0], pts[3]);
    for (int i = 0; i < 4; ++i) g_last_ms[i] = t[i];
    cudaGetLastError();
  }
};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int device_state(int dev, DeviceState** out) {
  if (dev < 0 || dev >= kMaxDevices) return IDX_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return IDX_ERR_CUDA;
    }
    cudaMemPoolProps props;
    memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) {
      cudaGetLastError();
      return IDX_ERR_CUDA;
    }
    uint64_t keep = UINT64_MAX;  // keep freed scratch reserved for the next call
    cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    d.init = true;
  }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
      cudaGetLastError();
      return IDX_ERR_CUDA;
    }
    g_encode = (EncodeTiledFn)fn;
  }
  *out = &d;
  return IDX_OK;
}

// ---------------------------------------------------------- validation ----

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > INT64_MAX / a) return false;
  *out = a * b;
  return true;
}

// Validates one descriptor: dtype, rank, non-negative shape, C-contiguous
// strides, 16-byte aligned base (unless empty or need_align is false: host
// tensors that are only copied).  Returns IDX_OK or an error.
int check_tensor(const idx_tensor_t* t, int dtype, int ndim, bool need_align = true) {
  if (!t) return IDX_ERR_INVALID_ARGUMENT;
  if (t->dtype != dtype || t->ndim != ndim) return IDX_ERR_INVALID_ARGUMENT;
  int64_t numel = 1;
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0) return IDX_ERR_INVALID_ARGUMENT;
    if (!mul_ok(numel, t->shape[i], &numel)) return IDX_ERR_OVERFLOW;
  }
  int64_t expect = 1;
  for (int i = ndim - 1; i >= 0; --i) {
    if (t->shape[i] > 1 && t->stride[i] != expect) return IDX_ERR_INVALID_ARGUMENT;
    if (!mul_ok(expect, t->shape[i] > 0 ? t->shape[i] : 1, &expect)) return IDX_ERR_OVERFLOW;
  }
  int64_t bytes;
  if (!mul_ok(numel, dtype == IDX_U8 ? 1 : 4, &bytes)) return IDX_ERR_OVERFLOW;
  if (numel > 0) {
    if (!t->data) return IDX_ERR_INVALID_ARGUMENT;
    if (need_align && ((uintptr_t)t->data & 15u) != 0) return IDX_ERR_INVALID_ARGUMENT;
  }
  return IDX_OK;
}

int64_t numel_of(const idx_tensor_t* t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

// Device that owns `ptr` (device or managed memory), or -1.
int device_of(const void* ptr) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return -1;
  return a.device;
}

class DeviceGuard {
 public:
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev_) != cudaSuccess) {
      cudaGetLastError();
      prev_ = -1;
    }
    if (prev_ != dev) ok_ = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev_ >= 0) cudaSetDevice(prev_);
  }
  bool ok() const { return ok_; }

 private:
  int prev_ = -1;
  bool ok_ = true;
};

struct Outputs {
  const idx_tensor_t* t[2] = {nullptr, nullptr};
};

// Fills valid outputs with -1 on `stream` and waits for it.
void fill_minus_one(const Outputs& o, cudaStream_t stream) {
  for (const idx_tensor_t* t : o.t) {
    if (!t) continue;
    const int64_t n = numel_of(t);
    if (n > 0) cudaMemsetAsync(t->data, 0xFF, (size_t)n * 4, stream);
  }
  cudaStreamSynchronize(stream);
  cudaGetLastError();
}

// Common checks of the scoring inputs; on success fills the sizes.
struct Sizes {
  int64_t rows = 0, num_pages = 0, num_req = 0, max_pages = 0;
};

int check_inputs(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                 const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                 const idx_tensor_t* weights, const idx_tensor_t* page_table,
                 const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                 const idx_tensor_t* row_end, Sizes* sz, const idx_tensor_t* k_pages = nullptr,
                 bool k_scale_mma = false) {
  int st;
  if ((st = check_tensor(q_fp4, IDX_U8, 3))) return st;
  if ((st = check_tensor(q_scale, IDX_U8, 3))) return st;
  if (k_pages) {
    // page-interleaved K cache: [NP, 64 * 64 code bytes + 64 * 4 scale bytes]
    if ((st = check_tensor(k_pages, IDX_U8, 2))) return st;
    if (k_pages->shape[1] != kPage * (kDimBytes + kNumSF)) return IDX_ERR_UNSUPPORTED;
  } else {
    if ((st = check_tensor(k_cache_fp4, IDX_U8, 3))) return st;
    // K scales: [NP, 64 slots, 4], or [NP, 256] in the MMA's scale-copy order
    if ((st = check_tensor(k_scale, IDX_U8, k_scale_mma ? 2 : 3))) return st;
  }
  if ((st = check_tensor(weights, IDX_F32, 2))) return st;
  if ((st = check_tensor(page_table, IDX_I32, 2))) return st;
  if ((st = check_tensor(row_req, IDX_I32, 1))) return st;
  if ((st = check_tensor(row_start, IDX_I32, 1))) return st;
  if ((st = check_tensor(row_end, IDX_I32, 1))) return st;
  // H = 64 heads, D = 128 (64 bytes, 4 scales), page size 64 are the supported
  // specialisation (aiter#5282 Scope)
  if (q_fp4->shape[1] != kHeads || q_fp4->shape[2] != kDimBytes) return IDX_ERR_UNSUPPORTED;
  if (!k_pages && (k_cache_fp4->shape[1] != kPage || k_cache_fp4->shape[2] != kDimBytes))
    return IDX_ERR_UNSUPPORTED;
  const int64_t R = q_fp4->shape[0];
  if (q_scale->shape[0] != R || q_scale->shape[1] != kHeads || q_scale->shape[2] != kNumSF)
    return IDX_ERR_INVALID_ARGUMENT;
  if (!k_pages && k_scale_mma &&
      (k_scale->shape[0] != k_cache_fp4->shape[0] || k_scale->shape[1] != kPage * kNumSF))
    return IDX_ERR_INVALID_ARGUMENT;
  if (!k_pages && !k_scale_mma &&
      (k_scale->shape[0] != k_cache_fp4->shape[0] || k_scale->shape[1] != kPage ||
       k_scale->shape[2] != kNumSF))
    return IDX_ERR_INVALID_ARGUMENT;
  if (weights->shape[0] != R || weights->shape[1] != kHeads) return IDX_ERR_INVALID_ARGUMENT;
  if (row_req->shape[0] != R || row_start->shape[0] != R || row_end->shape[0] != R)
    return IDX_ERR_INVALID_ARGUMENT;
  sz->rows = R;
  sz->num_pages = k_pages ? k_pages->shape[0] : k_cache_fp4->shape[0];
  sz->num_req = page_table->shape[0];
  sz->max_pages = page_table->shape[1];
  // physical slots and logical positions are int32 (aiter#5309 Implementation:
  // 64-bit addressing inside, overflow rejected at the int32 outputs)
  if (R > INT32_MAX || sz->num_pages * (int64_t)kPage > INT32_MAX ||
      sz->max_pages * (int64_t)kPage > INT32_MAX || sz->num_req > INT32_MAX ||
      R * (int64_t)kHeads > INT32_MAX)
    return IDX_ERR_OVERFLOW;
  if (R > 0 && (sz->num_pages < 1 || sz->num_req < 1 || sz->max_pages < 1))
    return IDX_ERR_INVALID_ARGUMENT;
  return IDX_OK;
}

int check_output(const idx_tensor_t* out, int64_t rows, int32_t topk, bool need_align = true) {
  int st = check_tensor(out, IDX_I32, 2, need_align);
  if (st) return st;
  if (out->shape[0] != rows || out->shape[1] != topk) return IDX_ERR_INVALID_ARGUMENT;
  return IDX_OK;
}

bool topk_supported(int32_t k) { return k == 512 || k == 1024; }

// Every non-empty tensor must be device memory of one device; returns it.
int common_device(const idx_tensor_t* const* ts, int n, int* dev) {
  int d = -1;
  for (int i = 0; i < n; ++i) {
    const idx_tensor_t* t = ts[i];
    if (!t || numel_of(t) == 0) continue;
    const int td = device_of(t->data);
    if (td < 0) return IDX_ERR_INVALID_ARGUMENT;
    if (d >= 0 && td != d) return IDX_ERR_INVALID_ARGUMENT;
    d = td;
  }
  if (d < 0 && cudaGetDevice(&d) != cudaSuccess) {
    cudaGetLastError();
    return IDX_ERR_CUDA;
  }
  *dev = d;
  return IDX_OK;
}

int check_stream(cudaStream_t stream, int dev) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return IDX_ERR_CUDA;
  }
  if (cs != cudaStreamCaptureStatusNone) return IDX_ERR_UNSUPPORTED;
  if (stream != nullptr) {
    int sd = -1;
    if (cudaStreamGetDevice(stream, &sd) != cudaSuccess) {
      cudaGetLastError();
      return IDX_ERR_INVALID_ARGUMENT;
    }
    if (sd != dev) return IDX_ERR_INVALID_ARGUMENT;
  }
  return IDX_OK;
}

int encode_2d_u8(CUtensorMap* map, void* base, uint64_t rows, uint32_t box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)kDimBytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kDimBytes};
  cuuint32_t box[2] = {(cuuint32_t)kDimBytes, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IDX_OK : IDX_ERR_CUDA;
}

// TMA map of the K codes as [page][64 slots][64 B] with `page_bytes` between
// pages (4096 for the separate-tensor layout, 4352 when the scales follow the
// codes inside each page); one box is one page.
int encode_k_pages(CUtensorMap* map, void* base, uint64_t num_pages, uint64_t page_bytes) {
  cuuint64_t dims[3] = {(cuuint64_t)kDimBytes, (cuuint64_t)kPage, (cuuint64_t)num_pages};
  cuuint64_t strides[2] = {(cuuint64_t)kDimBytes, (cuuint64_t)page_bytes};
  cuuint32_t box[3] = {(cuuint32_t)kDimBytes, (cuuint32_t)kPage, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IDX_OK : IDX_ERR_CUDA;
}

struct Scratch {
  void* base = nullptr;
  ScratchLayout L{};
  PlanHeader* hdr() const { return (PlanHeader*)((char*)base + L.header); }
  template <typename T>
  T* at(size_t off) const {
    return (T*)((char*)base + off);
  }
};

enum class Path { kFused, kDense, kDebug };

struct Call {
  const idx_tensor_t *q_fp4, *q_scale, *k_cache_fp4, *k_scale, *weights, *page_table, *row_req,
      *row_start, *row_end;
  int32_t topk;
  const idx_tensor_t *out_phys, *out_raw;   // prefill outputs
  const idx_tensor_t *scores, *logits;      // dense / debug score outputs
  Path path;
  const idx_tensor_t* k_pages = nullptr;    // page-interleaved K cache (replaces the two K tensors)
  bool k_scale_mma = false;                 // k_scale [NP, 256] in the MMA's scale-copy order
};

// Where the scorer finds a page's codes and scales for a call.
struct KSource {
  void* codes;
  uint64_t page_bytes;
  const uint8_t* scales;
  int64_t scale_stride_words;
};

KSource k_source(const Call& c) {
  if (c.k_pages)
    return {c.k_pages->data, (uint64_t)kPage * (kDimBytes + kNumSF),
            (const uint8_t*)c.k_pages->data + kPage * kDimBytes,
            (int64_t)kPage * (kDimBytes + kNumSF) / 4};
  return {c.k_cache_fp4->data, (uint64_t)kPage * kDimBytes, (const uint8_t*)c.k_scale->data,
          (int64_t)kPage};
}

int read_status_and_free(const Scratch& s, cudaStream_t stream, uint32_t* status) {
  // pageable destination: returns once the copy (and all earlier work on the
  // stream) has completed
  cudaError_t e1 = cudaMemcpyAsync(status, s.hdr(), sizeof(uint32_t), cudaMemcpyDeviceToHost, stream);
  cudaError_t e2 = cudaFreeAsync(s.base, stream);
  if (e1 != cudaSuccess || e2 != cudaSuccess) {
    cudaGetLastError();
    return IDX_ERR_CUDA;
  }
  return IDX_OK;
}

int run(const Call& c, cudaStream_t stream) {
  Outputs outs;
  const bool prefill = c.path != Path::kDebug;
  // outputs first, so that later errors can fail closed
  int64_t rows_hint = c.q_fp4 ? c.q_fp4->shape[0] : 0;
  if (prefill) {
    int st = check_output(c.out_phys, rows_hint, c.topk);
    if (st) return st;
    outs.t[0] = c.out_phys;
    if (c.out_raw) {
      st = check_output(c.out_raw, rows_hint, c.topk);
      if (st) return st;
      outs.t[1] = c.out_raw;
    }
  }
  const idx_tensor_t* all[] = {c.q_fp4, c.q_scale, c.k_cache_fp4, c.k_scale, c.weights, c.page_table,
                               c.row_req, c.row_start, c.row_end, c.out_phys, c.out_raw,
                               c.scores, c.logits, c.k_pages};
  int dev = -1;
  int st = common_device(all, 14, &dev);
  if (st) return st;
  DeviceGuard guard(dev);
  if (!guard.ok()) return IDX_ERR_CUDA;
  st = check_stream(stream, dev);
  if (st == IDX_ERR_UNSUPPORTED) return st;  // capturing: enqueue nothing
  auto fail = [&](int code) {
    fill_minus_one(outs, stream);
    return code;
  };
  if (st) return fail(st);
  if (prefill && !topk_supported(c.topk)) return fail(IDX_ERR_UNSUPPORTED);
  Sizes sz;
  st = check_inputs(c.q_fp4, c.q_scale, c.k_cache_fp4, c.k_scale, c.weights, c.page_table,
                    c.row_req, c.row_start, c.row_end, &sz, c.k_pages, c.k_scale_mma);
  if (st) return fail(st);
  int64_t score_stride = 0, logits_stride = 0, check_end = 0;
  if (c.path != Path::kFused && c.scores) {
    if ((st = check_tensor(c.scores, IDX_F32, 2))) return fail(st);
    if (c.scores->shape[0] != sz.rows) return fail(IDX_ERR_INVALID_ARGUMENT);
    score_stride = c.scores->shape[1];
    if (score_stride > INT32_MAX) return fail(IDX_ERR_OVERFLOW);
    check_end = score_stride;
  }
  if (c.path == Path::kDebug) {
    if (!c.scores) return fail(IDX_ERR_INVALID_ARGUMENT);
    if (c.logits) {
      if ((st = check_tensor(c.logits, IDX_F32, 3))) return fail(st);
      if (c.logits->shape[0] != sz.rows || c.logits->shape[1] != kHeads)
        return fail(IDX_ERR_INVALID_ARGUMENT);
      logits_stride = c.logits->shape[2];
      if (logits_stride < check_end) check_end = logits_stride;
    }
  }
  if (sz.rows == 0) return IDX_OK;
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds))) return fail(st);
  if (!(ds->cc_major == 10 && ds->cc_minor == 3)) return fail(IDX_ERR_UNSUPPORTED);

  const int grid = ds->sm_count;
  const bool with_cands = c.path == Path::kFused;
  Scratch s;
  s.L = scratch_layout(sz.rows, c.topk, grid, with_cands);
  // the dense path without a caller workspace materialises [rows, max_pages*64]
  size_t ws_off = 0;
  size_t total = s.L.total;
  if (c.path == Path::kDense && !c.scores) {
    int64_t width = sz.max_pages * kPage, bytes;
    if (!mul_ok(sz.rows, width, &bytes) || !mul_ok(bytes, 4, &bytes)) return fail(IDX_ERR_OVERFLOW);
    ws_off = align_up(total, 256);
    total = ws_off + (size_t)bytes;
    score_stride = width;
    check_end = width;
  }
  if (cudaMallocFromPoolAsync(&s.base, total, ds->pool, stream) != cudaSuccess) {
    cudaGetLastError();
    return fail(IDX_ERR_CUDA);
  }
  float* score_buf = nullptr;
  if (c.path != Path::kFused)
    score_buf = c.scores ? (float*)c.scores->data : s.at<float>(ws_off);

  PlanParams pp{};
  pp.row_req = (const int32_t*)c.row_req->data;
  pp.row_start = (const int32_t*)c.row_start->data;
  pp.row_end = (const int32_t*)c.row_end->data;
  pp.page_table = (const int32_t*)c.page_table->data;
  pp.rows = (int32_t)sz.rows;
  pp.num_req = (int32_t)sz.num_req;
  pp.max_pages = (int32_t)sz.max_pages;
  pp.num_pages = (int32_t)sz.num_pages;
  pp.score_thr = c.path == Path::kDebug ? 0 : c.topk;
  pp.grid = grid;
  pp.check_end_le = c.path == Path::kFused ? -1 : (int32_t)check_end;
  pp.clear_hdr = 1;
  pp.max_units = s.L.max_units;
  pp.max_row_slots = s.L.max_row_slots;
  pp.hdr = s.hdr();
  pp.row_block = s.at<int32_t>(s.L.row_block);
  pp.blocks = s.at<BlockInfo>(s.L.blocks);
  pp.units = s.at<UnitInfo>(s.L.units);
  pp.sched = s.at<int32_t>(s.L.sched);
  int cuda_err = 0;
  CallTimer timer;
  timer.mark(0, stream);
  cuda_err |= launch_plan(pp, stream) != cudaSuccess;

  CUtensorMap tmap_k, tmap_q;
  const KSource ks = k_source(c);
  if (encode_k_pages(&tmap_k, ks.codes, (uint64_t)sz.num_pages, ks.page_bytes) ||
      encode_2d_u8(&tmap_q, c.q_fp4->data, (uint64_t)sz.rows * kHeads, kRowsPerChunk * kHeads)) {
    uint32_t dummy;
    read_status_and_free(s, stream, &dummy);
    return fail(IDX_ERR_CUDA);
  }
  ScoreParams sp{};
  sp.q_scale = (const uint8_t*)c.q_scale->data;
  sp.k_scale = ks.scales;
  sp.k_scale_stride = ks.scale_stride_words;
  sp.k_scale_mma = c.k_scale_mma ? 1 : 0;
  sp.weights = (const float*)c.weights->data;
  sp.page_table = pp.page_table;
  sp.row_start = pp.row_start;
  sp.row_end = pp.row_end;
  sp.rows = pp.rows;
  sp.max_pages = pp.max_pages;
  sp.num_pages = pp.num_pages;
  sp.topk = c.topk;
  sp.mode = c.path == Path::kFused ? kModeSelect : kModeDense;
  sp.dyn = sz.num_req > 1 ? 1 : 0;  // units of several requests differ in length
  sp.score_thr = pp.score_thr;
  sp.hdr = pp.hdr;
  sp.blocks = pp.blocks;
  sp.units = pp.units;
  sp.sched = pp.sched;
  sp.cand_cnt = with_cands ? s.at<uint32_t>(s.L.cand_cnt) : nullptr;
  sp.cand_keys = with_cands ? s.at<uint64_t>(s.L.cand_keys) : nullptr;
  sp.dense_out = score_buf;
  sp.dense_stride = score_stride;
  sp.logits_out = c.logits ? (float*)c.logits->data : nullptr;
  sp.logits_stride = logits_stride;
  timer.mark(1, stream);
  cuda_err |= launch_score(tmap_k, tmap_q, sp, grid, stream) != cudaSuccess;
  timer.mark(2, stream);

  if (prefill) {
    FinishParams fp{};
    fp.row_req = pp.row_req;
    fp.row_start = pp.row_start;
    fp.row_end = pp.row_end;
    fp.page_table = pp.page_table;
    fp.rows = pp.rows;
    fp.max_pages = pp.max_pages;
    fp.num_pages = pp.num_pages;
    fp.topk = c.topk;
    fp.hdr = pp.hdr;
    fp.row_block = pp.row_block;
    fp.blocks = pp.blocks;
    fp.cand_cnt = sp.cand_cnt;
    fp.cand_keys = sp.cand_keys;
    fp.scores = c.path == Path::kDense ? score_buf : nullptr;
    fp.score_stride = score_stride;
    fp.out_phys = (int32_t*)c.out_phys->data;
    fp.out_raw = c.out_raw ? (int32_t*)c.out_raw->data : nullptr;
    cuda_err |= launch_finish(fp, stream) != cudaSuccess;
  }
  timer.mark(3, stream);
  cudaEvent_t end_ev = nullptr;
  if (timer.on && cudaEventCreate(&end_ev) == cudaSuccess) cudaEventRecord(end_ev, stream);
  uint32_t status = 0;
  st = read_status_and_free(s, stream, &status);
  if (end_ev) {
    timer.collect(end_ev);
    cudaEventDestroy(end_ev);
  }
  if (cuda_err || st || cudaGetLastError() != cudaSuccess) return fail(IDX_ERR_CUDA);
  if (status != kOk) return fail((int)status);
  return IDX_OK;
}

// ------------------------------------------------ fixed scratch buffer ----
//
// Scratch of idx_topk_fp4_prefill_noalloc: one buffer per device inside the
// library's own device image (placed there when the image is loaded, not
// allocated by a call).  Its address on a device is looked up once, on the
// first call that uses the device, with that device current.
static __device__ __align__(256) unsigned char g_fixed_scratch[IDX_NOALLOC_SCRATCH_BYTES];
void* g_fixed_ptr[kMaxDevices] = {};
// held for the whole of a call that uses a device's buffer: concurrent calls
// from several host threads run one after another instead of sharing it
std::mutex g_fixed_call_mu[kMaxDevices];

int fixed_scratch(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_fixed_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_fixed_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return IDX_ERR_CUDA;
    }
    g_fixed_ptr[dev] = ptr;
  }
  *out = g_fixed_ptr[dev];
  return IDX_OK;
}

// SM count and compute capability of `dev`, and the tensor-map encoder; unlike
// device_state this creates no memory pool.
int device_info_no_pool(int dev, int* sm, int* major, int* minor) {
  if (dev < 0 || dev >= kMaxDevices) return IDX_ERR_INVALID_ARGUMENT;
  if (cudaDeviceGetAttribute(sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return IDX_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
      cudaGetLastError();
      return IDX_ERR_CUDA;
    }
    g_encode = (EncodeTiledFn)fn;
  }
  return IDX_OK;
}

// The fused path of run() with its scratch taken from the fixed buffer: the
// same checks, kernels, status read-back and fail-closed behaviour, and no
// allocation, pool or event creation.
int run_fixed_scratch(const Call& c, cudaStream_t stream) {
  Outputs outs;
  int st = check_output(c.out_phys, c.q_fp4 ? c.q_fp4->shape[0] : 0, c.topk);
  if (st) return st;
  outs.t[0] = c.out_phys;
  if (c.out_raw) {
    st = check_output(c.out_raw, c.q_fp4 ? c.q_fp4->shape[0] : 0, c.topk);
    if (st) return st;
    outs.t[1] = c.out_raw;
  }
  const idx_tensor_t* all[] = {c.q_fp4, c.q_scale, c.k_cache_fp4, c.k_scale, c.weights,
                               c.page_table, c.row_req, c.row_start, c.row_end, c.out_phys,
                               c.out_raw};
  int dev = -1;
  if ((st = common_device(all, 11, &dev))) return st;
  // the per-device lock and buffer tables are indexed by dev
  if (dev < 0 || dev >= kMaxDevices) return IDX_ERR_INVALID_ARGUMENT;
  DeviceGuard guard(dev);
  if (!guard.ok()) return IDX_ERR_CUDA;
  st = check_stream(stream, dev);
  if (st == IDX_ERR_UNSUPPORTED) return st;  // capturing: enqueue nothing
  auto fail = [&](int code) {
    fill_minus_one(outs, stream);  // also waits for the stream
    return code;
  };
  if (st) return fail(st);
  if (!topk_supported(c.topk)) return fail(IDX_ERR_UNSUPPORTED);
  Sizes sz;
  st = check_inputs(c.q_fp4, c.q_scale, c.k_cache_fp4, c.k_scale, c.weights, c.page_table,
                    c.row_req, c.row_start, c.row_end, &sz);
  if (st) return fail(st);
  if (sz.rows == 0) return IDX_OK;
  std::lock_guard<std::mutex> call_lock(g_fixed_call_mu[dev]);
  int sm = 0, major = 0, minor = 0;
  if ((st = device_info_no_pool(dev, &sm, &major, &minor))) return fail(st);
  if (!(major == 10 && minor == 3)) return fail(IDX_ERR_UNSUPPORTED);
  const int grid = sm;
  Scratch s;
  s.L = scratch_layout(sz.rows, c.topk, grid, true);
  if (s.L.total > (size_t)IDX_NOALLOC_SCRATCH_BYTES) return fail(IDX_ERR_SCRATCH_LIMIT);
  if ((st = fixed_scratch(dev, &s.base))) return fail(st);

  PlanParams pp{};
  pp.row_req = (const int32_t*)c.row_req->data;
  pp.row_start = (const int32_t*)c.row_start->data;
  pp.row_end = (const int32_t*)c.row_end->data;
  pp.page_table = (const int32_t*)c.page_table->data;
  pp.rows = (int32_t)sz.rows;
  pp.num_req = (int32_t)sz.num_req;
  pp.max_pages = (int32_t)sz.max_pages;
  pp.num_pages = (int32_t)sz.num_pages;
  pp.score_thr = c.topk;
  pp.grid = grid;
  pp.check_end_le = -1;
  pp.clear_hdr = 1;
  pp.max_units = s.L.max_units;
  pp.max_row_slots = s.L.max_row_slots;
  pp.hdr = s.hdr();
  pp.row_block = s.at<int32_t>(s.L.row_block);
  pp.blocks = s.at<BlockInfo>(s.L.blocks);
  pp.units = s.at<UnitInfo>(s.L.units);
  pp.sched = s.at<int32_t>(s.L.sched);
  int cuda_err = launch_plan(pp, stream) != cudaSuccess;

  CUtensorMap tmap_k, tmap_q;
  const KSource ks = k_source(c);
  if (encode_k_pages(&tmap_k, ks.codes, (uint64_t)sz.num_pages, ks.page_bytes) ||
      encode_2d_u8(&tmap_q, c.q_fp4->data, (uint64_t)sz.rows * kHeads, kRowsPerChunk * kHeads)) {
    cudaStreamSynchronize(stream);
    cudaGetLastError();
    return fail(IDX_ERR_CUDA);
  }
  ScoreParams sp{};
  sp.q_scale = (const uint8_t*)c.q_scale->data;
  sp.k_scale = ks.scales;
  sp.k_scale_stride = ks.scale_stride_words;
  sp.weights = (const float*)c.weights->data;
  sp.page_table = pp.page_table;
  sp.row_start = pp.row_start;
  sp.row_end = pp.row_end;
  sp.rows = pp.rows;
  sp.max_pages = pp.max_pages;
  sp.num_pages = pp.num_pages;
  sp.topk = c.topk;
  sp.mode = kModeSelect;
  sp.dyn = sz.num_req > 1 ? 1 : 0;  // units of several requests differ in length
  sp.score_thr = pp.score_thr;
  sp.hdr = pp.hdr;
  sp.blocks = pp.blocks;
  sp.units = pp.units;
  sp.sched = pp.sched;
  sp.cand_cnt = s.at<uint32_t>(s.L.cand_cnt);
  sp.cand_keys = s.at<uint64_t>(s.L.cand_keys);
  cuda_err |= launch_score(tmap_k, tmap_q, sp, grid, stream) != cudaSuccess;

  FinishParams fp{};
  fp.row_req = pp.row_req;
  fp.row_start = pp.row_start;
  fp.row_end = pp.row_end;
  fp.page_table = pp.page_table;
  fp.rows = pp.rows;
  fp.max_pages = pp.max_pages;
  fp.num_pages = pp.num_pages;
  fp.topk = c.topk;
  fp.hdr = pp.hdr;
  fp.row_block = pp.row_block;
  fp.blocks = pp.blocks;
  fp.cand_cnt = sp.cand_cnt;
  fp.cand_keys = sp.cand_keys;
  fp.out_phys = (int32_t*)c.out_phys->data;
  fp.out_raw = c.out_raw ? (int32_t*)c.out_raw->data : nullptr;
  cuda_err |= launch_finish(fp, stream) != cudaSuccess;

  // pageable destination: returns once all of the call's work has completed
  uint32_t status = 0;
  if (cudaMemcpyAsync(&status, s.hdr(), sizeof(uint32_t), cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    cuda_err = 1;
  if (cuda_err || cudaGetLastError() != cudaSuccess) {
    // a launch or the read-back failed: wait until every kernel that was
    // enqueued has finished with the shared buffer before the lock is released
    cudaStreamSynchronize(stream);
    cudaGetLastError();
    return fail(IDX_ERR_CUDA);
  }
  if (status != kOk) return fail((int)status);
  return IDX_OK;
}

// ----------------------------------------- context-tiled comparison path ----
//
// Scores one context chunk of `tile` positions at a time into a bounded fp32
// buffer [rows, tile] (the fused kernel's dense mode on the chunk's part of
// each window) and folds every chunk into each row's running TopK; the
// outputs are the fused path's.  Scratch: plan + rows * tile * 4 B + rows *
// topk * 8 B, independent of the context length.
int run_tiled(const Call& c, int32_t tile, cudaStream_t stream) {
  Outputs outs;
  int st = check_output(c.out_phys, c.q_fp4 ? c.q_fp4->shape[0] : 0, c.topk);
  if (st) return st;
  outs.t[0] = c.out_phys;
  if (c.out_raw) {
    if ((st = check_output(c.out_raw, c.q_fp4 ? c.q_fp4->shape[0] : 0, c.topk))) return st;
    outs.t[1] = c.out_raw;
  }
  const idx_tensor_t* all[] = {c.q_fp4, c.q_scale, c.k_cache_fp4, c.k_scale, c.weights,
                               c.page_table, c.row_req, c.row_start, c.row_end, c.out_phys,
                               c.out_raw};
  int dev = -1;
  if ((st = common_device(all, 11, &dev))) return st;
  DeviceGuard guard(dev);
  if (!guard.ok()) return IDX_ERR_CUDA;
  st = check_stream(stream, dev);
  if (st == IDX_ERR_UNSUPPORTED) return st;
  auto fail = [&](int code) {
    fill_minus_one(outs, stream);
    return code;
  };
  if (st) return fail(st);
  if (!topk_supported(c.topk)) return fail(IDX_ERR_UNSUPPORTED);
  if (tile < 1024 || tile % kTile != 0) return fail(IDX_ERR_INVALID_ARGUMENT);
  Sizes sz;
  if ((st = check_inputs(c.q_fp4, c.q_scale, c.k_cache_fp4, c.k_scale, c.weights, c.page_table,
                         c.row_req, c.row_start, c.row_end, &sz)))
    return fail(st);
  if (sz.rows == 0) return IDX_OK;
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds))) return fail(st);
  if (!(ds->cc_major == 10 && ds->cc_minor == 3)) return fail(IDX_ERR_UNSUPPORTED);
  const int grid = ds->sm_count;
  const int64_t R = sz.rows;
  Scratch s;
  s.L = scratch_layout(R, c.topk, grid, false);
  int64_t chunk_bytes, run_bytes;
  if (!mul_ok(R, (int64_t)tile * 4, &chunk_bytes) || !mul_ok(R, (int64_t)c.topk * 8, &run_bytes))
    return fail(IDX_ERR_OVERFLOW);
  const size_t off_chunk = align_up(s.L.total, 256);
  const size_t off_run = align_up(off_chunk + (size_t)chunk_bytes, 256);
  const size_t off_cnt = align_up(off_run + (size_t)run_bytes, 256);
  const size_t off_tau = align_up(off_cnt + (size_t)R * 4, 256);
  const size_t off_win = align_up(off_tau + (size_t)R * 8, 256);
  const size_t total = off_win + align_up((size_t)R * 8, 256);
  if (cudaMallocFromPoolAsync(&s.base, total, ds->pool, stream) != cudaSuccess) {
    cudaGetLastError();
    return fail(IDX_ERR_CUDA);
  }
  cudaMemsetAsync(s.hdr(), 0, sizeof(PlanHeader), stream);
  int32_t* cs = s.at<int32_t>(off_win);
  int32_t* ce = cs + R;
  int32_t max_end = 0;
  {
    // the chunk loop needs the largest window end; a short read of row_end
    // (the call synchronises on the caller stream anyway)
    std::vector<int32_t> ends((size_t)R);
    if (cudaMemcpyAsync(ends.data(), c.row_end->data, (size_t)R * 4, cudaMemcpyDeviceToHost,
                        stream) != cudaSuccess) {
      cudaGetLastError();
      uint32_t dummy;
      read_status_and_free(s, stream, &dummy);
      return fail(IDX_ERR_CUDA);
    }
    for (int32_t e : ends) max_end = e > max_end ? e : max_end;
  }
  if ((int64_t)max_end > sz.max_pages * kPage) {  // also bounds the chunk loop
    uint32_t dummy;
    read_status_and_free(s, stream, &dummy);
    return fail(IDX_ERR_INVALID_METADATA);
  }
  CUtensorMap tmap_k, tmap_q;
  const KSource ks = k_source(c);
  if (encode_k_pages(&tmap_k, ks.codes, (uint64_t)sz.num_pages, ks.page_bytes) ||
      encode_2d_u8(&tmap_q, c.q_fp4->data, (uint64_t)R * kHeads, kRowsPerChunk * kHeads)) {
    uint32_t dummy;
    read_status_and_free(s, stream, &dummy);
    return fail(IDX_ERR_CUDA);
  }
  int cuda_err = 0;
  CallTimer timer;
  timer.mark(0, stream);
  const int32_t n_chunks = max_end > 0 ? (max_end + tile - 1) / tile : 1;
  for (int32_t k = 0; k < n_chunks; ++k) {
    const int32_t c0 = k * tile, c1 = c0 + tile;
    cuda_err |= launch_clip_windows((const int32_t*)c.row_start->data,
                                    (const int32_t*)c.row_end->data, (int32_t)R, c0, c1, c.topk,
                                    cs, ce, stream) != cudaSuccess;
    PlanParams pp{};
    pp.row_req = (const int32_t*)c.row_req->data;
    pp.row_start = cs;
    pp.row_end = ce;
    pp.page_table = (const int32_t*)c.page_table->data;
    pp.rows = (int32_t)R;
    pp.num_req = (int32_t)sz.num_req;
    pp.max_pages = (int32_t)sz.max_pages;
    pp.num_pages = (int32_t)sz.num_pages;
    pp.score_thr = 0;
    pp.grid = grid;
    pp.check_end_le = -1;
    pp.max_units = s.L.max_units;
    pp.max_row_slots = s.L.max_row_slots;
    pp.hdr = s.hdr();
    pp.row_block = s.at<int32_t>(s.L.row_block);
    pp.blocks = s.at<BlockInfo>(s.L.blocks);
    pp.units = s.at<UnitInfo>(s.L.units);
    pp.sched = s.at<int32_t>(s.L.sched);
    cuda_err |= launch_plan(pp, stream) != cudaSuccess;
    ScoreParams sp{};
    sp.q_scale = (const uint8_t*)c.q_scale->data;
    sp.k_scale = ks.scales;
    sp.k_scale_stride = ks.scale_stride_words;
    sp.weights = (const float*)c.weights->data;
    sp.page_table = pp.page_table;
    sp.row_start = cs;
    sp.row_end = ce;
    sp.rows = pp.rows;
    sp.max_pages = pp.max_pages;
    sp.num_pages = pp.num_pages;
    sp.topk = 0;
    sp.mode = kModeDense;
    sp.score_thr = 0;
    sp.hdr = pp.hdr;
    sp.blocks = pp.blocks;
    sp.units = pp.units;
    sp.sched = pp.sched;
    sp.dense_out = s.at<float>(off_chunk);
    sp.dense_stride = tile;
    sp.dense_col0 = c0;
    cuda_err |= launch_score(tmap_k, tmap_q, sp, grid, stream) != cudaSuccess;
    TileMergeParams mp{};
    mp.row_req = pp.row_req;
    mp.row_start = (const int32_t*)c.row_start->data;
    mp.row_end = (const int32_t*)c.row_end->data;
    mp.page_table = pp.page_table;
    mp.rows = (int32_t)R;
    mp.max_pages = pp.max_pages;
    mp.num_pages = pp.num_pages;
    mp.topk = c.topk;
    mp.c0 = c0;
    mp.c1 = c1;
    mp.first = k == 0;
    mp.last = k == n_chunks - 1;
    mp.stride = tile;
    mp.chunk = sp.dense_out;
    mp.run_keys = s.at<uint64_t>(off_run);
    mp.run_cnt = s.at<uint32_t>(off_cnt);
    mp.run_tau = s.at<uint64_t>(off_tau);
    mp.hdr = pp.hdr;
    mp.out_phys = (int32_t*)c.out_phys->data;
    mp.out_raw = c.out_raw ? (int32_t*)c.out_raw->data : nullptr;
    cuda_err |= launch_tile_merge(mp, stream) != cudaSuccess;
  }
  timer.mark(1, stream);
  timer.mark(2, stream);
  timer.mark(3, stream);
  cudaEvent_t end_ev = nullptr;
  if (timer.on && cudaEventCreate(&end_ev) == cudaSuccess) cudaEventRecord(end_ev, stream);
  uint32_t status = 0;
  st = read_status_and_free(s, stream, &status);
  if (end_ev) {
    timer.collect(end_ev);
    cudaEventDestroy(end_ev);
  }
  if (cuda_err || st || cudaGetLastError() != cudaSuccess) return fail(IDX_ERR_CUDA);
  if (status != kOk) return fail((int)status);
  return IDX_OK;
}

// ------------------------------------------------ context-parallel pieces ----
//
// A context shard: every row is scored against the part of its window inside
// [c0, c1) only, and emits that part's exact TopK with the scores (sorted,
// padded with -1 / NaN).  Rows whose whole window is at most topk long emit
// nothing: the merge gives them the closed form.  The shards of a context
// partition, gathered into [S, rows, topk] lists, are merged exactly by
// run_merge_shards ("[FlyDSL][DSv4] Prototype FP4 MQA streaming TopK",
// ROCm/aiter#5282, Changes: exact merge of split candidates; "[AMD][DSv4] Add
// experimental AITER FP4 streaming TopK", sglang#38101, Changes: context-
// parallel paths).
int run_shard(const Call& c, int32_t c0, int32_t c1, const idx_tensor_t* out_score,
              cudaStream_t stream) {
  const int64_t R0 = c.q_fp4 ? c.q_fp4->shape[0] : 0;
  int st = check_output(c.out_raw, R0, c.topk);
  if (st) return st;
  if ((st = check_tensor(out_score, IDX_F32, 2))) return st;
  if (out_score->shape[0] != R0 || out_score->shape[1] != c.topk) return IDX_ERR_INVALID_ARGUMENT;
  Outputs outs;
  outs.t[0] = c.out_raw;
  outs.t[1] = out_score;  // 0xFF bytes: NaN scores
  const idx_tensor_t* all[] = {c.q_fp4, c.q_scale, c.k_cache_fp4, c.k_scale, c.weights,
                               c.page_table, c.row_req, c.row_start, c.row_end, c.out_raw,
                               out_score};
  int dev = -1;
  if ((st = common_device(all, 11, &dev))) return st;
  DeviceGuard guard(dev);
  if (!guard.ok()) return IDX_ERR_CUDA;
  st = check_stream(stream, dev);
  if (st == IDX_ERR_UNSUPPORTED) return st;
  auto fail = [&](int code) {
    fill_minus_one(outs, stream);
    return code;
  };
  if (st) return fail(st);
  if (!topk_supported(c.topk)) return fail(IDX_ERR_UNSUPPORTED);
  if (c0 < 0 || c1 < c0) return fail(IDX_ERR_INVALID_ARGUMENT);
  Sizes sz;
  if ((st = check_inputs(c.q_fp4, c.q_scale, c.k_cache_fp4, c.k_scale, c.weights, c.page_table,
                         c.row_req, c.row_start, c.row_end, &sz)))
    return fail(st);
  if (sz.rows == 0) return IDX_OK;
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds))) return fail(st);
  if (!(ds->cc_major == 10 && ds->cc_minor == 3)) return fail(IDX_ERR_UNSUPPORTED);
  const int grid = ds->sm_count;
  const int64_t R = sz.rows;
  Scratch s;
  s.L = scratch_layout(R, c.topk, grid, true);
  const size_t off_win = align_up(s.L.total, 256);
  const size_t total = off_win + align_up((size_t)R * 8, 256);
  if (cudaMallocFromPoolAsync(&s.base, total, ds->pool, stream) != cudaSuccess) {
    cudaGetLastError();
    return fail(IDX_ERR_CUDA);
  }
  cudaMemsetAsync(s.hdr(), 0, sizeof(PlanHeader), stream);
  int32_t* cs = s.at<int32_t>(off_win);
  int32_t* ce = cs + R;
  int cuda_err = 0;
  // the whole windows first (the clipped ones are what the plan checks)
  cuda_err |= launch_validate_windows((const int32_t*)c.row_start->data,
                                      (const int32_t*)c.row_end->data, (int32_t)R,
                                      sz.max_pages * kPage, s.hdr(), stream,
                                      (const int32_t*)c.row_req->data, (int32_t)sz.num_req) !=
              cudaSuccess;
  cuda_err |= launch_clip_windows((const int32_t*)c.row_start->data,
                                  (const int32_t*)c.row_end->data, (int32_t)R, c0, c1, c.topk, cs,
                                  ce, stream) != cudaSuccess;
  PlanParams pp{};
  pp.row_req = (const int32_t*)c.row_req->data;
  pp.row_start = cs;
  pp.row_end = ce;
  pp.page_table = (const int32_t*)c.page_table->data;
  pp.rows = (int32_t)R;
  pp.num_req = (int32_t)sz.num_req;
  pp.max_pages = (int32_t)sz.max_pages;
  pp.num_pages = (int32_t)sz.num_pages;
  pp.score_thr = 0;  // every nonempty clipped window is scored
  pp.grid = grid;
  pp.check_end_le = -1;
  pp.max_units = s.L.max_units;
  pp.max_row_slots = s.L.max_row_slots;
  pp.hdr = s.hdr();
  pp.row_block = s.at<int32_t>(s.L.row_block);
  pp.blocks = s.at<BlockInfo>(s.L.blocks);
  pp.units = s.at<UnitInfo>(s.L.units);
  pp.sched = s.at<int32_t>(s.L.sched);
  cuda_err |= launch_plan(pp, stream) != cudaSuccess;
  CUtensorMap tmap_k, tmap_q;
  const KSource ks = k_source(c);
  if (encode_k_pages(&tmap_k, ks.codes, (uint64_t)sz.num_pages, ks.page_bytes) ||
      encode_2d_u8(&tmap_q, c.q_fp4->data, (uint64_t)R * kHeads, kRowsPerChunk * kHeads)) {
    uint32_t dummy;
    read_status_and_free(s, stream, &dummy);
    return fail(IDX_ERR_CUDA);
  }
  ScoreParams sp{};
  sp.q_scale = (const uint8_t*)c.q_scale->data;
  sp.k_scale = ks.scales;
  sp.k_scale_stride = ks.scale_stride_words;
  sp.weights = (const float*)c.weights->data;
  sp.page_table = pp.page_table;
  sp.row_start = cs;
  sp.row_end = ce;
  sp.rows = pp.rows;
  sp.max_pages = pp.max_pages;
  sp.num_pages = pp.num_pages;
  sp.topk = c.topk;
  sp.mode = kModeSelect;
  sp.dyn = sz.num_req > 1 ? 1 : 0;  // units of several requests differ in length
  sp.score_thr = 0;
  sp.hdr = pp.hdr;
  sp.blocks = pp.blocks;
  sp.units = pp.units;
  sp.sched = pp.sched;
  sp.cand_cnt = s.at<uint32_t>(s.L.cand_cnt);
  sp.cand_keys = s.at<uint64_t>(s.L.cand_keys);
  cuda_err |= launch_score(tmap_k, tmap_q, sp, grid, stream) != cudaSuccess;
  FinishParams fp{};
  fp.row_req = pp.row_req;
  fp.row_start = cs;
  fp.row_end = ce;
  fp.page_table = nullptr;  // a shard emits positions and scores, no slots
  fp.rows = pp.rows;
  fp.max_pages = pp.max_pages;
  fp.num_pages = pp.num_pages;
  fp.topk = c.topk;
  fp.hdr = pp.hdr;
  fp.row_block = pp.row_block;
  fp.blocks = pp.blocks;
  fp.cand_cnt = sp.cand_cnt;
  fp.cand_keys = sp.cand_keys;
  fp.out_raw = (int32_t*)c.out_raw->data;
  fp.out_score = (float*)out_score->data;
  cuda_err |= launch_finish(fp, stream) != cudaSuccess;
  uint32_t status = 0;
  st = read_status_and_free(s, stream, &status);
  if (cuda_err || st || cudaGetLastError() != cudaSuccess) return fail(IDX_ERR_CUDA);
  if (status != kOk) return fail((int)status);
  return IDX_OK;
}

int run_merge_shards(const idx_tensor_t* shard_score, const idx_tensor_t* shard_raw,
                     const idx_tensor_t* page_table, const idx_tensor_t* row_req,
                     const idx_tensor_t* row_start, const idx_tensor_t* row_end, int32_t topk,
                     const idx_tensor_t* out_phys, const idx_tensor_t* out_raw,
                     cudaStream_t stream) {
  if (!out_phys) return IDX_ERR_INVALID_ARGUMENT;
  const int64_t R = out_phys->shape[0];
  int st = check_output(out_phys, R, topk);
  if (st) return st;
  if (out_raw && (st = check_output(out_raw, R, topk))) return st;
  Outputs outs;
  outs.t[0] = out_phys;
  outs.t[1] = out_raw;
  const idx_tensor_t* all[] = {shard_score, shard_raw, page_table, row_req, row_start, row_end,
                               out_phys, out_raw};
  int dev = -1;
  if ((st = common_device(all, 8, &dev))) return st;
  DeviceGuard guard(dev);
  if (!guard.ok()) return IDX_ERR_CUDA;
  st = check_stream(stream, dev);
  if (st == IDX_ERR_UNSUPPORTED) return st;
  auto fail = [&](int code) {
    fill_minus_one(outs, stream);
    return code;
  };
  if (st) return fail(st);
  if (!topk_supported(topk)) return fail(IDX_ERR_UNSUPPORTED);
  if ((st = check_tensor(shard_score, IDX_F32, 3)) || (st = check_tensor(shard_raw, IDX_I32, 3)) ||
      (st = check_tensor(page_table, IDX_I32, 2)) || (st = check_tensor(row_req, IDX_I32, 1)) ||
      (st = check_tensor(row_start, IDX_I32, 1)) || (st = check_tensor(row_end, IDX_I32, 1)))
    return fail(st);
  const int64_t S = shard_raw->shape[0];
  for (int i = 0; i < 3; ++i)
    if (shard_score->shape[i] != shard_raw->shape[i]) return fail(IDX_ERR_INVALID_ARGUMENT);
  if (S < 1 || shard_raw->shape[1] != R || shard_raw->shape[2] != topk ||
      row_req->shape[0] != R || row_start->shape[0] != R || row_end->shape[0] != R)
    return fail(IDX_ERR_INVALID_ARGUMENT);
  const int64_t num_req = page_table->shape[0], max_pages = page_table->shape[1];
  if (R > INT32_MAX || S > INT32_MAX || num_req > INT32_MAX || max_pages * (int64_t)kPage > INT32_MAX)
    return fail(IDX_ERR_OVERFLOW);
  if (R == 0) return IDX_OK;
  if (num_req < 1 || max_pages < 1) return fail(IDX_ERR_INVALID_ARGUMENT);
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds))) return fail(st);
  if (!(ds->cc_major == 10 && ds->cc_minor == 3)) return fail(IDX_ERR_UNSUPPORTED);
  Scratch s;
  s.L = scratch_layout(0, topk, 0, false);
  if (cudaMallocFromPoolAsync(&s.base, s.L.total, ds->pool, stream) != cudaSuccess) {
    cudaGetLastError();
    return fail(IDX_ERR_CUDA);
  }
  cudaMemsetAsync(s.hdr(), 0, sizeof(PlanHeader), stream);
  int cuda_err = 0;
  cuda_err |= launch_validate_windows((const int32_t*)row_start->data, (const int32_t*)row_end->data,
                                      (int32_t)R, max_pages * kPage, s.hdr(), stream,
                                      (const int32_t*)row_req->data, (int32_t)num_req) != cudaSuccess;
  FinishParams fp{};
  fp.row_req = (const int32_t*)row_req->data;
  fp.row_start = (const int32_t*)row_start->data;
  fp.row_end = (const int32_t*)row_end->data;
  fp.page_table = (const int32_t*)page_table->data;
  fp.rows = (int32_t)R;
  fp.max_pages = (int32_t)max_pages;
  // the K cache is not an argument of the merge: its page count is unknown here,
  // so a mapped entry is only required to be non-negative
  fp.num_pages = INT32_MAX;
  fp.topk = topk;
  fp.hdr = s.hdr();
  fp.n_shards = (int32_t)S;
  fp.shard_score = (const float*)shard_score->data;
  fp.shard_raw = (const int32_t*)shard_raw->data;
  fp.out_phys = (int32_t*)out_phys->data;
  fp.out_raw = out_raw ? (int32_t*)out_raw->data : nullptr;
  cuda_err |= launch_finish(fp, stream) != cudaSuccess;
  uint32_t status = 0;
  st = read_status_and_free(s, stream, &status);
  if (cuda_err || st || cudaGetLastError() != cudaSuccess) return fail(IDX_ERR_CUDA);
  if (status != kOk) return fail((int)status);
  return IDX_OK;
}

// ------------------------------------------------ stream-ordered call ----
//
// The fused path with a caller workspace and a device status word: no
// allocation, no host synchronisation, so it may be captured into a CUDA graph.
// Host-side argument errors return at once with nothing enqueued; everything
// the device detects is published to *status_out by the last kernel, which
// also fills the outputs with -1 in that case.
int run_stream_ordered(const Call& c, void* workspace, uint64_t workspace_bytes,
                       uint32_t* status_out, cudaStream_t stream) {
  int st = check_output(c.out_phys, c.q_fp4 ? c.q_fp4->shape[0] : 0, c.topk);
  if (st) return st;
  if (c.out_raw && (st = check_output(c.out_raw, c.q_fp4 ? c.q_fp4->shape[0] : 0, c.topk)))
    return st;
  if (!status_out || ((uintptr_t)status_out & 3u) != 0) return IDX_ERR_INVALID_ARGUMENT;
  const idx_tensor_t* all[] = {c.q_fp4, c.q_scale, c.k_cache_fp4, c.k_scale, c.weights,
                               c.page_table, c.row_req, c.row_start, c.row_end, c.out_phys,
                               c.out_raw};
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return IDX_ERR_CUDA;
  }
  const bool capturing = cs != cudaStreamCaptureStatusNone;
  int dev = -1;
  if (capturing) {
    // pointer and stream-device queries fail while a stream is captured: the
    // device is the current one (the caller guarantees that the stream and
    // the tensors belong to it)
    if (cudaGetDevice(&dev) != cudaSuccess) {
      cudaGetLastError();
      return IDX_ERR_CUDA;
    }
  } else {
    if ((st = common_device(all, 11, &dev))) return st;
    if (device_of(status_out) != dev) return IDX_ERR_INVALID_ARGUMENT;
  }
  DeviceGuard guard(dev);
  if (!guard.ok()) return IDX_ERR_CUDA;
  if (stream != nullptr && !capturing) {
    int sd = -1;
    if (cudaStreamGetDevice(stream, &sd) != cudaSuccess) {
      cudaGetLastError();
      return IDX_ERR_INVALID_ARGUMENT;
    }
    if (sd != dev) return IDX_ERR_INVALID_ARGUMENT;
  }
  if (!topk_supported(c.topk)) return IDX_ERR_UNSUPPORTED;
  Sizes sz;
  if ((st = check_inputs(c.q_fp4, c.q_scale, c.k_cache_fp4, c.k_scale, c.weights, c.page_table,
                         c.row_req, c.row_start, c.row_end, &sz)))
    return st;
  int sm = 0, major = 0, minor = 0;
  if ((st = device_info_no_pool(dev, &sm, &major, &minor))) return st;
  if (!(major == 10 && minor == 3)) return IDX_ERR_UNSUPPORTED;
  const int grid = sm;
  Scratch s;
  s.L = scratch_layout(sz.rows, c.topk, grid, true);
  if (sz.rows > 0) {
    if (!workspace || ((uintptr_t)workspace & 255u) != 0 || workspace_bytes < s.L.total ||
        (!capturing && device_of(workspace) != dev))
      return IDX_ERR_INVALID_ARGUMENT;
  }
  if (sz.rows == 0) {
    return cudaMemsetAsync(status_out, 0, sizeof(uint32_t), stream) == cudaSuccess ? IDX_OK
                                                                                   : IDX_ERR_CUDA;
  }
  s.base = workspace;
  int cuda_err = 0;

  PlanParams pp{};
  pp.row_req = (const int32_t*)c.row_req->data;
  pp.row_start = (const int32_t*)c.row_start->data;
  pp.row_end = (const int32_t*)c.row_end->data;
  pp.page_table = (const int32_t*)c.page_table->data;
  pp.rows = (int32_t)sz.rows;
  pp.num_req = (int32_t)sz.num_req;
  pp.max_pages = (int32_t)sz.max_pages;
  pp.num_pages = (int32_t)sz.num_pages;
  pp.score_thr = c.topk;
  pp.grid = grid;
  pp.check_end_le = -1;
  pp.clear_hdr = 1;
  pp.max_units = s.L.max_units;
  pp.max_row_slots = s.L.max_row_slots;
  pp.hdr = s.hdr();
  pp.row_block = s.at<int32_t>(s.L.row_block);
  pp.blocks = s.at<BlockInfo>(s.L.blocks);
  pp.units = s.at<UnitInfo>(s.L.units);
  pp.sched = s.at<int32_t>(s.L.sched);
  cuda_err |= launch_plan(pp, stream) != cudaSuccess;

  CUtensorMap tmap_k, tmap_q;
  const KSource ks = k_source(c);
  if (encode_k_pages(&tmap_k, ks.codes, (uint64_t)sz.num_pages, ks.page_bytes) ||
      encode_2d_u8(&tmap_q, c.q_fp4->data, (uint64_t)sz.rows * kHeads, kRowsPerChunk * kHeads))
    return IDX_ERR_CUDA;
  ScoreParams sp{};
  sp.q_scale = (const uint8_t*)c.q_scale->data;
  sp.k_scale = ks.scales;
  sp.k_scale_stride = ks.scale_stride_words;
  sp.weights = (const float*)c.weights->data;
  sp.page_table = pp.page_table;
  sp.row_start = pp.row_start;
  sp.row_end = pp.row_end;
  sp.rows = pp.rows;
  sp.max_pages = pp.max_pages;
  sp.num_pages = pp.num_pages;
  sp.topk = c.topk;
  sp.mode = kModeSelect;
  sp.dyn = sz.num_req > 1 ? 1 : 0;  // units of several requests differ in length
  sp.score_thr = pp.score_thr;
  sp.hdr = pp.hdr;
  sp.blocks = pp.blocks;
  sp.units = pp.units;
  sp.sched = pp.sched;
  sp.cand_cnt = s.at<uint32_t>(s.L.cand_cnt);
  sp.cand_keys = s.at<uint64_t>(s.L.cand_keys);
  cuda_err |= launch_score(tmap_k, tmap_q, sp, grid, stream) != cudaSuccess;

  FinishParams fp{};
  fp.row_req = pp.row_req;
  fp.row_start = pp.row_start;
  fp.row_end = pp.row_end;
  fp.page_table = pp.page_table;
  fp.rows = pp.rows;
  fp.max_pages = pp.max_pages;
  fp.num_pages = pp.num_pages;
  fp.topk = c.topk;
  fp.hdr = pp.hdr;
  fp.row_block = pp.row_block;
  fp.blocks = pp.blocks;
  fp.cand_cnt = sp.cand_cnt;
  fp.cand_keys = sp.cand_keys;
  fp.out_phys = (int32_t*)c.out_phys->data;
  fp.out_raw = c.out_raw ? (int32_t*)c.out_raw->data : nullptr;
  fp.status_out = status_out;  // published by the finishing kernel's last CTA
  cuda_err |= launch_finish(fp, stream) != cudaSuccess;
  if (cuda_err) {
    cudaGetLastError();
    return IDX_ERR_CUDA;
  }
  return IDX_OK;
}

// ---------------------------------------------------- host-buffer call ----
//
// idx_topk_fp4_prefill_host: the inputs and outputs live in host memory.  The
// call stages them through one block of the device's pool (one
// cudaMemcpyAsync per tensor on the caller's stream), runs the fused path on
// the staged copies and copies the outputs back.

// True when t is empty or its data is host memory (pageable or pinned).
bool is_host_tensor(const idx_tensor_t* t) {
  if (!t || numel_of(t) == 0) return true;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, t->data) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeUnregistered;
}

size_t tensor_bytes(const idx_tensor_t* t) {
  return t ? (size_t)numel_of(t) * (t->dtype == IDX_U8 ? 1u : 4u) : 0u;
}

int run_host(const Call& h, int32_t device, cudaStream_t stream) {
  const int64_t R = h.q_fp4 ? h.q_fp4->shape[0] : 0;
  int st = check_output(h.out_phys, R, h.topk, false);
  if (st) return st;
  if (h.out_raw && (st = check_output(h.out_raw, R, h.topk, false))) return st;
  if (!is_host_tensor(h.out_phys) || !is_host_tensor(h.out_raw)) return IDX_ERR_INVALID_ARGUMENT;
  const idx_tensor_t* outs[2] = {h.out_phys, h.out_raw};
  auto host_fail = [&](int code) {
    for (const idx_tensor_t* t : outs)
      if (t && numel_of(t) > 0) std::memset(t->data, 0xFF, tensor_bytes(t));
    return code;
  };
  const idx_tensor_t* in[9] = {h.q_fp4, h.q_scale, h.k_cache_fp4, h.k_scale, h.weights,
                               h.page_table, h.row_req, h.row_start, h.row_end};
  const int in_dtype[9] = {IDX_U8, IDX_U8, IDX_U8, IDX_U8, IDX_F32, IDX_I32, IDX_I32, IDX_I32, IDX_I32};
  const int in_ndim[9] = {3, 3, 3, 3, 2, 2, 1, 1, 1};
  for (int i = 0; i < 9; ++i) {
    if ((st = check_tensor(in[i], in_dtype[i], in_ndim[i], false))) return host_fail(st);
    if (!is_host_tensor(in[i])) return host_fail(IDX_ERR_INVALID_ARGUMENT);
  }
  int n_dev = 0;
  if (cudaGetDeviceCount(&n_dev) != cudaSuccess) {
    cudaGetLastError();
    return host_fail(IDX_ERR_CUDA);
  }
  if (device < 0 || device >= n_dev) return host_fail(IDX_ERR_INVALID_ARGUMENT);
  DeviceGuard guard(device);
  if (!guard.ok()) return host_fail(IDX_ERR_CUDA);
  if ((st = check_stream(stream, device))) return host_fail(st);
  if (R == 0) return IDX_OK;
  DeviceState* ds = nullptr;
  if ((st = device_state(device, &ds))) return host_fail(st);
  // staging layout: the nine inputs, then the two outputs, 256-byte aligned
  size_t off[11], total = 0;
  const idx_tensor_t* all[11] = {in[0], in[1], in[2], in[3], in[4], in[5], in[6], in[7], in[8],
                                 h.out_phys, h.out_raw};
  for (int i = 0; i < 11; ++i) {
    off[i] = total;
    total = align_up(total + tensor_bytes(all[i]), 256);
  }
  void* base = nullptr;
  if (cudaMallocFromPoolAsync(&base, total, ds->pool, stream) != cudaSuccess) {
    cudaGetLastError();
    return host_fail(IDX_ERR_CUDA);
  }
  idx_tensor_t dev_t[11];
  bool cuda_ok = true;
  for (int i = 0; i < 11; ++i) {
    if (!all[i]) continue;
    dev_t[i] = *all[i];
    const size_t bytes = tensor_bytes(all[i]);
    dev_t[i].data = bytes ? (char*)base + off[i] : nullptr;
    if (i < 9 && bytes)
      cuda_ok &= cudaMemcpyAsync(dev_t[i].data, all[i]->data, bytes, cudaMemcpyHostToDevice,
                                 stream) == cudaSuccess;
  }
  int code = IDX_ERR_CUDA;
  if (cuda_ok) {
    Call c{&dev_t[0], &dev_t[1], &dev_t[2], &dev_t[3], &dev_t[4], &dev_t[5], &dev_t[6], &dev_t[7],
           &dev_t[8], h.topk, &dev_t[9], h.out_raw ? &dev_t[10] : nullptr, nullptr, nullptr,
           Path::kFused};
    code = run(c, stream);
  }
  if (code == IDX_OK)
    for (int i = 9; i < 11; ++i)
      if (all[i] && tensor_bytes(all[i]))
        cuda_ok &= cudaMemcpyAsync(all[i]->data, dev_t[i].data, tensor_bytes(all[i]),
                                   cudaMemcpyDeviceToHost, stream) == cudaSuccess;
  cuda_ok &= cudaFreeAsync(base, stream) == cudaSuccess;
  cuda_ok &= cudaStreamSynchronize(stream) == cudaSuccess;
  if (!cuda_ok) {
    cudaGetLastError();
    return host_fail(IDX_ERR_CUDA);
  }
  return code == IDX_OK ? IDX_OK : host_fail(code);
}

const int32_t kSupportedK[2] = {512, 1024};

}  // namespace

extern "C" {

int idx_topk_fp4_prefill(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                         const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                         const idx_tensor_t* weights, const idx_tensor_t* page_table,
                         const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                         const idx_tensor_t* row_end, int32_t topk,
                         const idx_tensor_t* out_phys_slot, const idx_tensor_t* out_raw_idx,
                         idx_stream_t stream) {
  Call c{q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req, row_start, row_end,
         topk, out_phys_slot, out_raw_idx, nullptr, nullptr, Path::kFused};
  return run(c, (cudaStream_t)stream);
}

int idx_topk_fp4_prefill_host(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                              const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                              const idx_tensor_t* weights, const idx_tensor_t* page_table,
                              const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                              const idx_tensor_t* row_end, int32_t topk,
                              const idx_tensor_t* out_phys_slot, const idx_tensor_t* out_raw_idx,
                              int32_t device, idx_stream_t stream) {
  Call c{q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req, row_start, row_end,
         topk, out_phys_slot, out_raw_idx, nullptr, nullptr, Path::kFused};
  return run_host(c, device, (cudaStream_t)stream);
}

int idx_topk_fp4_prefill_noalloc(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                                 const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                                 const idx_tensor_t* weights, const idx_tensor_t* page_table,
                                 const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                                 const idx_tensor_t* row_end, int32_t topk,
                                 const idx_tensor_t* out_phys_slot,
                                 const idx_tensor_t* out_raw_idx, idx_stream_t stream) {
  Call c{q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req, row_start, row_end,
         topk, out_phys_slot, out_raw_idx, nullptr, nullptr, Path::kFused};
  return run_fixed_scratch(c, (cudaStream_t)stream);
}

int idx_topk_fp4_prefill_async(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                               const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                               const idx_tensor_t* weights, const idx_tensor_t* page_table,
                               const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                               const idx_tensor_t* row_end, int32_t topk,
                               const idx_tensor_t* out_phys_slot, const idx_tensor_t* out_raw_idx,
                               void* workspace, uint64_t workspace_bytes, uint32_t* status,
                               idx_stream_t stream) {
  Call c{q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req, row_start, row_end,
         topk, out_phys_slot, out_raw_idx, nullptr, nullptr, Path::kFused};
  return run_stream_ordered(c, workspace, workspace_bytes, status, (cudaStream_t)stream);
}

int idx_topk_fp4_prefill_paged(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                               const idx_tensor_t* k_pages, const idx_tensor_t* weights,
                               const idx_tensor_t* page_table, const idx_tensor_t* row_req,
                               const idx_tensor_t* row_start, const idx_tensor_t* row_end,
                               int32_t topk, const idx_tensor_t* out_phys_slot,
                               const idx_tensor_t* out_raw_idx, idx_stream_t stream) {
  Call c{q_fp4, q_scale, nullptr, nullptr, weights, page_table, row_req, row_start, row_end,
         topk, out_phys_slot, out_raw_idx, nullptr, nullptr, Path::kFused, k_pages};
  return run(c, (cudaStream_t)stream);
}

int idx_topk_fp4_prefill_mma_scales(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                                    const idx_tensor_t* k_cache_fp4,
                                    const idx_tensor_t* k_scale_mma, const idx_tensor_t* weights,
                                    const idx_tensor_t* page_table, const idx_tensor_t* row_req,
                                    const idx_tensor_t* row_start, const idx_tensor_t* row_end,
                                    int32_t topk, const idx_tensor_t* out_phys_slot,
                                    const idx_tensor_t* out_raw_idx, idx_stream_t stream) {
  Call c{q_fp4, q_scale, k_cache_fp4, k_scale_mma, weights, page_table, row_req, row_start,
         row_end, topk, out_phys_slot, out_raw_idx, nullptr, nullptr, Path::kFused};
  c.k_scale_mma = true;
  return run(c, (cudaStream_t)stream);
}

int idx_topk_fp4_prefill_shard(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                               const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                               const idx_tensor_t* weights, const idx_tensor_t* page_table,
                               const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                               const idx_tensor_t* row_end, int32_t ctx_begin, int32_t ctx_end,
                               int32_t topk, const idx_tensor_t* out_score,
                               const idx_tensor_t* out_raw_idx, idx_stream_t stream) {
  Call c{q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req, row_start, row_end,
         topk, nullptr, out_raw_idx, nullptr, nullptr, Path::kFused};
  return run_shard(c, ctx_begin, ctx_end, out_score, (cudaStream_t)stream);
}

int idx_topk_merge_shards(const idx_tensor_t* shard_score, const idx_tensor_t* shard_raw,
                          const idx_tensor_t* page_table, const idx_tensor_t* row_req,
                          const idx_tensor_t* row_start, const idx_tensor_t* row_end,
                          int32_t topk, const idx_tensor_t* out_phys_slot,
                          const idx_tensor_t* out_raw_idx, idx_stream_t stream) {
  return run_merge_shards(shard_score, shard_raw, page_table, row_req, row_start, row_end, topk,
                          out_phys_slot, out_raw_idx, (cudaStream_t)stream);
}

int idx_tiled_topk_fp4_prefill(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                               const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                               const idx_tensor_t* weights, const idx_tensor_t* page_table,
                               const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                               const idx_tensor_t* row_end, int32_t topk, int32_t context_tile,
                               const idx_tensor_t* out_phys_slot, const idx_tensor_t* out_raw_idx,
                               idx_stream_t stream) {
  Call c{q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req, row_start, row_end,
         topk, out_phys_slot, out_raw_idx, nullptr, nullptr, Path::kFused};
  return run_tiled(c, context_tile, (cudaStream_t)stream);
}

int idx_dense_topk_fp4_prefill(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                               const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                               const idx_tensor_t* weights, const idx_tensor_t* page_table,
                               const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                               const idx_tensor_t* row_end, int32_t topk,
                               const idx_tensor_t* out_phys_slot,
                               const idx_tensor_t* out_raw_idx,
                               const idx_tensor_t* score_workspace, idx_stream_t stream) {
  Call c{q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req, row_start, row_end,
         topk, out_phys_slot, out_raw_idx, score_workspace, nullptr, Path::kDense};
  return run(c, (cudaStream_t)stream);
}

int idx_fp4_debug_scores(const idx_tensor_t* q_fp4, const idx_tensor_t* q_scale,
                         const idx_tensor_t* k_cache_fp4, const idx_tensor_t* k_scale,
                         const idx_tensor_t* weights, const idx_tensor_t* page_table,
                         const idx_tensor_t* row_req, const idx_tensor_t* row_start,
                         const idx_tensor_t* row_end, const idx_tensor_t* out_scores,
                         const idx_tensor_t* out_logits, idx_stream_t stream) {
  Call c{q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req, row_start, row_end,
         0, nullptr, nullptr, out_scores, out_logits, Path::kDebug};
  return run(c, (cudaStream_t)stream);
}

int idx_topk_select_scores(const idx_tensor_t* scores, const idx_tensor_t* row_start,
                           const idx_tensor_t* row_end, int32_t topk,
                           const idx_tensor_t* out_raw_idx, idx_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  int st = check_tensor(scores, IDX_F32, 2);
  if (st) return st;
  const int64_t R = scores->shape[0];
  if ((st = check_output(out_raw_idx, R, topk))) return st;
  Outputs outs;
  outs.t[0] = out_raw_idx;
  const idx_tensor_t* all[] = {scores, row_start, row_end, out_raw_idx};
  int dev = -1;
  if ((st = common_device(all, 4, &dev))) return st;
  DeviceGuard guard(dev);
  if (!guard.ok()) return IDX_ERR_CUDA;
  st = check_stream(stream, dev);
  if (st == IDX_ERR_UNSUPPORTED) return st;
  auto fail = [&](int code) {
    fill_minus_one(outs, stream);
    return code;
  };
  if (st) return fail(st);
  if (!topk_supported(topk)) return fail(IDX_ERR_UNSUPPORTED);
  if ((st = check_tensor(row_start, IDX_I32, 1)) || (st = check_tensor(row_end, IDX_I32, 1)))
    return fail(st);
  if (row_start->shape[0] != R || row_end->shape[0] != R) return fail(IDX_ERR_INVALID_ARGUMENT);
  if (R > INT32_MAX || scores->shape[1] > INT32_MAX) return fail(IDX_ERR_OVERFLOW);
  if (R == 0) return IDX_OK;
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds))) return fail(st);
  if (!(ds->cc_major == 10 && ds->cc_minor == 3)) return fail(IDX_ERR_UNSUPPORTED);
  Scratch s;
  s.L = scratch_layout(0, topk, 0, false);
  if (cudaMallocFromPoolAsync(&s.base, s.L.total, ds->pool, stream) != cudaSuccess) {
    cudaGetLastError();
    return fail(IDX_ERR_CUDA);
  }
  cudaMemsetAsync(s.hdr(), 0, sizeof(PlanHeader), stream);
  int cuda_err = 0;
  cuda_err |= launch_validate_windows((const int32_t*)row_start->data, (const int32_t*)row_end->data,
                                      (int32_t)R, scores->shape[1], s.hdr(), stream) != cudaSuccess;
  FinishParams fp{};
  fp.row_start = (const int32_t*)row_start->data;
  fp.row_end = (const int32_t*)row_end->data;
  fp.rows = (int32_t)R;
  fp.topk = topk;
  fp.hdr = s.hdr();
  fp.scores = (const float*)scores->data;
  fp.score_stride = scores->shape[1];
  fp.out_raw = (int32_t*)out_raw_idx->data;
  cuda_err |= launch_finish(fp, stream) != cudaSuccess;
  uint32_t status = 0;
  st = read_status_and_free(s, stream, &status);
  if (cuda_err || st || cudaGetLastError() != cudaSuccess) return fail(IDX_ERR_CUDA);
  if (status != kOk) return fail((int)status);
  return IDX_OK;
}

int idx_topk_supported_k(const int32_t** ks, int32_t* n) {
  if (!ks || !n) return IDX_ERR_INVALID_ARGUMENT;
  *ks = kSupportedK;
  *n = 2;
  return IDX_OK;
}

const char* idx_topk_status_string(int code) {
  switch (code) {
    case IDX_OK: return "ok";
    case IDX_ERR_INVALID_ARGUMENT: return "invalid argument";
    case IDX_ERR_UNSUPPORTED: return "unsupported";
    case IDX_ERR_INVALID_METADATA: return "invalid row metadata";
    case IDX_ERR_INVALID_PAGE: return "invalid page-table entry";
    case IDX_ERR_OVERFLOW: return "size overflow";
    case IDX_ERR_CUDA: return "CUDA error";
    case IDX_ERR_INTERNAL: return "internal selector failure";
    case IDX_ERR_TIMEOUT: return "device wait timed out";
    case IDX_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the fixed buffer holds";
    case IDX_ERR_INVALID_VALUE:
      return "scale byte above 167 or weight not finite or above 2^24 in magnitude";
    default: return "unknown status";
  }
}

int idx_topk_fp4_scratch_bytes(int32_t rows, int32_t topk, int32_t device, uint64_t* bytes) {
  if (!bytes || rows < 0) return IDX_ERR_INVALID_ARGUMENT;
  if (!topk_supported(topk)) return IDX_ERR_UNSUPPORTED;
  int sm = 0;
  if (cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    cudaGetLastError();
    return IDX_ERR_CUDA;
  }
  *bytes = (uint64_t)scratch_layout(rows, topk, sm, true).total;
  return IDX_OK;
}

int idx_topk_set_timing(int32_t enable) {
  g_timing = enable != 0;
  return IDX_OK;
}

int idx_topk_last_timings(float* ms4) {
  if (!ms4) return IDX_ERR_INVALID_ARGUMENT;
  for (int i = 0; i < 4; ++i) ms4[i] = g_last_ms[i];
  return IDX_OK;
}

int idx_debug_bounded_wait(int32_t device, int32_t never_completes, idx_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  DeviceState* ds = nullptr;
  int st = device_state(device, &ds);
  if (st) return st;
  DeviceGuard guard(device);
  if (!guard.ok()) return IDX_ERR_CUDA;
  if ((st = check_stream(stream, device))) return st;
  Scratch s;
  s.L.header = 0;
  s.L.total = align_up(sizeof(PlanHeader), 256);
  if (cudaMallocFromPoolAsync(&s.base, s.L.total, ds->pool, stream) != cudaSuccess) {
    cudaGetLastError();
    return IDX_ERR_CUDA;
  }
  cudaMemsetAsync(s.hdr(), 0, sizeof(PlanHeader), stream);
  const bool launch_err = launch_wait_probe(s.hdr(), never_completes != 0, stream) != cudaSuccess;
  uint32_t status = kOk;
  st = read_status_and_free(s, stream, &status);
  if (launch_err || st || cudaGetLastError() != cudaSuccess) return IDX_ERR_CUDA;
  return (int)status;
}

int idx_topk_scratch_high_water(int32_t device, uint64_t* bytes) {
  if (!bytes) return IDX_ERR_INVALID_ARGUMENT;
  DeviceState* ds = nullptr;
  int st = device_state(device, &ds);
  if (st) return st;
  uint64_t v = 0;
  if (cudaMemPoolGetAttribute(ds->pool, cudaMemPoolAttrReservedMemHigh, &v) != cudaSuccess) {
    cudaGetLastError();
    return IDX_ERR_CUDA;
  }
  *bytes = v;
  return IDX_OK;
}

}  // extern "C"
