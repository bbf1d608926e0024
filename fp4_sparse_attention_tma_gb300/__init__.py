"""GB300 (sm_103a) FP4 paged-MQA indexer prefill with fused exact TopK.

Thin Python binding of the C ABI in include/idxtopk.h: every function below
only marshals torch tensors into descriptors and calls the library of the same
name on the caller's current CUDA stream; every step of the computation runs in
the library's CUDA kernels.  There is no CPU fallback: a missing or unloadable
library raises.

The operation follows "[FlyDSL] Add FP4 LiteTopK prefill operator"
(ROCm/aiter#5309) and "[FlyDSL][DSv4] Prototype FP4 MQA streaming TopK"
(ROCm/aiter#5282): score every query row against its C4 window of the paged FP4
K cache, score = sum_h w * ReLU(q_h . k), and return the exact TopK positions
(physical slots and optional raw positions) without materialising the
[rows, context] score matrix.
"""
from __future__ import annotations

import ctypes
import struct

from . import _lib

__all__ = ["IdxError", "SUPPORTED_K", "idx_topk_fp4_prefill", "idx_topk_fp4_prefill_noalloc",
           "idx_topk_fp4_prefill_host",
           "idx_topk_fp4_prefill_async", "idx_topk_fp4_prefill_paged",
           "idx_topk_fp4_prefill_shard", "idx_topk_merge_shards",
           "idx_topk_fp4_prefill_mma_scales",
           "idx_dense_topk_fp4_prefill", "idx_tiled_topk_fp4_prefill",
           "idx_fp4_debug_scores", "idx_topk_select_scores", "idx_topk_supported_k",
           "idx_topk_status_string", "idx_topk_fp4_scratch_bytes", "idx_topk_scratch_high_water",
           "dense_score_bytes", "STATUS", "idx_topk_set_timing",
           "idx_topk_last_timings", "idx_debug_bounded_wait"]

STATUS = {0: "OK", 1: "INVALID_ARGUMENT", 2: "UNSUPPORTED", 3: "INVALID_METADATA",
          4: "INVALID_PAGE", 5: "OVERFLOW", 6: "CUDA_ERROR", 7: "INTERNAL", 8: "TIMEOUT",
          9: "SCRATCH_LIMIT", 10: "INVALID_VALUE"}
SUPPORTED_K = (512, 1024)

_DT = {"uint8": 1, "int32": 2, "float32": 3}


class IdxError(RuntimeError):
    def __init__(self, code: int, fn: str):
        self.code = int(code)
        super().__init__(f"{fn}: {STATUS.get(code, code)} ({idx_topk_status_string(code)})")


def _desc(t):
    """idx_tensor_t descriptor of a torch tensor (no copy, no layout change)."""
    if t is None:
        return None
    d = _lib.IdxTensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _dtype_code(t.dtype)
    d.ndim = t.dim()
    for i in range(min(4, t.dim())):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


# idx_tensor_t as packed bytes: data pointer, dtype, ndim, shape[4], stride[4]
_DESC = struct.Struct("=Qii4q4q")
_ZERO4 = (0, 0, 0, 0)
_DT_CODE = {}  # torch.dtype -> code, filled on first use


def _dtype_code(dt) -> int:
    c = _DT_CODE.get(dt)
    if c is None:
        c = _DT_CODE[dt] = _DT.get(str(dt).replace("torch.", ""), 0)
    return c


def _descs(ts):
    """Descriptors of the tensors `ts` (None: absent) packed into one buffer.
    Returns the buffer, which must stay alive for the call, and each
    descriptor's address (None for an absent tensor)."""
    buf = ctypes.create_string_buffer(_DESC.size * len(ts))
    base = ctypes.addressof(buf)
    addrs = [None] * len(ts)
    for i, t in enumerate(ts):
        if t is None:
            continue
        sh = t.shape
        st = t.stride()
        n = len(sh)
        if n < 4:
            sh = (*sh, *_ZERO4[n:])
            st = (*st, *_ZERO4[n:])
        _DESC.pack_into(buf, _DESC.size * i, t.data_ptr() if t.numel() else 0,
                        _dtype_code(t.dtype), n, *sh[:4], *st[:4])
        addrs[i] = base + _DESC.size * i
    return buf, addrs


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code: int, fn: str, raise_on_error: bool):
    if code != 0 and raise_on_error:
        raise IdxError(code, fn)
    return code


def idx_topk_fp4_prefill(q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                         row_start, row_end, topk, out_phys_slot, out_raw_idx=None, stream=None,
                         raise_on_error=True) -> int:
    """Fused scoring + exact TopK + page mapping; writes the outputs in place."""
    lib = _lib.load()
    keep, ds = _descs((q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                        row_start, row_end, out_phys_slot, out_raw_idx))
    code = lib.idx_topk_fp4_prefill(*ds[:9], int(topk), ds[9],
                                    ds[10], _stream(stream))
    return _check(code, "idx_topk_fp4_prefill", raise_on_error)


def idx_topk_fp4_prefill_host(q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                              row_start, row_end, topk, out_phys_slot, out_raw_idx=None, device=0,
                              stream=None, raise_on_error=True) -> int:
    """idx_topk_fp4_prefill on CPU tensors (pinned for asynchronous copies): the
    library stages them on `device`, runs the fused path and writes the CPU
    outputs in place before returning."""
    import torch
    lib = _lib.load()
    keep, ds = _descs((q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                        row_start, row_end, out_phys_slot, out_raw_idx))
    if stream is None:
        stream = torch.cuda.current_stream(int(device))
    code = lib.idx_topk_fp4_prefill_host(*ds[:9], int(topk), ds[9],
                                         ds[10], int(device), _stream(stream))
    return _check(code, "idx_topk_fp4_prefill_host", raise_on_error)


def idx_topk_fp4_prefill_paged(q_fp4, q_scale, k_pages, weights, page_table, row_req, row_start,
                               row_end, topk, out_phys_slot, out_raw_idx=None, stream=None,
                               raise_on_error=True) -> int:
    """idx_topk_fp4_prefill on a page-interleaved K cache u8 [NP, 4352]
    (each page: 4096 code bytes, then 256 scale bytes)."""
    lib = _lib.load()
    keep, ds = _descs((q_fp4, q_scale, k_pages, weights, page_table, row_req, row_start,
                        row_end, out_phys_slot, out_raw_idx))
    code = lib.idx_topk_fp4_prefill_paged(*ds[:8], int(topk), ds[8],
                                          ds[9], _stream(stream))
    return _check(code, "idx_topk_fp4_prefill_paged", raise_on_error)


def idx_topk_fp4_prefill_async(q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table,
                               row_req, row_start, row_end, topk, out_phys_slot, workspace, status,
                               out_raw_idx=None, stream=None, raise_on_error=True) -> int:
    """Stream-ordered call: no host sync, no allocation (graph-capturable).
    `workspace` is a uint8 device tensor of at least idx_topk_fp4_scratch_bytes
    bytes; `status` an int32 device tensor of one element that receives the
    device-side status."""
    lib = _lib.load()
    keep, ds = _descs((q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                        row_start, row_end, out_phys_slot, out_raw_idx))
    code = lib.idx_topk_fp4_prefill_async(*ds[:9], int(topk), ds[9],
                                          ds[10], ctypes.c_void_p(workspace.data_ptr()),
                                          ctypes.c_uint64(workspace.numel() * workspace.element_size()),
                                          ctypes.c_void_p(status.data_ptr()), _stream(stream))
    return _check(code, "idx_topk_fp4_prefill_async", raise_on_error)


def idx_topk_fp4_prefill_noalloc(q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table,
                                 row_req, row_start, row_end, topk, out_phys_slot, out_raw_idx=None,
                                 stream=None, raise_on_error=True) -> int:
    """idx_topk_fp4_prefill with its scratch in the library's fixed per-device
    buffer: allocates no device memory.  Calls on one device are serialised by
    a per-device lock held until the call's work has completed, so they never
    overlap on the buffer; the call returns after its stream has finished."""
    lib = _lib.load()
    keep, ds = _descs((q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                        row_start, row_end, out_phys_slot, out_raw_idx))
    code = lib.idx_topk_fp4_prefill_noalloc(*ds[:9], int(topk), ds[9],
                                            ds[10], _stream(stream))
    return _check(code, "idx_topk_fp4_prefill_noalloc", raise_on_error)


def idx_topk_fp4_prefill_mma_scales(q_fp4, q_scale, k_cache_fp4, k_scale_mma, weights,
                                    page_table, row_req, row_start, row_end, topk, out_phys_slot,
                                    out_raw_idx=None, stream=None, raise_on_error=True) -> int:
    """idx_topk_fp4_prefill with the K scales [NP, 256] in the MMA's
    scale-copy order: byte 8j + 4h + b of a page = scale b of slot 32h + j."""
    lib = _lib.load()
    keep, ds = _descs((q_fp4, q_scale, k_cache_fp4, k_scale_mma, weights, page_table,
                        row_req, row_start, row_end, out_phys_slot, out_raw_idx))
    code = lib.idx_topk_fp4_prefill_mma_scales(*ds[:9], int(topk),
                                               ds[9], ds[10], _stream(stream))
    return _check(code, "idx_topk_fp4_prefill_mma_scales", raise_on_error)


def idx_topk_fp4_prefill_shard(q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table,
                               row_req, row_start, row_end, ctx_begin, ctx_end, topk, out_score,
                               out_raw_idx, stream=None, raise_on_error=True) -> int:
    """One context shard: each row longer than topk scored against the part of
    its window inside [ctx_begin, ctx_end); writes that part's exact TopK
    (scores f32 and positions i32 [R, topk], -1 / NaN padded) in place."""
    lib = _lib.load()
    keep, ds = _descs((q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                        row_start, row_end, out_score, out_raw_idx))
    code = lib.idx_topk_fp4_prefill_shard(*ds[:9], int(ctx_begin),
                                          int(ctx_end), int(topk), ds[9], ds[10],
                                          _stream(stream))
    return _check(code, "idx_topk_fp4_prefill_shard", raise_on_error)


def idx_topk_merge_shards(shard_score, shard_raw, page_table, row_req, row_start, row_end, topk,
                          out_phys_slot, out_raw_idx=None, stream=None,
                          raise_on_error=True) -> int:
    """Exact merge of S context-shard lists [S, R, topk] into the TopK outputs
    (short-row contract and page mapping included)."""
    lib = _lib.load()
    keep, ds = _descs((shard_score, shard_raw, page_table, row_req, row_start, row_end,
                        out_phys_slot, out_raw_idx))
    code = lib.idx_topk_merge_shards(*ds[:6], int(topk), ds[6],
                                     ds[7], _stream(stream))
    return _check(code, "idx_topk_merge_shards", raise_on_error)


def idx_dense_topk_fp4_prefill(q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                               row_start, row_end, topk, out_phys_slot, out_raw_idx=None,
                               score_workspace=None, stream=None, raise_on_error=True) -> int:
    """Comparison path: materialised fp32 scores, then a separate TopK."""
    lib = _lib.load()
    keep, ds = _descs((q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                        row_start, row_end, out_phys_slot, out_raw_idx, score_workspace))
    code = lib.idx_dense_topk_fp4_prefill(*ds[:9], int(topk), ds[9],
                                          ds[10], ds[11], _stream(stream))
    return _check(code, "idx_dense_topk_fp4_prefill", raise_on_error)


def idx_tiled_topk_fp4_prefill(q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                               row_start, row_end, topk, out_phys_slot, out_raw_idx=None,
                               context_tile=16384, stream=None, raise_on_error=True) -> int:
    """Comparison path: score `context_tile` positions at a time into a bounded
    fp32 buffer, fold each chunk into the rows' running TopK."""
    lib = _lib.load()
    keep, ds = _descs((q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                        row_start, row_end, out_phys_slot, out_raw_idx))
    code = lib.idx_tiled_topk_fp4_prefill(*ds[:9], int(topk), int(context_tile),
                                          ds[9], ds[10], _stream(stream))
    return _check(code, "idx_tiled_topk_fp4_prefill", raise_on_error)


def idx_fp4_debug_scores(q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                         row_start, row_end, out_scores, out_logits=None, stream=None,
                         raise_on_error=True) -> int:
    """Scores (and optionally per-head logits) from the same scoring kernel."""
    lib = _lib.load()
    keep, ds = _descs((q_fp4, q_scale, k_cache_fp4, k_scale, weights, page_table, row_req,
                        row_start, row_end, out_scores, out_logits))
    code = lib.idx_fp4_debug_scores(*ds, _stream(stream))
    return _check(code, "idx_fp4_debug_scores", raise_on_error)


def idx_topk_select_scores(scores, row_start, row_end, topk, out_raw_idx, stream=None,
                           raise_on_error=True) -> int:
    """Exact TopK of a materialised fp32 score matrix under the total order."""
    lib = _lib.load()
    keep, ds = _descs((scores, row_start, row_end, out_raw_idx))
    code = lib.idx_topk_select_scores(ds[0], ds[1], ds[2], int(topk),
                                      ds[3], _stream(stream))
    return _check(code, "idx_topk_select_scores", raise_on_error)


def idx_topk_supported_k():
    lib = _lib.load()
    ptr = ctypes.POINTER(ctypes.c_int32)()
    n = ctypes.c_int32(0)
    code = lib.idx_topk_supported_k(ctypes.byref(ptr), ctypes.byref(n))
    _check(code, "idx_topk_supported_k", True)
    return tuple(ptr[i] for i in range(n.value))


def idx_topk_status_string(code: int) -> str:
    return _lib.load().idx_topk_status_string(int(code)).decode()


def idx_topk_fp4_scratch_bytes(rows: int, topk: int, device: int = 0) -> int:
    v = ctypes.c_uint64(0)
    code = _lib.load().idx_topk_fp4_scratch_bytes(int(rows), int(topk), int(device),
                                                  ctypes.byref(v))
    _check(code, "idx_topk_fp4_scratch_bytes", True)
    return int(v.value)


def idx_topk_scratch_high_water(device: int = 0) -> int:
    v = ctypes.c_uint64(0)
    code = _lib.load().idx_topk_scratch_high_water(int(device), ctypes.byref(v))
    _check(code, "idx_topk_scratch_high_water", True)
    return int(v.value)


def idx_debug_bounded_wait(never_completes: bool, device: int = 0, stream=None) -> int:
    """Failure-detection diagnostic: the status a bounded device wait records
    (0, or IDX_ERR_TIMEOUT = 8 after its 2 s limit when nothing completes it)."""
    return int(_lib.load().idx_debug_bounded_wait(int(device), 1 if never_completes else 0,
                                                  _stream(stream)))


def idx_topk_set_timing(enable: bool) -> None:
    _lib.load().idx_topk_set_timing(1 if enable else 0)


def idx_topk_last_timings() -> dict:
    """Kernel-phase times (ms) of this thread's last call, when timing is on."""
    buf = (ctypes.c_float * 4)()
    _lib.load().idx_topk_last_timings(buf)
    return {"plan_ms": buf[0], "score_ms": buf[1], "finish_ms": buf[2], "kernels_ms": buf[3]}


def dense_score_bytes(rows: int, context: int) -> int:
    """Bytes of the materialised fp32 [rows, context] score matrix of the dense path."""
    return int(rows) * int(context) * 4
