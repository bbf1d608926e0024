"""CPU checks of the C-ABI library: it builds for sm_103a, loads without a GPU,
exports every function that include/idxtopk.h declares, and answers the
host-only queries.  No compute call is made here."""
import ctypes
import os
import re

import numpy as np
import pytest

from fp4_sparse_attention_tma_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "idxtopk.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(idx_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    fns = declared_functions()
    for name in ("idx_topk_fp4_prefill", "idx_topk_supported_k", "idx_topk_status_string",
                 "idx_topk_fp4_scratch_bytes", "idx_fp4_debug_scores", "idx_topk_select_scores",
                 "idx_dense_topk_fp4_prefill", "idx_topk_scratch_high_water"):
        assert name in fns


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and the binding declares a signature for each
    assert set(declared_functions()) <= set(_lib.EXPORTS)


def test_supported_k_and_status_strings():
    import fp4_sparse_attention_tma_gb300 as m
    assert m.idx_topk_supported_k() == (512, 1024)
    assert m.SUPPORTED_K == (512, 1024)
    for code, name in m.STATUS.items():
        s = m.idx_topk_status_string(code)
        assert isinstance(s, str) and s
    assert m.idx_topk_status_string(99) == "unknown status"


def test_null_output_descriptor_is_rejected_before_any_device_work():
    lib = _lib.load()
    code = lib.idx_topk_fp4_prefill(*([None] * 9), 512, None, None, None)
    assert code == 1  # IDX_ERR_INVALID_ARGUMENT


def test_supported_k_null_args():
    lib = _lib.load()
    assert lib.idx_topk_supported_k(None, None) == 1


def test_binding_has_no_cpu_fallback(monkeypatch):
    """A missing library must raise, not compute elsewhere."""
    import fp4_sparse_attention_tma_gb300 as m
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "build", lambda *a, **k: "/nonexistent/libidxtopk.so")
    with pytest.raises(OSError):
        m.idx_topk_supported_k()


def test_pages_memory_geometry():
    """The dense path's fp32 score storage reproduces the pages' arithmetic."""
    import fp4_sparse_attention_tma_gb300 as m
    path = os.path.join(ROOT, "tests", "golden", "memory_geometry.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    for r, ctx, mib in rows:
        assert m.dense_score_bytes(int(r), int(ctx)) / 2**20 == pytest.approx(float(mib))
