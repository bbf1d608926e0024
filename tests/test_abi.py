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


def test_range_checked_build_exports_the_same_symbols():
    # the -DIDX_DEBUG_BOUNDS variant that the GPU tests run on small cases
    lib = _lib.load(_lib.build(debug_bounds=True))
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.idx_topk_fp4_prefill(*([None] * 9), 512, None, None, None) == 1


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


def test_header_is_plain_c_and_links(tmp_path):
    """include/idxtopk.h compiles as strict C99 and a C program linked against the
    in-tree library calls the host-only entry points through it."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    lib_path = _lib.build()
    src = tmp_path / "abi_c.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "idxtopk.h"

int main(void) {
  const int32_t* ks = NULL;
  int32_t n = 0;
  if (idx_topk_supported_k(&ks, &n) != IDX_OK || n != 2 || ks[0] != 512 || ks[1] != 1024)
    return 1;
  if (strcmp(idx_topk_status_string(IDX_OK), idx_topk_status_string(IDX_ERR_INVALID_PAGE)) == 0)
    return 2;
  /* a null output descriptor fails before any device work */
  if (idx_topk_fp4_prefill(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 512, NULL, NULL,
                           (idx_stream_t)0) != IDX_ERR_INVALID_ARGUMENT)
    return 3;
  idx_tensor_t t;
  memset(&t, 0, sizeof(t));
  t.dtype = IDX_I32;
  printf("ok %d %zu\n", (int)n, sizeof(t));
  return 0;
}
''')
    exe = tmp_path / "abi_c"
    lib_dir = os.path.dirname(lib_path)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", lib_dir, "-l:" + os.path.basename(lib_path),
                        "-Wl,-rpath," + lib_dir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.split()[:2] == ["ok", "2"]


def test_every_declaration_cites_its_passage():
    """Each entry point's comment cites the passage that defines it, or says that
    the pages have no counterpart."""
    text = open(HEADER).read()
    for m in re.finditer(r"^(?:int|const char\*)\s+(idx_\w+)\s*\(", text, re.M):
        before = text[:m.start()]
        j = before.rfind("/*")
        comment = re.sub(r"\s*\n\s*\*\s?", " ", before[j:before.rfind("*/")])
        assert re.search(r"aiter#\d+|sglang#\d+|no counterpart on the pages", comment), m.group(1)


def test_packed_descriptors_match_the_struct_layout():
    """The binding packs idx_tensor_t descriptors into one buffer per call: the
    bytes must be those of the ctypes struct (data, dtype, ndim, shape[4],
    stride[4]) for every tensor shape the entry points take."""
    import ctypes
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    ts = [torch.zeros((7, 64, 64), dtype=torch.uint8), torch.zeros(5, dtype=torch.int32),
          torch.zeros((3, 4), dtype=torch.float32)[:, ::2], torch.zeros(0, dtype=torch.int32),
          torch.zeros((2, 3, 4, 5), dtype=torch.float32), torch.zeros((2, 3, 4, 5, 6)),
          torch.zeros((6, 2), dtype=torch.float64), None]
    buf, addrs = m._descs(ts)
    assert ctypes.sizeof(_lib.IdxTensor) == m._DESC.size == 80
    for i, t in enumerate(ts):
        if t is None:
            assert addrs[i] is None
            continue
        assert addrs[i] == ctypes.addressof(buf) + 80 * i
        want = bytes(m._desc(t))
        got = ctypes.string_at(addrs[i], 80)
        assert got == want, (i, tuple(t.shape))
