"""Fail-closed contract through the C ABI on the GPU: every error returns its
code and leaves -1 in valid outputs; graph capture is rejected without
enqueueing work; calls run on the caller's stream; scratch does not depend on
the context length.  Faults are injected on the host by corrupting metadata
or descriptors -- no case makes the device fault."""
import ctypes

import numpy as np
import pytest

from fp4_sparse_attention_tma_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def base():
    return inputs.make_problem(51, [2000, 900], [[(0, 2000), (0, 1999), (40, 1500)],
                                                 [(0, 900), (0, 800)]], topk=512)


def _call(p, d, K=512, **kw):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    phys = torch.zeros((p.rows, K), dtype=torch.int32, device="cuda")
    raw = torch.zeros((p.rows, K), dtype=torch.int32, device="cuda")
    code = m.idx_topk_fp4_prefill(**d, topk=K, out_phys_slot=phys, out_raw_idx=raw,
                                  raise_on_error=False, **kw)
    torch.cuda.synchronize()
    return code, phys.cpu().numpy(), raw.cpu().numpy()


def test_ok_baseline(base):
    code, phys, raw = _call(base, H.to_device(base))
    assert code == 0 and (raw >= 0).any()


@pytest.mark.parametrize("K", [1, 256, 511, 2048])
def test_unsupported_topk(base, K):
    code, phys, raw = _call(base, H.to_device(base), K=K)
    assert code == 2
    assert np.all(phys == -1) and np.all(raw == -1)


def test_invalid_page_entry(base):
    d = H.to_device(base)
    d["page_table"][0, 5] = base.num_pages + 7
    code, phys, raw = _call(base, d)
    assert code == 4 and np.all(phys == -1) and np.all(raw == -1)
    d = H.to_device(base)
    d["page_table"][1, 3] = -1
    assert _call(base, d)[0] == 4


@pytest.fixture(scope="module")
def short_rows():
    # request 0 has only rows of at most topk positions (not scored: every
    # position is emitted and mapped through the page table); request 1 a
    # scored row
    return inputs.make_problem(53, [700, 3000], [[(0, 300), (100, 612)], [(0, 3000)]], topk=512)


@pytest.mark.parametrize("page,expect", [(0, 4), (2, 4), (9, 4), (10, 0), (20, 0)])
def test_page_check_covers_unscored_rows(short_rows, page, expect):
    """An entry under a row that is not scored is checked where the finishing
    step maps the row's positions: pages 0..9 lie under request 0's windows
    [0, 300) and [100, 612); page 10 and later do not and are never read."""
    p = short_rows
    for bad in (-1, p.num_pages):
        d = H.to_device(p)
        d["page_table"][0, page] = bad
        code, phys, raw = _call(p, d)
        assert code == expect
        if expect:
            assert np.all(phys == -1) and np.all(raw == -1)


def test_page_check_unscored_rows_stream_ordered(short_rows):
    """The stream-ordered call publishes the same status from the finishing
    kernel's last CTA, with -1 outputs."""
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    p = short_rows
    d = H.to_device(p)
    d["page_table"][0, 4] = p.num_pages + 3
    ws = torch.empty(m.idx_topk_fp4_scratch_bytes(p.rows, 512), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    phys = torch.full((p.rows, 512), 7, dtype=torch.int32, device="cuda")
    raw = torch.full((p.rows, 512), 7, dtype=torch.int32, device="cuda")
    assert m.idx_topk_fp4_prefill_async(**d, topk=512, out_phys_slot=phys, out_raw_idx=raw,
                                        workspace=ws, status=st, raise_on_error=False) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 4
    assert (phys.cpu().numpy() == -1).all() and (raw.cpu().numpy() == -1).all()
    d = H.to_device(p)
    assert m.idx_topk_fp4_prefill_async(**d, topk=512, out_phys_slot=phys, out_raw_idx=raw,
                                        workspace=ws, status=st, raise_on_error=False) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    code, want_phys, want_raw = _call(p, d)
    assert code == 0
    np.testing.assert_array_equal(phys.cpu().numpy(), want_phys)
    np.testing.assert_array_equal(raw.cpu().numpy(), want_raw)


def test_page_check_tiled_path(short_rows):
    """The context-tiled path checks the entries it maps as well: under the
    unscored rows (its last chunk's closed form) and under the scored row."""
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    p = short_rows
    for req, page in ((0, 3), (1, 30)):
        d = H.to_device(p)
        d["page_table"][req, page] = -2
        phys = torch.zeros((p.rows, 512), dtype=torch.int32, device="cuda")
        raw = torch.zeros((p.rows, 512), dtype=torch.int32, device="cuda")
        code = m.idx_tiled_topk_fp4_prefill(**d, topk=512, out_phys_slot=phys, out_raw_idx=raw,
                                            context_tile=1024, raise_on_error=False)
        torch.cuda.synchronize()
        assert code == 4, (req, page)
        assert (phys.cpu().numpy() == -1).all()


def test_page_entries_outside_windows_are_not_read(base):
    d = H.to_device(base)
    # request 1's windows end at 900 -> logical pages >= 15 are never covered
    d["page_table"][1, 20:] = 123456789
    code, _, _ = _call(base, d)
    assert code == 0


@pytest.mark.parametrize("page,expect", [(900, 4), (937, 4), (938, 0), (1020, 0)])
def test_page_check_covers_long_windows(page, expect):
    # one row whose window [0, 60000) spans logical pages 0..937 of a
    # 1024-page request: an invalid entry anywhere under it fails the call
    # closed; entries past the window's last page are never read
    p = inputs.make_problem(52, [65536, 64], [[(0, 60000)], [(0, 64)]], topk=512)
    d = H.to_device(p)
    d["page_table"][0, page] = -5 if expect else 987654321
    code, phys, raw = _call(p, d)
    assert code == expect
    if expect:
        assert np.all(phys == -1) and np.all(raw == -1)
    else:
        assert (raw[0] >= 0).all()


@pytest.mark.parametrize("field,value,row", [("row_req", 5, 1), ("row_req", -1, 0),
                                             ("row_start", -3, 2), ("row_end", 10**6, 0),
                                             ("row_start", 1600, 2)])
def test_invalid_metadata(base, field, value, row):
    d = H.to_device(base)
    d[field][row] = value
    code, phys, raw = _call(base, d)
    assert code == 3 and np.all(phys == -1) and np.all(raw == -1)


def test_misaligned_and_noncontiguous(base):
    import torch
    d = H.to_device(base)
    buf = torch.zeros(d["weights"].numel() + 1, dtype=torch.float32, device="cuda")
    d["weights"] = buf[1:].view(base.rows, 64)           # 4-byte offset: not 16-byte aligned
    assert _call(base, d)[0] == 1
    d = H.to_device(base)
    d["weights"] = torch.zeros((64, base.rows), device="cuda").t()   # non-contiguous
    assert _call(base, d)[0] == 1
    d = H.to_device(base)
    d["weights"] = d["weights"].double()                 # wrong dtype
    assert _call(base, d)[0] == 1


def test_unsupported_shapes(base):
    import torch
    d = H.to_device(base)
    d["q_fp4"] = torch.zeros((base.rows, 32, 64), dtype=torch.uint8, device="cuda")
    assert _call(base, d)[0] == 2


def test_overflow_descriptor_rejected(base):
    """A K cache whose slot count exceeds int32 is refused before any access."""
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    from fp4_sparse_attention_tma_gb300 import _lib
    d = H.to_device(base)
    lib = _lib.load()
    descs = {k: m._desc(v) for k, v in d.items()}
    big = descs["k_cache_fp4"]
    big.shape[0] = (1 << 25) + 1          # (2^25 + 1) * 64 slots > INT32_MAX
    ks = descs["k_scale"]
    ks.shape[0] = big.shape[0]
    phys = torch.zeros((base.rows, 512), dtype=torch.int32, device="cuda")
    order = ["q_fp4", "q_scale", "k_cache_fp4", "k_scale", "weights", "page_table", "row_req",
             "row_start", "row_end"]
    phys_d = m._desc(phys)
    code = lib.idx_topk_fp4_prefill(*[ctypes.addressof(descs[k]) for k in order], 512,
                                    ctypes.addressof(phys_d), None,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert code == 5
    assert np.all(phys.cpu().numpy() == -1)


def test_graph_capture_rejected(base):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    d = H.to_device(base)
    phys = torch.full((base.rows, 512), 7, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    codes = []
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            codes.append(m.idx_topk_fp4_prefill(**d, topk=512, out_phys_slot=phys,
                                                raise_on_error=False))
    torch.cuda.synchronize()
    assert codes == [2]
    assert np.all(phys.cpu().numpy() == 7)      # nothing was enqueued


def test_runs_on_caller_stream(base):
    import torch
    d = H.to_device(base)
    s = torch.cuda.Stream()
    _, want_phys, want_raw = _call(base, d)
    with torch.cuda.stream(s):
        code, phys, raw = _call(base, d)
    assert code == 0 and np.array_equal(phys, want_phys) and np.array_equal(raw, want_raw)


def test_scratch_is_context_independent():
    # the workspace the query reports for (rows, topk) -- it takes no context
    # argument -- serves the stream-ordered call at contexts 16x apart
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    rows, K = 48, 512
    need = m.idx_topk_fp4_scratch_bytes(rows, K)
    assert 0 < m.idx_topk_fp4_scratch_bytes(8, K) < need
    for L in (4096, 65536):
        p = inputs.make_problem(53, [L], [[(0, L - rows + 1 + i) for i in range(rows)]], topk=K)
        d = H.to_device(p)
        _, want_phys, want_raw = _call(p, d, K)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        phys = torch.zeros((rows, K), dtype=torch.int32, device="cuda")
        raw = torch.zeros((rows, K), dtype=torch.int32, device="cuda")
        code = m.idx_topk_fp4_prefill_async(**d, topk=K, out_phys_slot=phys, out_raw_idx=raw,
                                            workspace=ws, status=st)
        torch.cuda.synchronize()
        assert code == 0 and int(st.item()) == 0
        assert np.array_equal(phys.cpu().numpy(), want_phys)
        assert np.array_equal(raw.cpu().numpy(), want_raw)


def test_repeated_calls_are_deterministic(base):
    d = H.to_device(base)
    r1 = _call(base, d)
    r2 = _call(base, d)
    assert np.array_equal(r1[1], r2[1]) and np.array_equal(r1[2], r2[2])


def test_expired_device_wait_returns_a_status_and_the_context_stays_usable(base):
    # a bounded mbarrier wait on a phase that nothing completes gives up after
    # its 2 s limit and the kernel records IDX_ERR_TIMEOUT instead of hanging;
    # the same wait completes normally when the phase is completed, and a
    # regular call afterwards still succeeds on the same context
    import time
    import fp4_sparse_attention_tma_gb300 as m
    assert m.idx_debug_bounded_wait(False) == 0
    t0 = time.perf_counter()
    assert m.idx_debug_bounded_wait(True) == 8
    assert 1.9 < time.perf_counter() - t0 < 60
    assert m.idx_debug_bounded_wait(False) == 0
    code, _, raw = _call(base, H.to_device(base))
    assert code == 0 and (raw >= 0).any()
