"""The allocation-free entry point (scratch in the library's fixed per-device
buffer) against the allocating one: two calls in a row on different problems
give bit-identical outputs, and a problem larger than the fixed buffer is
refused with IDX_ERR_SCRATCH_LIMIT and -1 outputs, and concurrent calls from
several host threads each get their own correct result."""
import numpy as np
import pytest

from fp4_sparse_attention_tma_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 9


def _both(p, d):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    out = []
    for fn in (m.idx_topk_fp4_prefill, m.idx_topk_fp4_prefill_noalloc):
        phys = torch.full((p.rows, p.topk), 7, dtype=torch.int32, device="cuda")
        raw = torch.full((p.rows, p.topk), 7, dtype=torch.int32, device="cuda")
        code = fn(**d, topk=p.topk, out_phys_slot=phys, out_raw_idx=raw, raise_on_error=False)
        torch.cuda.synchronize()
        out.append((code, phys.cpu().numpy(), raw.cpu().numpy()))
    return out


def test_noalloc_matches_allocating_entry_two_calls():
    # two different problems back to back: the second call reuses the buffer
    # the first one left behind
    probs = [inputs.config(1), inputs.small_problem(seed=11, topk=1024)]
    for p in probs:
        (c0, phys0, raw0), (c1, phys1, raw1) = _both(p, H.to_device(p))
        assert c0 == 0 and c1 == 0
        np.testing.assert_array_equal(raw1, raw0)
        np.testing.assert_array_equal(phys1, phys0)


def test_noalloc_repeat_same_problem():
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    p = inputs.config(4)
    d = H.to_device(p)
    res = []
    for _ in range(2):
        raw = torch.zeros((p.rows, p.topk), dtype=torch.int32, device="cuda")
        phys = torch.zeros((p.rows, p.topk), dtype=torch.int32, device="cuda")
        assert m.idx_topk_fp4_prefill_noalloc(**d, topk=p.topk, out_phys_slot=phys,
                                              out_raw_idx=raw) == 0
        res.append(raw.cpu().numpy())
    np.testing.assert_array_equal(res[0], res[1])
    code, _, raw_ref = H.run_fused(p, d)
    assert code == 0
    np.testing.assert_array_equal(res[0], raw_ref)


def test_noalloc_refuses_problem_beyond_buffer():
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    # 8192 rows at topk 1024 need ~82 MB of candidate scratch (> 48 MiB); the
    # windows themselves are short, so the allocating path handles it quickly
    rows = 8192
    p = inputs.make_problem(23, [2048], [[(0, 2048)] * rows], topk=1024)
    need = m.idx_topk_fp4_scratch_bytes(rows, 1024)
    assert need > 48 * 1024 * 1024
    d = H.to_device(p)
    phys = torch.zeros((rows, 1024), dtype=torch.int32, device="cuda")
    raw = torch.zeros((rows, 1024), dtype=torch.int32, device="cuda")
    code = m.idx_topk_fp4_prefill_noalloc(**d, topk=1024, out_phys_slot=phys, out_raw_idx=raw,
                                          raise_on_error=False)
    torch.cuda.synchronize()
    assert code == SCRATCH_LIMIT
    assert (phys.cpu().numpy() == -1).all() and (raw.cpu().numpy() == -1).all()


def test_noalloc_concurrent_host_threads():
    # several host threads, each on its own stream and problem, call the
    # allocation-free entry at once: the per-device lock keeps them off each
    # other's scratch, so every result equals the allocating call's
    import threading
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    probs = [inputs.small_problem(seed=40 + i, topk=(512, 1024)[i % 2]) for i in range(4)]
    devs = [H.to_device(p) for p in probs]
    want = []
    for p, d in zip(probs, devs):
        code, _, raw_ref = H.run_fused(p, d)
        assert code == 0
        want.append(raw_ref)
    got = [[] for _ in probs]
    errors = []

    def worker(i):
        try:
            p, d = probs[i], devs[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(3):
                    raw = torch.full((p.rows, p.topk), 7, dtype=torch.int32, device="cuda")
                    phys = torch.full((p.rows, p.topk), 7, dtype=torch.int32, device="cuda")
                    code = m.idx_topk_fp4_prefill_noalloc(**d, topk=p.topk, out_phys_slot=phys,
                                                          out_raw_idx=raw, raise_on_error=False)
                    s.synchronize()
                    got[i].append((code, raw.cpu().numpy()))
        except Exception as e:  # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(probs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(len(probs)):
        assert len(got[i]) == 3
        for code, raw in got[i]:
            assert code == 0
            np.testing.assert_array_equal(raw, want[i])
