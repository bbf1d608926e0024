"""idx_topk_fp4_prefill_host through the C ABI on the GPU: host (pinned or
pageable) inputs and outputs give the same results as the device entry point
on the same data, and every error leaves -1 in the host outputs."""
import numpy as np
import pytest

from fp4_sparse_attention_tma_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _host(p, pinned=True):
    import torch
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    d = dict(q_fp4=f(p.q_fp4), q_scale=f(p.q_scale), k_cache_fp4=f(p.k_cache_fp4),
             k_scale=f(p.k_scale), weights=f(p.weights), page_table=f(p.page_table),
             row_req=f(p.row_req), row_start=f(p.row_start), row_end=f(p.row_end))
    return {k: (v.pin_memory() if pinned else v.clone()) for k, v in d.items()}


def _call_host(p, d, pinned=True, raw=True):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    mk = lambda: torch.zeros((p.rows, p.topk), dtype=torch.int32)
    phys = mk().pin_memory() if pinned else mk()
    rawt = (mk().pin_memory() if pinned else mk()) if raw else None
    code = m.idx_topk_fp4_prefill_host(**d, topk=p.topk, out_phys_slot=phys, out_raw_idx=rawt,
                                       device=0, raise_on_error=False)
    return code, phys.numpy(), (rawt.numpy() if raw else None)


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("prob", ["config0", "small"])
def test_host_call_equals_device_call(prob, pinned):
    p = inputs.config(0) if prob == "config0" else inputs.small_problem(seed=23)
    code_d, phys_d, raw_d = H.run_fused(p)
    assert code_d == 0
    code, phys, raw = _call_host(p, _host(p, pinned), pinned=pinned)
    assert code == 0
    assert np.array_equal(phys, phys_d) and np.array_equal(raw, raw_d)


def test_host_call_without_raw_output():
    p = inputs.small_problem(seed=5)
    _, phys_d, _ = H.run_fused(p)
    code, phys, _ = _call_host(p, _host(p), raw=False)
    assert code == 0 and np.array_equal(phys, phys_d)


def test_host_call_repeats_on_one_stream():
    p = inputs.small_problem(seed=8)
    d = _host(p)
    first = _call_host(p, d)
    for _ in range(3):
        again = _call_host(p, d)
        assert again[0] == 0
        assert np.array_equal(again[1], first[1]) and np.array_equal(again[2], first[2])


def test_host_call_invalid_metadata_fails_closed():
    p = inputs.small_problem(seed=9)
    d = _host(p)
    d["row_end"][2] = int(p.page_table.shape[1]) * 64 + 5   # beyond the request's pages
    code, phys, raw = _call_host(p, d)
    assert code == 3
    assert np.all(phys == -1) and np.all(raw == -1)


def test_host_call_invalid_page_fails_closed():
    p = inputs.small_problem(seed=10)
    d = _host(p)
    d["page_table"][0, 0] = p.num_pages + 3
    code, phys, raw = _call_host(p, d)
    assert code == 4
    assert np.all(phys == -1) and np.all(raw == -1)


def test_host_call_rejects_device_tensors():
    p = inputs.small_problem(seed=11)
    d = _host(p)
    d["weights"] = d["weights"].cuda()
    code, phys, raw = _call_host(p, d)
    assert code == 1
    assert np.all(phys == -1) and np.all(raw == -1)


def test_host_call_unsupported_topk_and_bad_device():
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    p = inputs.small_problem(seed=12)
    d = _host(p)
    for K, dev, want in ((256, 0, 2), (p.topk, torch.cuda.device_count() + 4, 1)):
        phys = torch.zeros((p.rows, K), dtype=torch.int32)
        code = m.idx_topk_fp4_prefill_host(**d, topk=K, out_phys_slot=phys, device=dev,
                                           stream=torch.cuda.current_stream(0),
                                           raise_on_error=False)
        assert code == want
        assert np.all(phys.numpy() == -1)
