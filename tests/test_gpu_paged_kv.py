"""The page-interleaved K cache entry point: each physical page's codes
followed by its scales in one 4352-byte record.  Its outputs are compared with
the oracle (every row of the small cases, sampled rows of the 1024-row
workloads) and, built from the same data as the two-tensor layout, must equal
that layout's outputs; the record width is checked on the host."""
import numpy as np
import pytest

from fp4_sparse_attention_tma_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu

UNSUPPORTED = 2


def _interleave(p):
    npg = p.k_cache_fp4.shape[0]
    return np.ascontiguousarray(np.concatenate(
        [p.k_cache_fp4.reshape(npg, 4096), p.k_scale.reshape(npg, 256)], axis=1))


def _paged_call(p, d, k_pages, K=None, raise_on_error=True):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    K = int(K or p.topk)
    phys = torch.full((p.rows, K), 7, dtype=torch.int32, device="cuda")
    raw = torch.full((p.rows, K), 7, dtype=torch.int32, device="cuda")
    args = {k: v for k, v in d.items() if k not in ("k_cache_fp4", "k_scale")}
    code = m.idx_topk_fp4_prefill_paged(**args, k_pages=k_pages, topk=K, out_phys_slot=phys,
                                        out_raw_idx=raw, raise_on_error=raise_on_error)
    torch.cuda.synchronize()
    return code, phys.cpu().numpy(), raw.cpu().numpy()


@pytest.mark.parametrize("which", ["small512", "small1024", "config1", "config4"])
def test_paged_matches_oracle_and_two_tensor_layout(which):
    import torch
    p = {"small512": lambda: inputs.small_problem(seed=21, topk=512),
         "small1024": lambda: inputs.small_problem(seed=22, topk=1024),
         "config1": lambda: inputs.config(1),
         "config4": lambda: inputs.config(4)}[which]()
    d = H.to_device(p)
    kp = torch.from_numpy(_interleave(p)).cuda()
    code, phys, raw = _paged_call(p, d, kp)
    assert code == 0
    rows = None if p.rows <= 64 else H.sample_rows(p, total=12, seed=5)
    H.check_against_oracle(p, phys, raw, rows)
    code2, want_phys, want_raw = H.run_fused(p, d)
    assert code2 == 0
    np.testing.assert_array_equal(raw, want_raw)
    np.testing.assert_array_equal(phys, want_phys)


def test_paged_record_width_checked():
    import torch
    p = inputs.small_problem(seed=23, topk=512)
    d = H.to_device(p)
    kp = torch.from_numpy(np.ascontiguousarray(_interleave(p)[:, :4096 + 128])).cuda()
    code, phys, raw = _paged_call(p, d, kp, raise_on_error=False)
    assert code == UNSUPPORTED
    assert (phys == -1).all() and (raw == -1).all()
