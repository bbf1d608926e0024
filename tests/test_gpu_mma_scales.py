"""The K-scale input in the block-scaled MMA's scale-copy order
(idx_topk_fp4_prefill_mma_scales; the pre-shuffled scale input that "[FlyDSL]
[DSv4] Prototype FP4 MQA streaming TopK", Scope, names as a consumer layout).
Built from the same data, it gives the outputs of the row-major layout bit for
bit, and they match the oracle (every row of the small cases, sampled rows of
the 1024-row workloads); the tensor's shape is checked on the host and the
value domain on the device."""
import numpy as np
import pytest

from fp4_sparse_attention_tma_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu

INVALID_ARGUMENT, INVALID_VALUE = 1, 10


def _call(p, d, k_scale_mma, raise_on_error=True):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    phys = torch.full((p.rows, p.topk), 7, dtype=torch.int32, device="cuda")
    raw = torch.full((p.rows, p.topk), 7, dtype=torch.int32, device="cuda")
    args = {k: v for k, v in d.items() if k != "k_scale"}
    code = m.idx_topk_fp4_prefill_mma_scales(**args, k_scale_mma=k_scale_mma, topk=p.topk,
                                             out_phys_slot=phys, out_raw_idx=raw,
                                             raise_on_error=raise_on_error)
    torch.cuda.synchronize()
    return code, phys.cpu().numpy(), raw.cpu().numpy()


@pytest.mark.parametrize("which", ["small512", "small1024", "config1", "config4"])
def test_mma_order_matches_oracle_and_row_major(which):
    import torch
    p = {"small512": lambda: inputs.small_problem(seed=61, topk=512),
         "small1024": lambda: inputs.small_problem(seed=62, topk=1024),
         "config1": lambda: inputs.config(1),
         "config4": lambda: inputs.config(4)}[which]()
    d = H.to_device(p)
    ksm = torch.from_numpy(inputs.k_scale_mma_order(p.k_scale)).cuda()
    code, phys, raw = _call(p, d, ksm)
    assert code == 0
    rows = None if p.rows <= 64 else H.sample_rows(p, total=12, seed=9)
    H.check_against_oracle(p, phys, raw, rows)
    code2, want_phys, want_raw = H.run_fused(p, d)
    assert code2 == 0
    np.testing.assert_array_equal(raw, want_raw)
    np.testing.assert_array_equal(phys, want_phys)


def test_mma_order_shape_and_domain_checked():
    import torch
    p = inputs.small_problem(seed=63, topk=512)
    d = H.to_device(p)
    code, phys, raw = _call(p, d, d["k_scale"], raise_on_error=False)   # [NP, 64, 4]
    assert code == INVALID_ARGUMENT and (phys == -1).all() and (raw == -1).all()
    ksm = torch.from_numpy(inputs.k_scale_mma_order(p.k_scale)).cuda()
    code, _, _ = _call(p, d, ksm[:, :128].contiguous(), raise_on_error=False)
    assert code == INVALID_ARGUMENT
    page = int(p.page_table[0, 10])      # positions 640..703: under request 0's windows
    ksm[page, 8 * 5 + 4 * 1 + 2] = 255   # slot 37, scale block 2
    code, phys, _ = _call(p, d, ksm, raise_on_error=False)
    assert code == INVALID_VALUE and (phys == -1).all()
