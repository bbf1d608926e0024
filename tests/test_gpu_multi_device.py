"""Device guard with more than one GPU ("[FlyDSL] Add FP4 LiteTopK prefill
operator", Validation: a non-current device): tensors and stream on device 1
while device 0 is current -- the call runs on device 1, returns the outputs of
the same call made with device 1 current, and leaves device 0 current; a stream
of the other device is refused.  Skipped where fewer than two GPUs are visible
(this run has one)."""
import numpy as np
import pytest

from fp4_sparse_attention_tma_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _two_gpus():
    import torch
    return torch.cuda.is_available() and torch.cuda.device_count() >= 2


@pytest.mark.skipif(not _two_gpus(), reason="needs two GPUs")
def test_tensors_on_a_non_current_device():
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    p = inputs.small_problem(seed=71, topk=512)
    d1 = H.to_device(p, device="cuda:1")
    phys = torch.zeros((p.rows, p.topk), dtype=torch.int32, device="cuda:1")
    raw = torch.zeros_like(phys)
    torch.cuda.set_device(0)
    s1 = torch.cuda.Stream(device=1)
    assert m.idx_topk_fp4_prefill(**d1, topk=p.topk, out_phys_slot=phys, out_raw_idx=raw,
                                  stream=s1) == 0
    s1.synchronize()
    assert torch.cuda.current_device() == 0
    with torch.cuda.device(1):
        code, want_phys, want_raw = H.run_fused(p, d1)
    assert code == 0
    np.testing.assert_array_equal(raw.cpu().numpy(), want_raw)
    np.testing.assert_array_equal(phys.cpu().numpy(), want_phys)
    # a stream of device 0 with tensors of device 1 is refused, outputs -1
    s0 = torch.cuda.Stream(device=0)
    code = m.idx_topk_fp4_prefill(**d1, topk=p.topk, out_phys_slot=phys, out_raw_idx=raw,
                                  stream=s0, raise_on_error=False)
    assert code == 1
    assert torch.cuda.current_device() == 0
