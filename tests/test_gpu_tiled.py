"""The context-tiled comparison path against the oracle (every row of the small
cases, sampled rows of the 1024-row workloads) and against the fused path
(identical outputs: same scoring arithmetic, same order keys), for several
chunk widths including ones that split pages' worth of positions across chunks
and chunks no row reaches; bad chunk widths are refused."""
import numpy as np
import pytest

from fp4_sparse_attention_tma_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _tiled(p, d, tile, raise_on_error=True):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    phys = torch.full((p.rows, p.topk), 7, dtype=torch.int32, device="cuda")
    raw = torch.full((p.rows, p.topk), 7, dtype=torch.int32, device="cuda")
    code = m.idx_tiled_topk_fp4_prefill(**d, topk=p.topk, out_phys_slot=phys, out_raw_idx=raw,
                                        context_tile=tile, raise_on_error=raise_on_error)
    torch.cuda.synchronize()
    return code, phys.cpu().numpy(), raw.cpu().numpy()


@pytest.mark.parametrize("which,tile", [("small512", 1024), ("small1024", 1152),
                                        ("config1", 4096), ("config1", 65536), ("config4", 16384)])
def test_tiled_matches_oracle_and_fused(which, tile):
    p = {"small512": lambda: inputs.small_problem(seed=31, topk=512),
         "small1024": lambda: inputs.small_problem(seed=32, topk=1024),
         "config1": lambda: inputs.config(1),
         "config4": lambda: inputs.config(4)}[which]()
    d = H.to_device(p)
    code, phys, raw = _tiled(p, d, tile)
    assert code == 0
    rows = None if p.rows <= 64 else H.sample_rows(p, total=12, seed=tile)
    H.check_against_oracle(p, phys, raw, rows)
    code2, want_phys, want_raw = H.run_fused(p, d)
    assert code2 == 0
    np.testing.assert_array_equal(raw, want_raw)
    np.testing.assert_array_equal(phys, want_phys)


@pytest.mark.parametrize("tile", [0, 1000, 1030])
def test_tiled_bad_chunk_width(tile):
    p = inputs.small_problem(seed=33, topk=512)
    code, phys, raw = _tiled(p, H.to_device(p), tile, raise_on_error=False)
    assert code == 1
    assert (phys == -1).all() and (raw == -1).all()
