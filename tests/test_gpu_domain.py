"""Accepted value domain through the C ABI on the GPU: a UE8M0 scale byte above
167 (the NaN byte 255 included) in a query block the scorer reads or in a K
page under a scored window, or a weight of a scored row that is not finite or
exceeds 2^24 in magnitude, fails the call closed with IDX_ERR_INVALID_VALUE and
-1 outputs ("[FlyDSL] Add FP4 LiteTopK prefill operator", Implementation: fail
closed rather than produce nonfinite scores).  Bytes the scorer never reads are
not checked, and values at the edge of the domain are scored like any other
(compared with the oracle).  The bad values are planted on the host."""
import numpy as np
import pytest

import oracle
from fp4_sparse_attention_tma_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu

INVALID_VALUE = 10


def _problem():
    # request 0 holds 2400 positions but no window reaches past 2000, so its
    # logical pages 32..37 are never read; row 1 (300 positions) is short
    return inputs.make_problem(61, [2400, 1000],
                               [[(0, 2000), (0, 300), (64, 1800)], [(0, 900), (0, 1000)]],
                               topk=512)


@pytest.fixture(scope="module")
def base():
    p = _problem()
    code, phys, raw = H.run_fused(p)
    assert code == 0
    return p, phys, raw


def _fails_closed(p, d):
    code, phys, raw = H.run_fused(p, d, raise_on_error=False)
    assert code == INVALID_VALUE
    assert np.all(phys == -1) and np.all(raw == -1)


@pytest.mark.parametrize("byte", [255, 168, 200])
def test_query_scale_byte_above_domain(byte):
    p = _problem()
    d = H.to_device(p)
    d["q_scale"][0, 37, 2] = byte          # row 0 is scored
    _fails_closed(p, d)


@pytest.mark.parametrize("byte", [255, 168])
def test_k_scale_byte_above_domain_under_window(byte):
    p = _problem()
    d = H.to_device(p)
    page = int(p.page_table[1, 7])         # request 1, positions 448..511: under its windows
    d["k_scale"][page, 11, 3] = byte
    _fails_closed(p, d)


@pytest.mark.parametrize("value", [float("nan"), float("inf"), -float("inf"),
                                   float(np.nextafter(np.float32(2.0 ** 24), np.float32(np.inf))),
                                   -3.0e30])
def test_weight_outside_domain(value):
    p = _problem()
    d = H.to_device(p)
    d["weights"][2, 63] = value            # row 2 is scored
    _fails_closed(p, d)


def test_dense_path_checks_the_domain_too():
    import fp4_sparse_attention_tma_gb300 as m
    import torch
    p = _problem()
    d = H.to_device(p)
    d["q_scale"][3, 0, 0] = 255
    phys = torch.zeros((p.rows, p.topk), dtype=torch.int32, device="cuda")
    code = m.idx_dense_topk_fp4_prefill(**d, topk=p.topk, out_phys_slot=phys,
                                        raise_on_error=False)
    torch.cuda.synchronize()
    assert code == INVALID_VALUE and bool((phys == -1).all())


def test_bytes_that_are_never_read_are_not_checked(base):
    p, phys0, raw0 = base
    d = H.to_device(p)
    unread = int(p.page_table[0, 34])      # request 0, positions 2176..2239: past every window
    d["k_scale"][unread] = 255
    d["q_scale"][1] = 255                  # row 1 is short (300 <= 512): never scored
    d["weights"][1] = float("nan")
    code, phys, raw = H.run_fused(p, d, raise_on_error=False)
    assert code == 0
    np.testing.assert_array_equal(phys, phys0)
    np.testing.assert_array_equal(raw, raw0)


def test_edge_of_domain_matches_oracle():
    # every exponent shifted up by 36 (bytes 159..167, the largest accepted is
    # 167) and weights of magnitude up to exactly 2^24: logits near 2^85,
    # scores near 2^110, all finite; compared with the oracle as usual
    p = _problem()
    p.q_scale = (p.q_scale.astype(np.int32) + 36).astype(np.uint8)
    p.k_scale = (p.k_scale.astype(np.int32) + 36).astype(np.uint8)
    assert p.q_scale.max() <= 167 and p.k_scale.max() <= 167
    p.weights = (p.weights * np.float32(2.0 ** 21)).astype(np.float32)
    p.weights[:, 0] = np.float32(2.0 ** 24)
    p.weights[:, 1] = np.float32(-(2.0 ** 24))
    code, g_phys, g_raw = H.run_fused(p, raise_on_error=False)
    assert code == 0
    o_phys, o_raw, _, inexact = oracle.prefill_rows(p, with_kth=True)
    assert inexact == 0
    rows = list(range(p.rows))
    scores = {r: oracle.row_scores(p, r)[0] for r in rows}
    assert np.isfinite(np.concatenate(list(scores.values()))).all()
    assert H.compare_rows(p, rows, g_raw, g_phys, o_raw, o_phys, scores) <= 2
