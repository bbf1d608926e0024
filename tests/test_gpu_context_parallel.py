"""Context-parallel scoring on one GPU: the context is cut into S disjoint
shards, each scored by idx_topk_fp4_prefill_shard (the part of every window
inside the shard), and the gathered [S, R, topk] lists are merged exactly by
idx_topk_merge_shards ("[AMD][DSv4] Add experimental AITER FP4 streaming TopK",
Changes: context-parallel paths; "[FlyDSL][DSv4] Prototype FP4 MQA streaming
TopK", Changes: merge split candidates exactly).  The merged outputs must equal
the unsharded fused call bit for bit and the oracle by the usual rules; each
shard's scores must meet the score tolerance against the oracle; malformed
lists fail closed."""
import numpy as np
import pytest

import oracle
from fp4_sparse_attention_tma_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu

INVALID_ARGUMENT, INVALID_METADATA = 1, 3


def _shard(p, d, c0, c1, raise_on_error=True):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    sc = torch.zeros((p.rows, p.topk), dtype=torch.float32, device="cuda")
    raw = torch.zeros((p.rows, p.topk), dtype=torch.int32, device="cuda")
    code = m.idx_topk_fp4_prefill_shard(**d, ctx_begin=c0, ctx_end=c1, topk=p.topk, out_score=sc,
                                        out_raw_idx=raw, raise_on_error=raise_on_error)
    torch.cuda.synchronize()
    return code, sc, raw


def _merge(p, d, scores, raws, raise_on_error=True):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    phys = torch.zeros((p.rows, p.topk), dtype=torch.int32, device="cuda")
    raw = torch.zeros((p.rows, p.topk), dtype=torch.int32, device="cuda")
    code = m.idx_topk_merge_shards(torch.stack(scores), torch.stack(raws), d["page_table"],
                                   d["row_req"], d["row_start"], d["row_end"], p.topk, phys, raw,
                                   raise_on_error=raise_on_error)
    torch.cuda.synchronize()
    return code, phys.cpu().numpy(), raw.cpu().numpy()


def _bounds(p, n_shards, unaligned=False):
    end = p.max_end()
    b = [round(end * i / n_shards) for i in range(n_shards + 1)]
    if unaligned and n_shards > 1:
        b[1] += 37  # a boundary inside a page and inside a tile
    return list(zip(b[:-1], b[1:]))


def _sharded(p, d, bounds):
    scores, raws = [], []
    for c0, c1 in bounds:
        code, sc, raw = _shard(p, d, c0, c1)
        assert code == 0
        scores.append(sc)
        raws.append(raw)
    return scores, raws


@pytest.mark.parametrize("which,n_shards,unaligned", [("small512", 2, True), ("small1024", 3, True),
                                                      ("config1", 2, False), ("config1", 4, True),
                                                      ("config4", 4, False)])
def test_sharded_equals_fused_and_oracle(which, n_shards, unaligned):
    p = {"small512": lambda: inputs.small_problem(seed=41, topk=512),
         "small1024": lambda: inputs.small_problem(seed=42, topk=1024),
         "config1": lambda: inputs.config(1),
         "config4": lambda: inputs.config(4)}[which]()
    d = H.to_device(p)
    scores, raws = _sharded(p, d, _bounds(p, n_shards, unaligned))
    code, phys, raw = _merge(p, d, scores, raws)
    assert code == 0
    code2, want_phys, want_raw = H.run_fused(p, d)
    assert code2 == 0
    np.testing.assert_array_equal(raw, want_raw)
    np.testing.assert_array_equal(phys, want_phys)
    rows = None if p.rows <= 64 else H.sample_rows(p, total=12, seed=n_shards)
    H.check_against_oracle(p, phys, raw, rows)


def test_768k_context_in_four_shards():
    L, K = 786432, 1024
    wins = [(0, L - 3 + j) for j in range(4)] + [(100000, 700001), (L - K - 1, L), (5, 5 + K)]
    p = inputs.make_problem(31, [L], [wins], topk=K, name="ctx768k-K1024")
    d = H.to_device(p)
    scores, raws = _sharded(p, d, _bounds(p, 4, unaligned=True))
    code, phys, raw = _merge(p, d, scores, raws)
    assert code == 0
    code2, want_phys, want_raw = H.run_fused(p, d)
    np.testing.assert_array_equal(raw, want_raw)
    np.testing.assert_array_equal(phys, want_phys)


def test_shard_lists_against_oracle():
    # each shard's list: the exact TopK of the clipped window (ties at the
    # boundary within tolerance), scores within the conditioned tolerance of the
    # oracle, -1 / NaN padding after the clipped window's last position, and
    # nothing for rows whose whole window is at most topk long
    p = inputs.small_problem(seed=43, topk=512)
    d = H.to_device(p)
    lens = p.lengths()
    for c0, c1 in _bounds(p, 3, unaligned=True):
        code, sc, raw = _shard(p, d, c0, c1)
        assert code == 0
        sc, raw = sc.cpu().numpy(), raw.cpu().numpy()
        for r in range(p.rows):
            s0, s1 = int(p.row_start[r]), int(p.row_end[r])
            a, b = max(s0, c0), min(s1, c1)
            if lens[r] <= p.topk or a >= b:
                assert (raw[r] == -1).all() and np.isnan(sc[r]).all()
                continue
            n = min(b - a, p.topk)
            assert (raw[r, :n] >= a).all() and (raw[r, :n] < b).all()
            assert (raw[r, n:] == -1).all() and np.isnan(sc[r, n:]).all()
            want = oracle.row_scores(p, r, a, b)[0]
            lg, _ = oracle.row_logits(p, r, a, b)
            got = sc[r, :n].astype(np.float64)
            sel = raw[r, :n] - a
            assert np.all(np.abs(got - want[sel]) <= H.score_bound(lg[sel], p.weights[r]))
            o_sel = oracle.select(want, p.topk, base=a)[:n]
            diff = set(o_sel.tolist()) ^ set(raw[r, :n].tolist())
            kth = want[o_sel[-1] - a]
            for i in diff:
                assert abs(want[i - a] - kth) <= H.ATOL + 2 * H.RTOL * abs(kth), (r, i)


def test_merge_fails_closed_on_malformed_lists():
    import torch
    p = inputs.small_problem(seed=44, topk=512)
    d = H.to_device(p)
    bounds = _bounds(p, 2)
    scores, raws = _sharded(p, d, bounds)
    long_row = int(np.nonzero(p.lengths() > p.topk)[0][0])
    # the same shard twice: positions listed twice
    code, phys, raw = _merge(p, d, [scores[0], scores[0], scores[1]], [raws[0], raws[0], raws[1]],
                             raise_on_error=False)
    assert code == INVALID_METADATA and (phys == -1).all() and (raw == -1).all()
    # a position outside the row's window
    bad = [r.clone() for r in raws]
    bad[0][long_row, 0] = int(p.row_end[long_row]) + 3
    code, phys, raw = _merge(p, d, scores, bad, raise_on_error=False)
    assert code == INVALID_METADATA and (phys == -1).all()
    # a missing shard: rows longer than topk underfilled
    code, phys, raw = _merge(p, d, scores[:1], raws[:1], raise_on_error=False)
    assert code == INVALID_METADATA and (phys == -1).all()
    # a bad context range of a shard call
    code, sc, raw = _shard(p, d, 100, 50, raise_on_error=False)
    assert code == INVALID_ARGUMENT and bool((raw == -1).all()) and bool(torch.isnan(sc).all())


def test_merge_fails_closed_on_negative_page_entry():
    """The merge maps every emitted position through the page table; a negative
    entry under an emitted position returns IDX_ERR_INVALID_PAGE with -1 outputs
    (the short rows' positions are all emitted, so an entry under a short row's
    window is always read)."""
    p = inputs.small_problem(seed=45, topk=512)
    d = H.to_device(p)
    scores, raws = _sharded(p, d, _bounds(p, 2))
    code, phys, raw = _merge(p, d, scores, raws)
    assert code == 0
    # a page under a position that the merge emits for row 0
    r0 = 0
    pos = int(raw[r0][raw[r0] >= 0][0])
    req = int(p.row_req[r0])
    bad = d["page_table"].clone()
    bad[req, pos // 64] = -1
    d2 = dict(d, page_table=bad)
    code, phys, raw = _merge(p, d2, scores, raws, raise_on_error=False)
    assert code == 4 and (phys == -1).all() and (raw == -1).all()
