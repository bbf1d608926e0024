"""Shared helpers of the GPU tests: move a generated problem to the device, run
the library entry points, and compare with the oracle.

Comparison rules (tolerance from the method's stated bar: scores within 1e-5
relative / 1e-6 absolute of the float64 oracle):
  * per-head logits: exact equality (both sides are exact FP4 dot products);
  * scores: |gpu - oracle| <= 1e-6 + 1e-5 * sum_h |w_h| * max(logit_h, 0), the
    conditioned form of the bar (fp32 rounding of a sum that cancels can exceed
    1e-5 of its result; it cannot exceed it relative to the sum of magnitudes);
    every selected score additionally meets pure rtol 1e-5 / atol 1e-6 (see
    check_selected_scores for the one counted exception);
  * indices: the GPU's selected set must be exactly the TopK of the GPU's own
    scores; against the oracle, differences may only involve scores within the
    tolerance of the oracle's topk-th score, and are counted; the GPU's order
    must follow the oracle scores except where two selected scores lie within
    tolerance of each other;
  * the pure bar on selected scores is waived only where the head sum cancels
    tenfold or more, and those waivers are counted (check_selected_scores).
"""
from __future__ import annotations

import numpy as np

RTOL = 1e-5
ATOL = 1e-6


def to_device(p, device="cuda"):
    import torch
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return dict(q_fp4=f(p.q_fp4), q_scale=f(p.q_scale), k_cache_fp4=f(p.k_cache_fp4),
                k_scale=f(p.k_scale), weights=f(p.weights), page_table=f(p.page_table),
                row_req=f(p.row_req), row_start=f(p.row_start), row_end=f(p.row_end))


def run_fused(p, d=None, topk=None, raw=True, raise_on_error=True):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    d = d or to_device(p)
    K = int(topk or p.topk)
    R = p.rows
    phys = torch.zeros((R, K), dtype=torch.int32, device="cuda")
    rawt = torch.zeros((R, K), dtype=torch.int32, device="cuda") if raw else None
    code = m.idx_topk_fp4_prefill(**d, topk=K, out_phys_slot=phys, out_raw_idx=rawt,
                                  raise_on_error=raise_on_error)
    torch.cuda.synchronize()
    return code, phys.cpu().numpy(), (rawt.cpu().numpy() if raw else None)


def run_dense(p, d=None, workspace=True):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    d = d or to_device(p)
    K, R = p.topk, p.rows
    phys = torch.zeros((R, K), dtype=torch.int32, device="cuda")
    rawt = torch.zeros((R, K), dtype=torch.int32, device="cuda")
    ws = torch.empty((R, max(1, p.max_end())), dtype=torch.float32, device="cuda") if workspace else None
    m.idx_dense_topk_fp4_prefill(**d, topk=K, out_phys_slot=phys, out_raw_idx=rawt,
                                 score_workspace=ws)
    torch.cuda.synchronize()
    return phys.cpu().numpy(), rawt.cpu().numpy()


def run_debug(p, d=None, logits=False, rows=None):
    """GPU scores [R, S] (NaN outside windows) and optionally logits [R, 64, S]."""
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    d = d or to_device(p)
    S = max(1, p.max_end())
    sc = torch.full((p.rows, S), float("nan"), dtype=torch.float32, device="cuda")
    lg = torch.full((p.rows, 64, S), float("nan"), dtype=torch.float32, device="cuda") if logits else None
    m.idx_fp4_debug_scores(**d, out_scores=sc, out_logits=lg)
    torch.cuda.synchronize()
    return sc, lg


def score_bound(logits: np.ndarray, w: np.ndarray) -> np.ndarray:
    """1e-6 + 1e-5 * sum_h |w_h| * max(logit_h, 0) per slot; logits [n, 64]."""
    return ATOL + RTOL * (np.maximum(logits, 0.0) @ np.abs(w.astype(np.float64)))


def check_selected_scores(got, want, logits_sel, w) -> int:
    """Scores of selected positions: every one within the conditioned bound,
    and within the pure bar (rtol 1e-5, atol 1e-6 of the oracle score) unless
    the head sum cancels tenfold or more (|score| * 10 <= sum_h |w_h| *
    max(logit_h, 0)), where fp32 rounding of the sum cannot meet a bound relative
    to its small result.  Returns how many selected scores needed that exemption.
    got/want [n], logits_sel [n, 64] (oracle logits of the selected positions)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    mag = np.maximum(logits_sel, 0.0) @ np.abs(np.asarray(w, dtype=np.float64))
    err = np.abs(got - want)
    assert np.all(err <= ATOL + RTOL * mag), float((err - RTOL * mag).max())
    pure_miss = err > ATOL + RTOL * np.abs(want)
    assert np.all(np.abs(want[pure_miss]) * 10 <= mag[pure_miss])
    return int(pure_miss.sum())


def brute_topk(scores: np.ndarray, k: int, base: int) -> np.ndarray:
    """Exact TopK under the total order of a float32/64 vector (for property checks)."""
    s = np.asarray(scores, dtype=np.float64)
    idx = np.arange(s.size)
    nan = np.isnan(s)
    val = np.where(nan, 0.0, s)
    neg_zero = (val == 0) & np.signbit(val)
    order = np.lexsort((idx, neg_zero, -val, nan))
    out = np.full(k, -1, dtype=np.int64)
    m = min(k, s.size)
    out[:m] = order[:m] + base
    return out


def order_follows_oracle(sel: np.ndarray, sc: np.ndarray, s0: int) -> bool:
    """True when the selected positions `sel` are in the order of their oracle
    scores `sc` (indexed from s0): no entry's score lies below a later entry's
    by more than the score tolerance, and entries with equal oracle scores come
    in ascending position.  Near-equal scores (within tolerance) may come in
    either order, since fp32 rounding can swap them."""
    v = sc[np.asarray(sel) - s0]
    if v.size < 2:
        return True
    later_max = np.maximum.accumulate(v[::-1])[::-1][1:]     # max over the entries after i
    if not np.all(v[:-1] >= later_max - (ATOL + RTOL * np.abs(later_max))):
        return False
    eq = v[:-1] == v[1:]
    return bool(np.all(np.asarray(sel)[:-1][eq] < np.asarray(sel)[1:][eq]))


def compare_rows(p, rows, g_raw, g_phys, o_raw, o_phys, o_scores_by_row):
    """Compare GPU and oracle outputs of the listed rows.

    Returns the number of set differences; asserts that each difference lies at
    the selection boundary (oracle score within tolerance of the oracle's
    topk-th score), that the GPU's order follows the oracle scores (up to swaps
    of scores within tolerance of each other) and that the physical slots match
    the raw positions.
    """
    n_diff = 0
    K = p.topk
    for i, r in enumerate(rows):
        req = int(p.row_req[r])
        s0, s1 = int(p.row_start[r]), int(p.row_end[r])
        gr, orr = g_raw[i], o_raw[i]
        m = gr >= 0
        assert np.array_equal(g_phys[i][m], p.page_table[req, gr[m] // 64] * 64 + gr[m] % 64), r
        assert np.all(g_phys[i][~m] == -1)
        if s1 - s0 <= K:
            assert np.array_equal(gr, orr), r
            continue
        assert m.all(), r
        if np.array_equal(gr, orr):
            continue
        assert order_follows_oracle(gr, o_scores_by_row[r], s0), ("order", r)
        sg, so = set(gr.tolist()), set(orr.tolist())
        diff = sg ^ so
        sc = o_scores_by_row[r]
        kth = sc[orr[-1] - s0]
        for idx in diff:
            v = sc[idx - s0]
            assert abs(v - kth) <= ATOL + RTOL * abs(kth) + 1e-7 * abs(kth), (r, idx, v, kth)
        n_diff += len(diff) // 2
    return n_diff


def sample_rows(p, total=32, seed=0):
    """First and last row of every request, random rows (at least `total` over
    all requests, spread evenly), and the first short rows."""
    rng = np.random.default_rng(seed)
    rows = set()
    reqs = np.unique(p.row_req)
    per_req = max(2, -(-total // len(reqs)))
    for req in reqs:
        idx = np.nonzero(p.row_req == req)[0]
        rows.update([int(idx[0]), int(idx[-1])])
        rows.update(int(x) for x in rng.choice(idx, size=min(per_req, idx.size), replace=False))
    short = np.nonzero(p.lengths() <= p.topk)[0]
    rows.update(int(x) for x in short[:4])
    return np.array(sorted(rows), dtype=np.int32)


def check_against_oracle(p, g_phys, g_raw, rows=None, max_diff=None):
    """Compare the GPU outputs of `rows` (default: every row; g_phys/g_raw hold
    all rows) with the oracle by the rules of compare_rows; returns the number
    of boundary differences."""
    import oracle
    if rows is None:
        rows = np.arange(p.rows, dtype=np.int32)
    rows = np.asarray(rows, dtype=np.int32)
    o_phys, o_raw, _, inexact = oracle.prefill_rows(p, rows=rows, with_kth=True)
    assert inexact == 0
    scores = {int(r): oracle.row_scores(p, int(r))[0] for r in rows if p.lengths()[r] > p.topk}
    n = compare_rows(p, rows, g_raw[rows], g_phys[rows], o_raw, o_phys, scores)
    assert n <= (max_diff if max_diff is not None else max(2, len(rows) // 4)), n
    return n
