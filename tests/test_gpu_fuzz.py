"""Seeded randomised problems against the oracle: random request counts and C4
lengths, windows that start after 0 and end anywhere (page boundaries, one
slot, exactly topk, topk + 1), rows of a request out of order, page tables
that map several logical pages of a request to the same physical page (exact
score ties across positions), both supported topk values.  Each case checks
the fused call against the oracle and the selected set against the exact TopK
of the GPU's own scores."""
import numpy as np
import pytest

import oracle
from fp4_sparse_attention_tma_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _random_problem(seed):
    rng = np.random.default_rng(1000 + seed)
    topk = int(rng.choice([512, 1024]))
    n_req = int(rng.integers(1, 6))
    lens = [int(rng.integers(1, 6000)) for _ in range(n_req)]
    wins = []
    for i, L in enumerate(lens):
        n = int(rng.integers(0 if i else 1, 7))
        w = []
        for _ in range(n):
            kind = rng.integers(0, 6)
            if kind == 0:                      # one slot
                s = int(rng.integers(0, L)); e = s + 1
            elif kind == 1 and L > topk:       # exactly topk or topk + 1 long
                e = int(rng.integers(topk + 1, L + 1)); s = e - topk - int(rng.integers(0, 2))
            elif kind == 2:                    # ends on a page boundary
                e = max(64, (int(rng.integers(1, L + 1)) // 64) * 64); e = min(e, L)
                s = int(rng.integers(0, e))
            elif kind == 3:                    # empty
                s = e = int(rng.integers(0, L + 1))
            else:                              # anywhere
                e = int(rng.integers(1, L + 1)); s = int(rng.integers(0, e))
            w.append((s, e))
        rng.shuffle(w)
        wins.append(w)
    p = inputs.make_problem(2000 + seed, lens, wins, topk=topk, name=f"fuzz{seed}")
    # alias some logical pages of a request onto another of its physical pages
    if seed % 2 == 0:
        for r in range(p.page_table.shape[0]):
            used = np.flatnonzero(p.page_table[r] >= 0)
            if used.size >= 4:
                src = rng.choice(used, size=2, replace=False)
                p.page_table[r, src[1]] = p.page_table[r, src[0]]
    return p


@pytest.mark.parametrize("seed", range(8))
def test_random_problem_against_oracle(seed):
    p = _random_problem(seed)
    d = H.to_device(p)
    code, g_phys, g_raw = H.run_fused(p, d)
    assert code == 0
    o_phys, o_raw, _, inexact = oracle.prefill_rows(p, with_kth=True)
    assert inexact == 0
    rows = list(range(p.rows))
    scores = {r: oracle.row_scores(p, r)[0] for r in rows}
    assert H.compare_rows(p, rows, g_raw, g_phys, o_raw, o_phys, scores) <= 2
    sc, _ = H.run_debug(p, d)
    sc = sc.cpu().numpy()
    for r in rows:
        s0, s1 = int(p.row_start[r]), int(p.row_end[r])
        if s1 - s0 <= p.topk:
            continue
        np.testing.assert_array_equal(g_raw[r], H.brute_topk(sc[r, s0:s1], p.topk, s0))
