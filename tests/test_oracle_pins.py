"""Pins of the CPU oracle against facts that do not come from the oracle itself.

* E2M1 / UE8M0 decoding against the bit-level definitions of the OCP MX v1.0
  formats, derived here from the sign/exponent/mantissa fields.
* Per-head dots against numpy float64 matmul of operands decoded here
  independently (exact: every operand is a short dyadic rational), and against
  Python Fractions.
* Scores through identities that a dropped ReLU, a wrong sign or a wrong head /
  row index would break.
* Selection through known answers and a brute-force lexsort on tiny inputs.
* Short rows and page mapping through their closed forms.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from fp4_sparse_attention_tma_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---- independent decode (bit fields of the OCP MX E2M1 / E8M0 formats) -----

def e2m1_from_bits(code: int) -> float:
    sign = -1.0 if (code >> 3) & 1 else 1.0
    exp = (code >> 1) & 3
    man = code & 1
    if exp == 0:                      # subnormal: 2^(1-bias) * (m / 2), bias 1
        mag = man * 0.5
    else:
        mag = 2.0 ** (exp - 1) * (1.0 + man / 2.0)
    return math.copysign(mag, sign)


def decode_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """[..., 64] bytes + [..., 4] scale bytes -> [..., 128] float64 values."""
    lut = np.array([e2m1_from_bits(c) for c in range(16)])
    lo = codes & 0xF
    hi = codes >> 4
    vals = np.stack([lut[lo], lut[hi]], axis=-1).reshape(*codes.shape[:-1], 128)
    sc = np.ldexp(1.0, scales.astype(np.int64) - 127)
    return vals * np.repeat(sc, 32, axis=-1)


def k_logical(p, req: int, s0: int, s1: int):
    """K codes / scales of logical slots [s0, s1) of request req."""
    s = np.arange(s0, s1)
    pages = p.page_table[req, s // 64]
    return p.k_cache_fp4[pages, s % 64], p.k_scale[pages, s % 64]


# ---- decoding -------------------------------------------------------------

def test_e2m1_matches_bit_definition():
    for code in range(16):
        want = e2m1_from_bits(code)
        got = oracle.e2m1_value(code)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), code
    # the format's eight magnitudes: 0, 0.5, 1, 1.5, 2, 3, 4, 6
    assert sorted({abs(oracle.e2m1_value(c)) for c in range(16)}) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_ue8m0_is_power_of_two():
    for b in (0, 1, 100, 123, 127, 131, 200, 254):
        assert oracle.ue8m0_value(b) == math.ldexp(1.0, b - 127)
    assert math.isnan(oracle.ue8m0_value(255))


# ---- per-head dots ----------------------------------------------------------

@pytest.fixture(scope="module")
def small():
    return inputs.small_problem(seed=3, topk=512)


def test_dots_equal_exact_matmul(small):
    p = small
    for row in (0, 7, p.rows - 1):
        req, s0, s1 = int(p.row_req[row]), int(p.row_start[row]), int(p.row_end[row])
        got, inexact = oracle.row_logits(p, row, s0, s1)
        assert inexact == 0
        q = decode_rows(p.q_fp4[row], p.q_scale[row])            # [64, 128]
        kc, ks = k_logical(p, req, s0, s1)
        k = decode_rows(kc, ks)                                   # [n, 128]
        want = k @ q.T                                            # [n, 64]
        assert np.array_equal(got, want)


def test_dots_equal_fractions(small):
    p = small
    row, req = 4, int(small.row_req[4])
    got, _ = oracle.row_logits(p, row, 10, 13)
    lut = [Fraction(e2m1_from_bits(c)) for c in range(16)]
    for si, s in enumerate(range(10, 13)):
        kc, ks = k_logical(p, req, s, s + 1)
        for h in (0, 31, 63):
            tot = Fraction(0)
            for d in range(128):
                qv = lut[(p.q_fp4[row, h, d // 2] >> (4 * (d & 1))) & 15]
                kv = lut[(kc[0, d // 2] >> (4 * (d & 1))) & 15]
                sc = Fraction(2) ** (int(p.q_scale[row, h, d // 32]) - 127 +
                                     int(ks[0, d // 32]) - 127)
                tot += qv * kv * sc
            assert Fraction(got[si, h]) == tot


def test_dot_closed_form():
    # all Q codes 0x2 (1.0), all K codes 0x5 (3.0), scales 2^1 and 2^-2:
    # every dot is 128 * 1 * 3 * 2^(1-2) = 192
    p = inputs.make_problem(1, [64], [[(0, 64)]], 512, page_perm=False)
    p.q_fp4[:] = 0x22
    p.q_scale[:] = 128
    p.k_cache_fp4[:] = 0x55
    p.k_scale[:] = 125
    got, inexact = oracle.row_logits(p, 0, 0, 64)
    assert inexact == 0 and np.all(got == 192.0)
    # alternate the sign of even K elements (low nibble 0xD = -3): dots are 0
    p.k_cache_fp4[:] = 0x5D
    got, _ = oracle.row_logits(p, 0, 0, 64)
    assert np.all(got == 0.0)


def test_generator_keeps_dots_fp32_exact():
    p = inputs.config(0)
    _, _, _, inexact = oracle.prefill_rows(p, with_kth=True)
    assert inexact == 0


def test_inexact_flag_fires_on_a_wide_exponent_span():
    # Q head 0 and K slot 0: codes 1.0 in blocks 0 and 1, block exponents +15
    # and 0 on both sides, so the dot is 32 * 2^30 + 32 = 2^5 * (2^30 + 1): 31
    # significant bits, exact in float64 but not in fp32's 24.  Every other dot
    # is 0.  The flag must count exactly that one dot, and the value itself must
    # still be exact.
    p = inputs.make_problem(2, [64], [[(0, 64)]], 512, page_perm=False)
    p.q_fp4[:] = 0
    p.k_cache_fp4[:] = 0
    p.q_fp4[0, 0, :32] = 0x22
    p.k_cache_fp4[0, 0, :32] = 0x22
    p.q_scale[:] = 127
    p.k_scale[:] = 127
    p.q_scale[0, 0, 0] = 127 + 15
    p.k_scale[0, 0, 0] = 127 + 15
    got, inexact = oracle.row_logits(p, 0, 0, 64)
    assert inexact == 1
    assert got[0, 0] == 32.0 * 2.0 ** 30 + 32.0
    assert np.count_nonzero(got) == 1
    # a span of 22 keeps the value inside 24 significant bits: exact again
    p.q_scale[0, 0, 0] = 127 + 11
    p.k_scale[0, 0, 0] = 127 + 11
    got, inexact = oracle.row_logits(p, 0, 0, 64)
    assert inexact == 0 and got[0, 0] == 32.0 * 2.0 ** 22 + 32.0


# ---- scores ---------------------------------------------------------------

def _negated_k(p):
    q = inputs.Problem(**{f: getattr(p, f) for f in p.__dataclass_fields__})
    q.k_cache_fp4 = p.k_cache_fp4 ^ 0x88          # flip both sign bits of every byte
    return q


def test_score_relu_identities(small):
    p = small
    pn = _negated_k(p)
    for row in (1, 9, 15):
        req, s0, s1 = int(p.row_req[row]), int(p.row_start[row]), int(p.row_end[row])
        sp, _ = oracle.row_scores(p, row)
        sn, _ = oracle.row_scores(pn, row)
        q = decode_rows(p.q_fp4[row], p.q_scale[row])
        kc, ks = k_logical(p, req, s0, s1)
        k = decode_rows(kc, ks)
        w = p.weights[row].astype(np.float64)
        # relu(x) - relu(-x) = x: difference is the weighted dot with sum_h w_h q_h
        lin = k @ (q.T @ w)
        assert np.allclose(sp - sn, lin, rtol=1e-12, atol=1e-9)
        # relu(x) + relu(-x) = |x|
        ab = np.abs(k @ q.T) @ w
        assert np.allclose(sp + sn, ab, rtol=1e-12, atol=1e-9)


def test_score_one_hot_weight_selects_head(small):
    p = inputs.Problem(**{f: getattr(small, f) for f in small.__dataclass_fields__})
    p.weights = np.zeros_like(small.weights)
    row, head = 6, 37
    p.weights[row, head] = 1.0
    s, _ = oracle.row_scores(p, row)
    dots, _ = oracle.row_logits(p, row, int(p.row_start[row]), int(p.row_end[row]))
    q = decode_rows(p.q_fp4[row, head], p.q_scale[row, head])
    kc, ks = k_logical(p, int(p.row_req[row]), int(p.row_start[row]), int(p.row_end[row]))
    want = np.maximum(decode_rows(kc, ks) @ q, 0.0)
    assert np.array_equal(s, want)
    assert np.array_equal(dots[:, head], decode_rows(kc, ks) @ q)


def test_score_linear_in_weights_and_head_permutation(small):
    p = small
    row = 11
    s1, _ = oracle.row_scores(p, row)
    p2 = inputs.Problem(**{f: getattr(p, f) for f in p.__dataclass_fields__})
    p2.weights = p.weights * 2.0
    s2, _ = oracle.row_scores(p2, row)
    assert np.array_equal(s2, 2.0 * s1)
    perm = np.random.default_rng(0).permutation(64)
    p3 = inputs.Problem(**{f: getattr(p, f) for f in p.__dataclass_fields__})
    p3.q_fp4 = p.q_fp4[:, perm].copy()
    p3.q_scale = p.q_scale[:, perm].copy()
    p3.weights = p.weights[:, perm].copy()
    s3, _ = oracle.row_scores(p3, row)
    assert np.allclose(s3, s1, rtol=1e-12, atol=1e-12)


def test_score_uses_own_row(small):
    p = small
    row = 12
    sub = inputs.Problem(**{f: getattr(p, f) for f in p.__dataclass_fields__})
    for f in ("q_fp4", "q_scale", "weights", "row_req", "row_start", "row_end"):
        setattr(sub, f, getattr(p, f)[row:row + 1].copy())
    a, _ = oracle.row_scores(p, row)
    b, _ = oracle.row_scores(sub, 0)
    assert np.array_equal(a, b)


# ---- selection ------------------------------------------------------------

def brute_select(scores: np.ndarray, k: int, base: int = 0) -> np.ndarray:
    """Brute-force total order: numbers before NaN, larger first, +0 before -0,
    then lower index."""
    s = np.asarray(scores, dtype=np.float64)
    idx = np.arange(s.size)
    nan = np.isnan(s)
    val = np.where(nan, 0.0, s)
    neg_zero = (val == 0) & np.signbit(val)
    order = np.lexsort((idx, neg_zero, -val, nan))
    out = np.full(k, -1, dtype=np.int32)
    m = min(k, s.size)
    out[:m] = order[:m] + base
    return out


def test_select_known_answers():
    nan = float("nan")
    assert list(oracle.select(np.array([nan, -0.0, 0.0, -np.inf, 1.0]), 3)) == [4, 2, 1]
    assert list(oracle.select(np.full(10, 2.5), 4)) == [0, 1, 2, 3]
    assert list(oracle.select(np.arange(10.0), 3)) == [9, 8, 7]
    assert list(oracle.select(np.array([1.0, 2.0]), 4)) == [1, 0, -1, -1]
    assert list(oracle.select(np.array([np.inf, 1e300, -np.inf, nan]), 4)) == [0, 1, 2, 3]
    assert list(oracle.select(np.array([-nan, nan, -np.inf]), 3)) == [2, 0, 1]
    assert list(oracle.select(np.array([3.0, 5.0, 5.0, 1.0]), 2, base=100)) == [101, 102]


def test_select_matches_brute_force():
    rng = np.random.default_rng(5)
    specials = np.array([np.nan, -np.nan, 0.0, -0.0, np.inf, -np.inf, 1.0, -1.0])
    for trial in range(200):
        n = int(rng.integers(0, 40))
        s = rng.choice(specials, size=n) if trial % 2 else \
            rng.integers(-3, 4, size=n).astype(np.float64)
        k = int(rng.integers(1, 12))
        assert np.array_equal(oracle.select(s, k, base=7), brute_select(s, k, base=7))


def test_prefill_matches_brute_force_tiny():
    # dyadic weights keep every float64 sum exact, so the ranking is unambiguous
    p = inputs.make_problem(11, [300, 200], [[(0, 300), (20, 250), (0, 5)], [(3, 200), (0, 0)]],
                            topk=16)
    p.weights = (np.random.default_rng(1).integers(-8, 9, size=p.weights.shape) / 4.0
                 ).astype(np.float32)
    phys, raw = oracle.prefill_rows(p)
    for r in range(p.rows):
        req, s0, s1 = int(p.row_req[r]), int(p.row_start[r]), int(p.row_end[r])
        if s1 - s0 <= p.topk:
            want = np.full(p.topk, -1)
            want[:s1 - s0] = np.arange(s0, s1)
        else:
            q = decode_rows(p.q_fp4[r], p.q_scale[r])
            kc, ks = k_logical(p, req, s0, s1)
            sc = np.maximum(decode_rows(kc, ks) @ q.T, 0.0) @ p.weights[r].astype(np.float64)
            want = brute_select(sc, p.topk, base=s0)
        assert np.array_equal(raw[r], want), r
        m = want >= 0
        assert np.array_equal(phys[r][m], p.page_table[req, want[m] // 64] * 64 + want[m] % 64)
        assert np.all(phys[r][~m] == -1)


def test_short_rows_and_empty_window():
    p = inputs.config(0)
    phys, raw = oracle.prefill_rows(p, rows=np.array([0, 1], dtype=np.int32))
    assert np.array_equal(raw[0], np.r_[np.arange(100), np.full(412, -1)])
    assert np.array_equal(raw[1], np.arange(512))          # len == topk is a short row
    p4 = inputs.make_problem(2, [128], [[(0, 0), (5, 9)]], 512)
    phys, raw = oracle.prefill_rows(p4)
    assert np.all(raw[0] == -1) and np.all(phys[0] == -1)
    assert np.array_equal(raw[1][:4], [5, 6, 7, 8]) and np.all(raw[1][4:] == -1)


def test_page_mapping_identity_and_shuffled():
    ident = inputs.make_problem(4, [1000], [[(0, 1000)] * 2], 512, page_perm=False)
    shuf = inputs.Problem(**{f: getattr(ident, f) for f in ident.__dataclass_fields__})
    # move every logical page to a shuffled physical page, data with it
    shuf.page_table = ident.page_table.copy()
    shuf.page_table[0] = np.random.default_rng(8).permutation(ident.num_pages)
    shuf.k_cache_fp4 = np.empty_like(ident.k_cache_fp4)
    shuf.k_scale = np.empty_like(ident.k_scale)
    for lp in range(ident.page_table.shape[1]):
        shuf.k_cache_fp4[shuf.page_table[0, lp]] = ident.k_cache_fp4[lp]
        shuf.k_scale[shuf.page_table[0, lp]] = ident.k_scale[lp]
    pi, ri = oracle.prefill_rows(ident)
    ps, rs = oracle.prefill_rows(shuf)
    assert np.array_equal(pi, ri)                     # identity table: phys == raw
    assert np.array_equal(rs, ri)                     # raw indices unchanged
    assert np.array_equal(ps, shuf.page_table[0, rs // 64] * 64 + rs % 64)
    assert not np.array_equal(ps, pi)


def test_duplicated_slots_tie_to_lower_index():
    p = inputs.config(0)
    row = 20
    sc, _ = oracle.row_scores(p, row)
    phys, raw = oracle.prefill_rows(p, rows=np.array([row], dtype=np.int32))
    sel = raw[0]
    vals = sc[sel]
    assert np.all(np.diff(vals) <= 0)
    # at least one exact tie exists among the duplicated slots, ordered by index
    ties = np.nonzero(np.diff(vals) == 0)[0]
    assert all(sel[i] < sel[i + 1] for i in ties)
    uniq, counts = np.unique(sc, return_counts=True)
    assert (counts > 1).sum() >= 32


def test_oracle_rejects_bad_metadata():
    p = inputs.make_problem(9, [256], [[(0, 256)]], 16)
    p.row_end = np.array([300], dtype=np.int32)          # beyond the page table
    with pytest.raises(oracle.OracleError):
        oracle.prefill_rows(p)
    p = inputs.make_problem(9, [256], [[(0, 256)]], 16)
    p.page_table[0, 2] = 99                              # page out of range
    with pytest.raises(oracle.OracleError):
        oracle.prefill_rows(p)
