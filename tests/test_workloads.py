"""The five seeded synthetic workloads (CPU only): shapes, the causal window rule,
the page tables and the value ranges the generator promises, and the totals the
benchmark's metric divides by.

Causal C4 rule ("[FlyDSL][DSv4] Prototype FP4 MQA streaming TopK", ROCm/aiter#5282,
Validation: causal rows at the end of a request): the row of raw token t sees C4
entries [0, (t + 1) // 4); a request of C4 length L whose n rows are its last raw
tokens holds t = 4L - n + j for row j.  The expected values below are computed
here from that rule with plain integers, not by the generator's own helper.
"""
import numpy as np
import pytest

from fp4_sparse_attention_tma_gb300 import inputs

H, D = 64, 128

# name, rows, requests, topk, sum of window lengths, scored pairs (rows with len > topk)
TABLE = [
    ("tiny-R32-S4096-K512", 32, 1, 512, 123_057, 122_445),
    ("mid-R1024-4req-8k..64k-K512", 1024, 4, 512, 31_424_256, 31_424_256),
    ("flash-R8192-S131072-K512", 8192, 1, 512, 1_065_351_168, 1_065_351_168),
    ("pro-R8192-S196608-K1024", 8192, 1, 1024, 1_602_222_080, 1_602_222_080),
    ("long-R1024-8req-up-to-262144-K1024", 1024, 8, 1024, 150_913_832, 150_912_832),
]

CAUSAL = {  # config -> (C4 lengths, rows per request, {(request, row): overridden end})
    1: ([8192, 16384, 32768, 65536], 256, {}),
    2: ([131072], 8192, {}),
    3: ([196608], 8192, {}),
    4: ([32768 * (i + 1) for i in range(8)], 128, {(0, 0): 0, (0, 1): 1000}),
}


@pytest.fixture(scope="module", params=range(5))
def workload(request):
    return request.param, inputs.config(request.param)


def test_shapes_and_totals(workload):
    idx, p = workload
    name, rows, n_req, topk, sum_len, scored = TABLE[idx]
    assert p.name == name and p.rows == rows and p.topk == topk
    assert len(np.unique(p.row_req)) == n_req
    assert p.q_fp4.shape == (rows, H, D // 2) and p.q_scale.shape == (rows, H, D // 32)
    assert p.weights.shape == (rows, H) and p.weights.dtype == np.float32
    assert p.k_cache_fp4.shape == (p.num_pages, 64, D // 2) and p.k_scale.shape == (p.num_pages, 64, 4)
    lengths = [int(e) - int(s) for s, e in zip(p.row_start, p.row_end)]
    assert sum(lengths) == sum_len
    assert sum(n for n in lengths if n > topk) == scored == p.scored_pairs()
    assert p.algorithmic_flop() == 2 * H * D * scored


def test_causal_windows(workload):
    idx, p = workload
    if idx == 0:
        want = [4065 + r for r in range(32)]
        want[0], want[1] = 100, 512
        assert p.row_start.tolist() == [0] * 32 and p.row_end.tolist() == want
        return
    lens, n, overrides = CAUSAL[idx]
    r = 0
    for i, L in enumerate(lens):
        for j in range(n):
            t = 4 * L - n + j
            end = overrides.get((i, j), (t + 1) // 4)
            assert (int(p.row_req[r]), int(p.row_start[r]), int(p.row_end[r])) == (i, 0, end)
            r += 1
    assert r == p.rows


def test_page_tables_are_one_permutation(workload):
    idx, p = workload
    c4 = [4096] if idx == 0 else CAUSAL[idx][0]
    used = []
    for i, L in enumerate(c4):
        n = -(-L // 64)
        assert (p.page_table[i, :n] >= 0).all() and (p.page_table[i, n:] == -1).all()
        used.extend(p.page_table[i, :n].tolist())
    assert sorted(used) == list(range(p.num_pages))


def test_value_ranges(workload):
    _, p = workload
    for sf in (p.q_scale, p.k_scale):
        e = sf.astype(np.int32) - 127
        assert e.min() >= -4 and e.max() <= 4
        assert (e.max(axis=-1) - e.min(axis=-1)).max() <= 4   # span rule: dots exact in fp32
    assert np.isfinite(p.weights).all()


def test_tiny_workload_has_exact_ties():
    p = inputs.config(0)
    slots = p.k_cache_fp4.reshape(-1, D // 2)
    scales = p.k_scale.reshape(-1, 4)
    keys = np.concatenate([slots, scales], axis=1)
    _, counts = np.unique(keys, axis=0, return_counts=True)
    assert (counts >= 2).sum() >= 64


def test_k_scale_mma_order_is_the_documented_permutation():
    # byte 8j + 4h + b of a page = scale b of slot 32h + j (a permutation of
    # each page's 256 bytes)
    k = np.random.default_rng(5).integers(0, 256, size=(3, 64, 4), dtype=np.uint8)
    o = inputs.k_scale_mma_order(k)
    assert o.shape == (3, 256) and o.flags["C_CONTIGUOUS"]
    for p in range(3):
        for j in range(32):
            for h in range(2):
                for b in range(4):
                    assert o[p, 8 * j + 4 * h + b] == k[p, 32 * h + j, b]
        assert sorted(o[p].tolist()) == sorted(k[p].ravel().tolist())


def test_decode_batch_recipe():
    """The bench's decode batch: 32 requests, two rows each with windows
    [0, L-1) and [0, L), C4 lengths in [4096, 65536), deterministic."""
    a = inputs.decode_batch(32, 512)
    b = inputs.decode_batch(32, 512)
    assert a.rows == 64 and a.topk == 512
    np.testing.assert_array_equal(a.row_req, np.repeat(np.arange(32), 2))
    L = a.row_end[1::2]
    assert np.all(a.row_start == 0) and np.all(a.row_end[0::2] == L - 1)
    assert np.all((L >= 4096) & (L < 65536))
    np.testing.assert_array_equal(a.q_fp4, b.q_fp4)
    np.testing.assert_array_equal(a.page_table, b.page_table)
    assert inputs.decode_batch(32, 1024).topk == 1024
