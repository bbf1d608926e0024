"""The range-checked build of the library (-DIDX_DEBUG_BOUNDS, a software
stand-in for a memory checker): every indexed scratch and output access of the
kernels is checked against its buffer, and an index outside it fails the call
with IDX_ERR_INTERNAL instead of touching memory.  On small cases of every
entry point it must return IDX_OK and the release build's outputs bit for bit
(which the other tests compare with the oracle); the fused case is also compared
with the oracle directly."""
import numpy as np
import pytest

import oracle
from fp4_sparse_attention_tma_gb300 import _lib, inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    return _lib.load(_lib.build(debug_bounds=True))


def _with(lib, fn, monkeypatch):
    """Run fn() with the binding routed to `lib`."""
    monkeypatch.setattr(_lib, "_lib", lib)
    return fn()


def _problems():
    rng = np.random.default_rng(91)
    wins = [[(int(a), int(a + b)) for a, b in zip(rng.integers(0, 1500, 9),
                                                 rng.integers(0, 2500, 9))],
            [(0, 3000), (5, 517), (0, 0), (2000, 3000)]]
    return {"config0": inputs.config(0),
            "small1024": inputs.small_problem(seed=92, topk=1024),
            "ragged512": inputs.make_problem(93, [4000, 3000], wins, topk=512, name="ragged")}


@pytest.mark.parametrize("which", ["config0", "small1024", "ragged512"])
def test_fused_dense_and_tiled_in_range(which, dbg, monkeypatch):
    p = _problems()[which]
    d = H.to_device(p)
    want = H.run_fused(p, d)
    got = _with(dbg, lambda: H.run_fused(p, d, raise_on_error=False), monkeypatch)
    assert got[0] == 0
    np.testing.assert_array_equal(got[1], want[1])
    np.testing.assert_array_equal(got[2], want[2])
    if which == "config0":
        H.check_against_oracle(p, got[1], got[2])
    dp, dr = _with(dbg, lambda: H.run_dense(p, d), monkeypatch)
    np.testing.assert_array_equal(dr, want[2])
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    phys = torch.zeros((p.rows, p.topk), dtype=torch.int32, device="cuda")
    raw = torch.zeros_like(phys)
    code = _with(dbg, lambda: m.idx_tiled_topk_fp4_prefill(
        **d, topk=p.topk, out_phys_slot=phys, out_raw_idx=raw, context_tile=1024,
        raise_on_error=False), monkeypatch)
    torch.cuda.synchronize()
    assert code == 0
    np.testing.assert_array_equal(raw.cpu().numpy(), want[2])


def test_shards_async_noalloc_and_scale_layouts_in_range(dbg, monkeypatch):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    p = _problems()["ragged512"]
    d = H.to_device(p)
    _, want_phys, want_raw = H.run_fused(p, d)
    monkeypatch.setattr(_lib, "_lib", dbg)
    R, K = p.rows, p.topk
    # two context shards and their merge
    end = p.max_end()
    scores, raws = [], []
    for c0, c1 in ((0, end // 2 + 13), (end // 2 + 13, end)):
        sc = torch.zeros((R, K), dtype=torch.float32, device="cuda")
        rw = torch.zeros((R, K), dtype=torch.int32, device="cuda")
        assert m.idx_topk_fp4_prefill_shard(**d, ctx_begin=c0, ctx_end=c1, topk=K, out_score=sc,
                                            out_raw_idx=rw, raise_on_error=False) == 0
        scores.append(sc)
        raws.append(rw)
    phys = torch.zeros((R, K), dtype=torch.int32, device="cuda")
    raw = torch.zeros_like(phys)
    assert m.idx_topk_merge_shards(torch.stack(scores), torch.stack(raws), d["page_table"],
                                   d["row_req"], d["row_start"], d["row_end"], K, phys, raw,
                                   raise_on_error=False) == 0
    torch.cuda.synchronize()
    np.testing.assert_array_equal(raw.cpu().numpy(), want_raw)
    # stream-ordered call with a caller workspace
    ws = torch.empty(m.idx_topk_fp4_scratch_bytes(R, K, 0), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    raw.zero_()
    assert m.idx_topk_fp4_prefill_async(**d, topk=K, out_phys_slot=phys, workspace=ws, status=st,
                                        out_raw_idx=raw, raise_on_error=False) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(raw.cpu().numpy(), want_raw)
    # fixed-buffer call
    raw.zero_()
    assert m.idx_topk_fp4_prefill_noalloc(**d, topk=K, out_phys_slot=phys, out_raw_idx=raw,
                                          raise_on_error=False) == 0
    np.testing.assert_array_equal(raw.cpu().numpy(), want_raw)
    # the MMA-order scale layout and the page-interleaved cache
    ksm = torch.from_numpy(inputs.k_scale_mma_order(p.k_scale)).cuda()
    args = {k: v for k, v in d.items() if k != "k_scale"}
    raw.zero_()
    assert m.idx_topk_fp4_prefill_mma_scales(**args, k_scale_mma=ksm, topk=K, out_phys_slot=phys,
                                             out_raw_idx=raw, raise_on_error=False) == 0
    torch.cuda.synchronize()
    np.testing.assert_array_equal(raw.cpu().numpy(), want_raw)
    npg = p.k_cache_fp4.shape[0]
    kp = torch.from_numpy(np.ascontiguousarray(np.concatenate(
        [p.k_cache_fp4.reshape(npg, 4096), p.k_scale.reshape(npg, 256)], axis=1))).cuda()
    args = {k: v for k, v in d.items() if k not in ("k_cache_fp4", "k_scale")}
    raw.zero_()
    assert m.idx_topk_fp4_prefill_paged(**args, k_pages=kp, topk=K, out_phys_slot=phys,
                                        out_raw_idx=raw, raise_on_error=False) == 0
    torch.cuda.synchronize()
    np.testing.assert_array_equal(raw.cpu().numpy(), want_raw)
