"""The stream-ordered entry point (caller workspace, device status word, no
host synchronisation): same outputs as the synchronous call, capturable into a
CUDA graph and replayable on new data, decode-shaped batches against the
oracle, device-detected errors published to the status word with -1 outputs,
host-side argument errors refused with nothing enqueued."""
import numpy as np
import pytest

import oracle
from fp4_sparse_attention_tma_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu

INVALID_ARGUMENT, INVALID_METADATA = 1, 3


def _decode_problem(seed=61, topk=512):
    # many requests with one or two query rows each (decode / MTP verify)
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(300, 20000, size=24)]
    wins = []
    for L in lens:
        n = 1 + int(rng.integers(0, 2))
        wins.append([(0, L - (n - 1 - j)) for j in range(n)])
    return inputs.make_problem(seed, lens, wins, topk=topk, name="decode-24req")


def _alloc(p, K=None):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    K = int(K or p.topk)
    ws = torch.empty(m.idx_topk_fp4_scratch_bytes(p.rows, K), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    phys = torch.full((p.rows, K), 7, dtype=torch.int32, device="cuda")
    raw = torch.full((p.rows, K), 7, dtype=torch.int32, device="cuda")
    return ws, st, phys, raw


def test_async_matches_sync():
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    p = inputs.small_problem(seed=17, topk=1024)
    d = H.to_device(p)
    ws, st, phys, raw = _alloc(p)
    assert m.idx_topk_fp4_prefill_async(**d, topk=p.topk, out_phys_slot=phys, out_raw_idx=raw,
                                        workspace=ws, status=st) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    code, want_phys, want_raw = H.run_fused(p, d)
    assert code == 0
    np.testing.assert_array_equal(raw.cpu().numpy(), want_raw)
    np.testing.assert_array_equal(phys.cpu().numpy(), want_phys)


@pytest.mark.parametrize("topk", [512, 1024])
def test_decode_batch_against_oracle(topk):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    p = _decode_problem(topk=topk)
    d = H.to_device(p)
    ws, st, phys, raw = _alloc(p)
    assert m.idx_topk_fp4_prefill_async(**d, topk=p.topk, out_phys_slot=phys, out_raw_idx=raw,
                                        workspace=ws, status=st) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_phys, o_raw, _, inexact = oracle.prefill_rows(p, with_kth=True)
    assert inexact == 0
    rows = list(range(p.rows))
    scores = {r: oracle.row_scores(p, r)[0] for r in rows if p.lengths()[r] > p.topk}
    ndiff = H.compare_rows(p, rows, raw.cpu().numpy(), phys.cpu().numpy(), o_raw, o_phys, scores)
    assert ndiff <= 2


def test_graph_capture_and_replay_on_new_data():
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    p = _decode_problem(seed=62)
    d = H.to_device(p)
    ws, st, phys, raw = _alloc(p)
    # the first call on the device outside the capture (library setup)
    assert m.idx_topk_fp4_prefill_async(**d, topk=p.topk, out_phys_slot=phys, out_raw_idx=raw,
                                        workspace=ws, status=st) == 0
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    codes = []
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            codes.append(m.idx_topk_fp4_prefill_async(**d, topk=p.topk, out_phys_slot=phys,
                                                      out_raw_idx=raw, workspace=ws, status=st))
    assert codes == [0]
    for trial in range(2):
        if trial == 1:
            # new weights in the same device buffer: the replay sees them
            rng = np.random.default_rng(5)
            d["weights"].copy_(torch.from_numpy(
                rng.standard_normal(p.weights.shape).astype(np.float32)))
        phys.fill_(7)
        raw.fill_(7)
        st.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        code, want_phys, want_raw = H.run_fused(p, d)
        assert code == 0
        np.testing.assert_array_equal(raw.cpu().numpy(), want_raw)
        np.testing.assert_array_equal(phys.cpu().numpy(), want_phys)


def test_device_error_published_and_outputs_failed_closed():
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    p = inputs.small_problem(seed=18, topk=512)
    d = H.to_device(p)
    bad = p.row_end.copy()
    bad[1] = p.page_table.shape[1] * 64 + 5          # past the page table: invalid metadata
    d["row_end"] = torch.from_numpy(bad).cuda()
    ws, st, phys, raw = _alloc(p)
    assert m.idx_topk_fp4_prefill_async(**d, topk=p.topk, out_phys_slot=phys, out_raw_idx=raw,
                                        workspace=ws, status=st, raise_on_error=False) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == INVALID_METADATA
    assert (phys.cpu().numpy() == -1).all() and (raw.cpu().numpy() == -1).all()


def test_small_workspace_refused_without_work():
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    p = inputs.small_problem(seed=19, topk=512)
    d = H.to_device(p)
    ws, st, phys, raw = _alloc(p)
    small = ws[: ws.numel() // 2]
    code = m.idx_topk_fp4_prefill_async(**d, topk=p.topk, out_phys_slot=phys, out_raw_idx=raw,
                                        workspace=small, status=st, raise_on_error=False)
    torch.cuda.synchronize()
    assert code == INVALID_ARGUMENT
    assert int(st.item()) == -7
    assert (phys.cpu().numpy() == 7).all()
