"""Concurrent calls through the C ABI on the GPU: several host threads, each on
its own CUDA stream and problem, call the synchronous, stream-ordered and
host-buffer entry points at the same time (sharing the library's per-device
state and scratch pool); every call returns exactly the result of the same
call made alone."""
import threading

import numpy as np
import pytest

from fp4_sparse_attention_tma_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _problems():
    return [inputs.small_problem(seed=31 + i, topk=512 if i % 2 == 0 else 1024,
                                 c4_lens=(1800 + 700 * i, 3100, 900), rows_per_req=(4, 7, 3))
            for i in range(4)]


def _run(kind, p, d, stream):
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    K = p.topk
    with torch.cuda.stream(stream):
        if kind == "host":
            phys = torch.zeros((p.rows, K), dtype=torch.int32).pin_memory()
            raw = torch.zeros((p.rows, K), dtype=torch.int32).pin_memory()
            hd = {k: v.cpu().pin_memory() for k, v in d.items()}
            code = m.idx_topk_fp4_prefill_host(**hd, topk=K, out_phys_slot=phys, out_raw_idx=raw,
                                               device=0, stream=stream)
            return code, phys.numpy().copy(), raw.numpy().copy()
        phys = torch.zeros((p.rows, K), dtype=torch.int32, device="cuda")
        raw = torch.zeros((p.rows, K), dtype=torch.int32, device="cuda")
        if kind == "sync":
            code = m.idx_topk_fp4_prefill(**d, topk=K, out_phys_slot=phys, out_raw_idx=raw,
                                          stream=stream)
        else:
            ws = torch.empty(m.idx_topk_fp4_scratch_bytes(p.rows, K), dtype=torch.uint8,
                             device="cuda")
            st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
            code = m.idx_topk_fp4_prefill_async(**d, topk=K, out_phys_slot=phys, out_raw_idx=raw,
                                                workspace=ws, status=st, stream=stream)
            stream.synchronize()
            code = code or int(st.item())
        stream.synchronize()
        return code, phys.cpu().numpy(), raw.cpu().numpy()


@pytest.mark.parametrize("kind", ["sync", "async", "host"])
def test_concurrent_threads_match_single_calls(kind):
    import torch
    probs = _problems()
    devs = [H.to_device(p) for p in probs]
    streams = [torch.cuda.Stream() for _ in probs]
    want = [_run(kind, p, d, s) for p, d, s in zip(probs, devs, streams)]
    for code, _, _ in want:
        assert code == 0
    errors = []

    def worker(i):
        try:
            torch.cuda.set_device(0)
            for _ in range(5):
                got = _run(kind, probs[i], devs[i], streams[i])
                assert got[0] == 0
                assert np.array_equal(got[1], want[i][1]) and np.array_equal(got[2], want[i][2])
        except Exception as e:  # reported by the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(probs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
