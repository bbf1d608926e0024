"""Seeded synthetic inputs for the FP4 paged-MQA indexer prefill.

This module only draws random numbers and lays out metadata. It holds none of
the method's arithmetic (no decoding, no dot products, no selection), so both
the CUDA path and the CPU oracle can be fed from it without sharing any code
that computes a result.

Workload shapes follow "[FlyDSL] Add FP4 LiteTopK prefill operator"
(ROCm/aiter#5309, Summary table: Q=8192, H=64, D=128, K in {512, 1024}, C4 KV
context) and "[FlyDSL][DSv4] Prototype FP4 MQA streaming TopK" (ROCm/aiter#5282,
Scope: page size 64, FP4 E2M1 payload with UE8M0 scales, ragged windows).

Value recipe (the pages only say "deterministic tensors with the released model
shapes"; the plain reading taken here):
  * FP4 E2M1 codes uniform over all 16 codes, two per byte, low nibble = even
    element along D.
  * one UE8M0 scale byte per 32 elements along D, exponent uniform in [-4, 4]
    (byte = exponent + 127).  The four exponents of one Q head row or one K slot
    are redrawn together until max - min <= 4, which keeps every per-head dot
    exactly representable in fp32.
  * weights float32 N(0, 1).
  * physical pages: exactly sum(ceil(L_i / 64)) pages, assigned to requests
    through one seeded permutation; unused page-table entries are -1.
  * causal C4 windows: a request of C4 length L whose rows are its last n raw
    tokens t = 4L - n + j sees C4 entries [0, floor((t + 1) / 4)).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

H = 64           # heads per query row
D = 128          # head dimension (FP4 elements)
PAGE = 64        # KV page size (C4 slots per page)
SF_BLOCK = 32    # elements per UE8M0 scale
D_BYTES = D // 2
N_SF = D // SF_BLOCK
SEED_BASE = 20260


@dataclasses.dataclass
class Problem:
    """One prefill call's inputs, host-side numpy arrays in the C-ABI layout."""
    name: str
    q_fp4: np.ndarray        # uint8 [R, H, D/2]
    q_scale: np.ndarray      # uint8 [R, H, D/32]
    k_cache_fp4: np.ndarray  # uint8 [NP, PAGE, D/2]
    k_scale: np.ndarray      # uint8 [NP, PAGE, D/32]
    weights: np.ndarray      # float32 [R, H]
    page_table: np.ndarray   # int32 [NR, MP]
    row_req: np.ndarray      # int32 [R]
    row_start: np.ndarray    # int32 [R]
    row_end: np.ndarray      # int32 [R]
    topk: int
    recipe: str = ""

    @property
    def rows(self) -> int:
        return int(self.q_fp4.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_cache_fp4.shape[0])

    def lengths(self) -> np.ndarray:
        return (self.row_end.astype(np.int64) - self.row_start.astype(np.int64))

    def max_end(self) -> int:
        return int(self.row_end.max()) if self.rows else 0

    def algorithmic_flop(self) -> int:
        """2*H*D per (row, slot) of every row whose window exceeds topk."""
        ln = self.lengths()
        return int(ln[ln > self.topk].sum()) * 2 * H * D

    def scored_pairs(self) -> int:
        ln = self.lengths()
        return int(ln[ln > self.topk].sum())


def _draw_exponents(rng: np.random.Generator, n: int) -> np.ndarray:
    """n rows of N_SF exponents in [-4, 4] with max - min <= 4 per row."""
    e = rng.integers(-4, 5, size=(n, N_SF), dtype=np.int16)
    bad = (e.max(axis=1) - e.min(axis=1)) > 4
    while bad.any():
        idx = np.nonzero(bad)[0]
        e[idx] = rng.integers(-4, 5, size=(idx.size, N_SF), dtype=np.int16)
        bad[idx] = (e[idx].max(axis=1) - e[idx].min(axis=1)) > 4
    return (e + 127).astype(np.uint8)


def _draw_codes(rng: np.random.Generator, n: int) -> np.ndarray:
    """n rows of D/2 bytes; each nibble is uniform over the 16 E2M1 codes."""
    return rng.integers(0, 256, size=(n, D_BYTES), dtype=np.uint8)


def causal_ends(c4_len: int, n_rows: int) -> np.ndarray:
    """Window ends of a request's last n_rows raw tokens (causal C4 rule)."""
    t = 4 * c4_len - n_rows + np.arange(n_rows, dtype=np.int64)
    return ((t + 1) // 4).astype(np.int32)


def make_problem(seed: int, c4_lens: Sequence[int], windows: Sequence[Sequence[tuple]],
                 topk: int, name: str = "custom", page_perm: bool = True,
                 duplicate_slots: int = 0, recipe: str = "") -> Problem:
    """Build a problem with explicit per-request windows.

    c4_lens[i] is request i's C4 length; windows[i] is the list of its rows'
    (start, end) windows in logical C4 positions.  Rows are laid out request by
    request.  duplicate_slots > 0 copies that many distinct logical K slots of
    request 0 onto as many other distinct slots (codes and scales), which
    forces exact score ties.
    """
    rng = np.random.default_rng(seed)
    n_req = len(c4_lens)
    pages_per = [int(math.ceil(L / PAGE)) for L in c4_lens]
    num_pages = max(1, sum(pages_per))
    max_pages = max(1, max(pages_per) if pages_per else 1)

    perm = rng.permutation(num_pages).astype(np.int32) if page_perm else \
        np.arange(num_pages, dtype=np.int32)
    page_table = np.full((max(1, n_req), max_pages), -1, dtype=np.int32)
    off = 0
    for i, n in enumerate(pages_per):
        page_table[i, :n] = perm[off:off + n]
        off += n

    k_codes = _draw_codes(rng, num_pages * PAGE).reshape(num_pages, PAGE, D_BYTES)
    k_sf = _draw_exponents(rng, num_pages * PAGE).reshape(num_pages, PAGE, N_SF)

    row_req, row_start, row_end = [], [], []
    for i, wins in enumerate(windows):
        for (s, e) in wins:
            row_req.append(i)
            row_start.append(s)
            row_end.append(e)
    R = len(row_req)
    q_codes = _draw_codes(rng, R * H).reshape(R, H, D_BYTES)
    q_sf = _draw_exponents(rng, R * H).reshape(R, H, N_SF)
    weights = rng.standard_normal((R, H)).astype(np.float32)

    if duplicate_slots > 0:
        L0 = c4_lens[0]
        picks = rng.choice(L0, size=2 * duplicate_slots, replace=False)
        src, dst = picks[:duplicate_slots], picks[duplicate_slots:]
        for s, d in zip(src, dst):
            ps, pd = page_table[0, s // PAGE], page_table[0, d // PAGE]
            k_codes[pd, d % PAGE] = k_codes[ps, s % PAGE]
            k_sf[pd, d % PAGE] = k_sf[ps, s % PAGE]

    return Problem(name=name, q_fp4=q_codes, q_scale=q_sf, k_cache_fp4=k_codes,
                   k_scale=k_sf, weights=weights, page_table=page_table,
                   row_req=np.asarray(row_req, dtype=np.int32),
                   row_start=np.asarray(row_start, dtype=np.int32),
                   row_end=np.asarray(row_end, dtype=np.int32),
                   topk=int(topk), recipe=recipe)


def causal_problem(seed: int, c4_lens: Sequence[int], rows_per_req: Sequence[int],
                   topk: int, name: str, overrides: Optional[dict] = None,
                   duplicate_slots: int = 0, recipe: str = "") -> Problem:
    """Requests whose rows are their last raw tokens, with causal C4 windows.

    overrides maps (request, row-in-request) -> new window end.
    """
    windows: List[List[tuple]] = []
    for i, (L, n) in enumerate(zip(c4_lens, rows_per_req)):
        ends = causal_ends(L, n)
        w = [(0, int(e)) for e in ends]
        if overrides:
            for (ri, j), e in overrides.items():
                if ri == i:
                    w[j] = (0, int(e))
        windows.append(w)
    return make_problem(seed, c4_lens, windows, topk, name=name,
                        duplicate_slots=duplicate_slots, recipe=recipe)


# --- the five workload configurations -------------------------------------

CONFIG_NAMES = [
    "tiny-R32-S4096-K512",
    "mid-R1024-4req-8k..64k-K512",
    "flash-R8192-S131072-K512",
    "pro-R8192-S196608-K1024",
    "long-R1024-8req-up-to-262144-K1024",
]


def config(idx: int) -> Problem:
    """Workload idx in 0..4 (seed = 20260 + idx)."""
    seed = SEED_BASE + idx
    if idx == 0:
        # one request, C4 length 4096; row r's window is [0, 4065 + r), rows 0
        # and 1 shortened to 100 and 512; 64 duplicated K slots force ties.
        ends = [4065 + r for r in range(32)]
        ends[0], ends[1] = 100, 512
        return make_problem(seed, [4096], [[(0, e) for e in ends]], 512,
                            name=CONFIG_NAMES[0], duplicate_slots=64,
                            recipe="1 request, S=4096, 32 rows, end=4065+r, "
                                   "rows 0/1 -> 100/512, 64 duplicated slots")
    if idx == 1:
        return causal_problem(seed, [8192, 16384, 32768, 65536], [256] * 4, 512,
                              name=CONFIG_NAMES[1],
                              recipe="4 requests x 256 rows, C4 8k/16k/32k/64k, causal")
    if idx == 2:
        return causal_problem(seed, [131072], [8192], 512, name=CONFIG_NAMES[2],
                              recipe="1 request, C4 131072, last 8192 rows, causal")
    if idx == 3:
        return causal_problem(seed, [196608], [8192], 1024, name=CONFIG_NAMES[3],
                              recipe="1 request, C4 196608, last 8192 rows, causal")
    if idx == 4:
        lens = [32768 * (i + 1) for i in range(8)]
        return causal_problem(seed, lens, [128] * 8, 1024, name=CONFIG_NAMES[4],
                              overrides={(0, 0): 0, (0, 1): 1000},
                              recipe="8 requests x 128 rows, C4 32768*(i+1), causal; "
                                     "req0 row0 empty, row1 end=1000")
    raise ValueError(f"no workload {idx}")


def decode_batch(n_req: int = 32, topk: int = 512, lo: int = 4096, hi: int = 65536,
                 seed: int = 5) -> Problem:
    """A decode-shaped batch: n_req requests whose C4 lengths L are drawn
    uniformly from [lo, hi), two query rows each (a decode step with one
    speculative token: windows [0, L - 1) and [0, L))."""
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(lo, hi, size=n_req)]
    return make_problem(seed, lens, [[(0, L - 1), (0, L)] for L in lens], topk,
                        name=f"decode-{n_req}x2-K{topk}",
                        recipe=f"{n_req} requests x 2 rows, C4 uniform in [{lo}, {hi}), "
                               f"windows [0, L-1) and [0, L)")


def k_scale_mma_order(k_scale: np.ndarray) -> np.ndarray:
    """A [NP, 64, 4] K-scale array rearranged (a pure permutation of bytes) into
    the [NP, 256] order of idx_topk_fp4_prefill_mma_scales: byte 8j + 4h + b of
    a page holds scale b of slot 32h + j."""
    npg = k_scale.shape[0]
    return np.ascontiguousarray(
        np.asarray(k_scale).reshape(npg, 2, 32, 4).transpose(0, 2, 1, 3).reshape(npg, 256))


def small_problem(seed: int = 7, topk: int = 512, c4_lens=(1500, 2600, 700),
                  rows_per_req=(5, 9, 3), start_offsets=True) -> Problem:
    """A small ragged multi-request case the oracle finishes in well under a second.

    Windows have nonzero starts for some rows when start_offsets is set, so
    ragged heads and tails of pages and tiles are both exercised.
    """
    rng = np.random.default_rng(seed + 1000)
    windows = []
    for L, n in zip(c4_lens, rows_per_req):
        ends = causal_ends(L, n)
        w = []
        for e in ends:
            s = int(rng.integers(0, max(1, int(e) // 3))) if start_offsets else 0
            w.append((s, int(e)))
        windows.append(w)
    return make_problem(seed, list(c4_lens), windows, topk, name=f"small-{seed}")
