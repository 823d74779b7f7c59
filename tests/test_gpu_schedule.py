"""The split scheduler's partition, read back from the workspace after a decode.

The scheduler lays the (row group, sequence) streams end to end, each X positions for a
unit's set-up followed by one position per key tile, and gives CTA c the tiles among the
positions [c q, (c + 1) q), q = ceil(W / grid); when the G row groups divide the grid, each
group gets grid / G CTAs and the same partition of its N positions instead
(q = ceil(N / (grid / G))). X (header word 4) is 0 when q would be at most 2 X. With more than 64 rows the workers are CTA pairs
(grid = #SM / 2), a row group is 128 rows and a tile 256 keys. Checked here on the device's own output: every tile of every
stream is covered exactly once, every CTA's units are a contiguous range holding exactly
its share of tiles, and only streams cut by a CTA boundary get partial slots (consecutive
ones). The workspace offsets below restate the
layout the library documents for its workspace (header, batch info, per-CTA first unit,
cut streams, units), 256-byte aligned.
"""
import numpy as np
import pytest
import torch

from gpu_harness import GpuCase
from mla_paged_decode_02_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _plan(R, nsm):
    """(rows per group, keys per tile, schedule workers) for R rows (either cache type)."""
    if R > 64:
        return 128, 256, nsm // 2
    return (16 if R <= 16 else 32 if R <= 32 else 64), 128, nsm


def _offsets(B, R, grid):
    rc = _plan(R, 2 * grid)[0]
    G = -(-R // rc)
    al = lambda x: (x + 255) // 256 * 256
    off = 256
    batch = off
    off = al(off + 16 * B)
    cta = off
    off = al(off + 4 * (grid + 1))
    split = off
    off = al(off + 16 * grid)
    units = off
    return rc, G, cta, split, units


BF, F8 = synth.KV_BF16, synth.KV_FP8_E4M3
CASES = [
    (2, 1, 16, 64, [100, 257], BF),
    (4, 1, 16, 64, [5000, 17, 640, 2049], BF),
    (3, 4, 128, 64, [1000, 67, 3000], BF),
    (2, 1, 128, 128, [300, 1000], BF),
    (2, 2, 128, 64, [4000, 70], BF),
    (3, 1, 96, 64, [500, 129, 20000], BF),
    (1, 1, 16, 64, [131072], BF),
    (300, 1, 16, 64, (1, 700), BF),
    (4, 1, 16, 64, [5000, 17, 640, 2049], F8),    # a set-up charge of 4 per stream
    (300, 1, 16, 64, (1, 700), F8),
    (2, 1, 16, 64, [100, 257], F8),               # shares too small for it: dropped
    (3, 1, 128, 64, [1500, 130, 9000], F8),
]


@pytest.mark.parametrize("B,s_q,H,P,lens,kv", CASES)
def test_partition_is_exact_and_balanced(B, s_q, H, P, lens, kv):
    case = synth.make_case(B=B, s_q=s_q, H=H, page_size=P, seq_lens=lens, seed=71 + B, kv_dtype=kv)
    g = GpuCase(case)
    g.decode()
    torch.cuda.synchronize()
    R = s_q * H
    _, tile, grid = _plan(R, torch.cuda.get_device_properties(0).multi_processor_count)
    rc, G, cta_off, split_off, units_off = _offsets(B, R, grid)
    ws = g.workspace.cpu().numpy().view(np.uint8)
    hdr = ws[:32].view(np.uint32)
    n_units, n_split, q, X = int(hdr[1]), int(hdr[2]), int(hdr[3]), int(hdr[4])
    assert hdr[0] == 0
    cta_first = ws[cta_off:cta_off + 4 * (grid + 1)].view(np.int32)
    units = ws[units_off:units_off + 16 * n_units].view(np.int32).reshape(n_units, 4)
    splits = ws[split_off:split_off + 16 * n_split].view(np.int32).reshape(n_split, 4)

    n_b = (case.seq_lens.astype(np.int64) + tile - 1) // tile
    aligned = G > 1 and grid % G == 0
    cpg = grid // G if aligned else grid
    qs = lambda x: -(-(int(n_b.sum()) + B * x) // cpg) if aligned else -(-G * (int(n_b.sum()) + B * x) // grid)
    # charged per stream: 2 for bf16 CTA pairs, 3 for FP8 pairs, 4 for the FP8 cache and 0 for
    # bf16 up to 64 rows,
    # dropped when a CTA's share would be at most twice that
    fp8 = case.kv_dtype == synth.KV_FP8_E4M3
    want = (3 if fp8 else 2) if R > 64 else (4 if fp8 else 0)
    assert X == (want if qs(want) > 2 * want else 0)
    N = int(n_b.sum()) + B * X                       # positions of one row group
    W = G * N
    assert q == qs(X)
    # every stream's tiles as an interval of positions
    starts = np.concatenate([[0], np.cumsum(n_b + X)[:-1]])
    tiles_of = {(b, gg): ((0 if aligned else gg * N) + int(starts[b]) + X, int(n_b[b]))
                for b in range(B) for gg in range(G)}
    assert cta_first[grid] == n_units and np.all(np.diff(cta_first) >= 0)
    tb = units[:, 2] & 0xFFFF
    te = units[:, 2] >> 16
    assert np.all(te > tb)
    for c in range(grid):
        cc = c % cpg if aligned else c
        lo, hi = cc * q, (cc + 1) * q
        share = sum(max(0, min(hi, t0 + n) - max(lo, t0)) for (b, gg), (t0, n) in tiles_of.items()
                    if not aligned or gg == c // cpg)
        sl = slice(cta_first[c], cta_first[c + 1])
        assert int((te[sl] - tb[sl]).sum()) == share, c
        if aligned:
            assert np.all(units[sl, 1] == c // cpg), c          # one row group per CTA block
    cover = {}
    for (b, gg, _, slot), s0, s1 in zip(units, tb, te):
        cover.setdefault((int(b), int(gg)), []).append((int(s0), int(s1), int(slot)))
    assert set(cover) == {(b, gg) for b in range(B) for gg in range(G)}
    cut = {}
    for (b, gg), pieces in cover.items():
        pieces.sort()
        assert pieces[0][0] == 0 and pieces[-1][1] == n_b[b]
        assert all(p[1] == nx[0] for p, nx in zip(pieces, pieces[1:]))
        slots = [p[2] for p in pieces]
        if len(pieces) == 1:
            assert slots == [-1]
        else:
            assert slots == list(range(slots[0], slots[0] + len(slots)))
            cut[(b, gg)] = (len(pieces), slots[0])
    assert {(int(b), int(gg)): (int(ns), int(s0)) for b, gg, ns, s0 in splits} == cut
    assert len(cut) <= grid - 1
