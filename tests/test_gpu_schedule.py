"""The split scheduler's partition, read back from the workspace after a decode.

The scheduler lays the (row group, sequence) streams of key tiles end to end and gives
CTA c the positions [c q, (c + 1) q), q = ceil(W / grid); when the G row groups divide the
grid, each group gets grid / G CTAs and the same partition of its N tiles instead
(q = ceil(N / (grid / G))). With more than 64 rows the workers are CTA pairs
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


CASES = [
    (2, 1, 16, 64, [100, 257]),
    (4, 1, 16, 64, [5000, 17, 640, 2049]),
    (3, 4, 128, 64, [1000, 67, 3000]),
    (2, 1, 128, 128, [300, 1000]),
    (2, 2, 128, 64, [4000, 70]),
    (3, 1, 96, 64, [500, 129, 20000]),
    (1, 1, 16, 64, [131072]),
    (300, 1, 16, 64, (1, 700)),
]


@pytest.mark.parametrize("B,s_q,H,P,lens", CASES)
def test_partition_is_exact_and_balanced(B, s_q, H, P, lens):
    case = synth.make_case(B=B, s_q=s_q, H=H, page_size=P, seq_lens=lens, seed=71 + B)
    g = GpuCase(case)
    g.decode()
    torch.cuda.synchronize()
    R = s_q * H
    _, tile, grid = _plan(R, torch.cuda.get_device_properties(0).multi_processor_count)
    rc, G, cta_off, split_off, units_off = _offsets(B, R, grid)
    ws = g.workspace.cpu().numpy().view(np.uint8)
    hdr = ws[:16].view(np.uint32)
    n_units, n_split, q = int(hdr[1]), int(hdr[2]), int(hdr[3])
    assert hdr[0] == 0
    cta_first = ws[cta_off:cta_off + 4 * (grid + 1)].view(np.int32)
    units = ws[units_off:units_off + 16 * n_units].view(np.int32).reshape(n_units, 4)
    splits = ws[split_off:split_off + 16 * n_split].view(np.int32).reshape(n_split, 4)

    n_b = (case.seq_lens.astype(np.int64) + tile - 1) // tile
    N = int(n_b.sum())
    W = G * N
    aligned = G > 1 and grid % G == 0
    cpg = grid // G if aligned else grid
    assert q == (-(-N // cpg) if aligned else -(-W // grid))
    assert cta_first[grid] == n_units and np.all(np.diff(cta_first) >= 0)
    tb = units[:, 2] & 0xFFFF
    te = units[:, 2] >> 16
    assert np.all(te > tb)
    for c in range(grid):
        cc, total = (c % cpg, N) if aligned else (c, W)
        share = max(0, min((cc + 1) * q, total) - cc * q)
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
