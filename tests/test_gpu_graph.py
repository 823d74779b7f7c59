"""CUDA-graph capture of the decode call.

The split schedule is computed on the device from ``seq_lens`` at every launch, and the
call neither allocates nor synchronises, so one capture serves later replays whose query
values and sequence lengths (up to the ``max_seq_len`` it was captured with) were written
in place. Each replay is compared with the float64 oracle on the inputs of that replay.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from gpu_harness import GpuCase, bits_to_torch_bf16, compare, oracle_decode
from mla_paged_decode_02_gb300 import api, synth

pytestmark = pytest.mark.gpu

BF, F8 = synth.KV_BF16, synth.KV_FP8_E4M3

# lengths at capture, then shorter ones written in place before the second replay (one
# sequence drops to a single key; the longest ones are split over several workers)
LENS_A = [4000, 130, 2500, 9000]
LENS_B = [3100, 129, 1, 8192]


@pytest.mark.parametrize("H,P,kv", [(16, 64, BF), (16, 64, F8), (128, 128, BF), (128, 64, F8)])
def test_one_capture_serves_new_queries_and_lengths(H, P, kv):
    case = synth.make_case(B=4, s_q=1, H=H, page_size=P, seq_lens=LENS_A, seed=71 + H, kv_dtype=kv)
    g = GpuCase(case)
    out0, lse0 = [t.clone() for t in g.decode()]   # eager: sets the kernels up once
    torch.cuda.synchronize()
    out = torch.full_like(out0, float("nan"))
    lse = torch.full_like(lse0, float("nan"))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        g.decode(out=out, lse=lse)
    torch.cuda.current_stream().wait_stream(side)

    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, out0) and torch.equal(lse, lse0)
    st, bits = api.decode_check(g.workspace)
    assert st == 0 and bits == 0

    q_new = synth.normal_bf16(np.random.default_rng(72 + H), case.q_bits.shape)
    g.q.copy_(bits_to_torch_bf16(q_new))
    g.seq_lens.copy_(torch.tensor(LENS_B, dtype=torch.int32))
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    st, bits = api.decode_check(g.workspace)
    assert st == 0 and bits == 0
    case_b = dataclasses.replace(case, q_bits=q_new, seq_lens=np.asarray(LENS_B, dtype=np.int32))
    ro, rl = oracle_decode(case_b, g.cache_numpy())
    compare(case_b, out, lse, ro, rl)
