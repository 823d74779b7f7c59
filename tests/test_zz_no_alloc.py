"""mla_decode_noalloc: the decode for callers that cannot allocate device memory (an
engine plugin that is handed only inputs and outputs, or a runtime that owns all device
memory and forbids cudaMalloc). It uses the library's static scratch array instead of a
caller workspace; its results must match mla_decode's.

This file is collected last on purpose, so that a run stopping at the first failure has
already run every other test. It passes alone in a fresh process (the first call looks up
the scratch array's address) and after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_harness import BF16_MAX_ABS, BF16_REL_L2, LSE_ABS, GpuCase
from mla_paged_decode_02_gb300 import api, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.lib()


def outputs(c):
    out = torch.full((c.B, c.s_q, c.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((c.B, c.s_q, c.H), float("nan"), dtype=torch.float32, device="cuda")
    return out, lse


def call_noalloc(g, out=None, lse=None):
    """One call through the C ABI entry point itself (into out, lse when given)."""
    c = g.case
    if out is None:
        out, lse = outputs(c)
    st = api.lib().mla_decode_noalloc(
        ctypes.byref(g.params), ctypes.c_void_p(g.q.data_ptr()), ctypes.c_void_p(g.cache.data_ptr()),
        ctypes.c_void_p(g.block_table.data_ptr()), ctypes.c_void_p(g.seq_lens.data_ptr()),
        ctypes.c_float(c.softmax_scale),
        ctypes.c_void_p(g.kv_scale.data_ptr()) if g.kv_scale is not None else None,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, api.status_string(st)
    return out, lse


def close(a_out, a_lse, b_out, b_lse):
    x = a_out.double().cpu().numpy()
    y = b_out.double().cpu().numpy()
    assert np.isfinite(x).all()
    assert np.abs(x - y).max() <= BF16_MAX_ABS
    assert np.linalg.norm(x - y) <= BF16_REL_L2 * np.linalg.norm(y)
    assert (a_lse - b_lse).abs().max().item() <= LSE_ABS


def test_noalloc_matches_mla_decode_on_two_calls_in_a_row():
    cases = [synth.make_case(B=6, s_q=1, H=16, page_size=64, seq_lens=(200, 4000), seed=71),
             synth.make_case(B=3, s_q=1, H=16, page_size=128, seq_lens=[3000, 90, 1500], seed=72,
                             kv_dtype=synth.KV_FP8_E4M3)]
    for g in cases:   # both fit the static scratch (row groups of 16 on this GPU)
        p = api.make_params(g.B, g.s_q, g.H, g.page_size, g.num_pages, g.max_blocks, g.max_seq_len,
                            g.kv_dtype, g.causal)
        assert api.lib().mla_decode_workspace_size(ctypes.byref(p), 0) <= api.NOALLOC_SCRATCH_BYTES
    gs = [GpuCase(c) for c in cases]
    refs = [[t.clone() for t in g.decode()] for g in gs]       # the existing entry point
    got = [call_noalloc(g) for g in gs]                          # two no-alloc calls in a row
    torch.cuda.synchronize()
    for (ro, rl), (o, l) in zip(refs, got):
        close(o, l, ro, rl)
    # a third call repeating the first: leftover scratch of the second does not matter
    o, l = call_noalloc(gs[0])
    torch.cuda.synchronize()
    close(o, l, refs[0][0], refs[0][1])
    assert api.decode_noalloc_check() == (0, 0)          # no device-side error


def test_a_warm_call_allocates_no_device_memory():
    g = GpuCase(synth.make_case(B=4, s_q=1, H=16, page_size=64, seq_lens=(100, 3000), seed=73))
    out, lse = outputs(g.case)
    call_noalloc(g, out, lse)                             # first call on the device: set-up
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    call_noalloc(g, out, lse)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0
    assert api.decode_noalloc_check() == (0, 0)


def test_noalloc_reports_a_block_table_entry_outside_the_pool():
    g = GpuCase(synth.make_case(B=2, s_q=1, H=16, page_size=64, seq_lens=[100, 200], seed=74))
    g.block_table[1, 2] = g.case.num_pages + 5
    call_noalloc(g)
    st, bits = api.decode_noalloc_check()
    assert st == -6 and bits & 0x1
    g.block_table[1, 2] = int(g.case.block_table[1, 2])   # a valid table: the word is clean again
    call_noalloc(g)
    assert api.decode_noalloc_check() == (0, 0)


def test_noalloc_refuses_work_beyond_its_scratch():
    p = api.make_params(512, 4, 128, 64, 100000, 4096, 1 << 18, api.KV_BF16)
    assert api.lib().mla_decode_workspace_size(ctypes.byref(p), 0) > api.NOALLOC_SCRATCH_BYTES
    vp = ctypes.c_void_p(1 << 20)
    st = api.lib().mla_decode_noalloc(ctypes.byref(p), vp, vp, vp, vp, ctypes.c_float(0.1), None,
                                      vp, vp, None)
    assert st == -3
