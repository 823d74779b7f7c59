"""The fused cache-write + decode call: a decode step's new tokens are written into the paged
cache by extra CTAs of the scheduler's launch and attended in the same launch chain. The cache must equal the oracle's cache write
bit for bit and the output the oracle's decode of that cache."""
import numpy as np
import pytest
import torch

from gpu_harness import GpuCase, bits_to_torch_bf16, compare, oracle_decode
from mla_paged_decode_02_gb300 import api, synth
from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu
BF, F8 = synth.KV_BF16, synth.KV_FP8_E4M3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.lib()


def fused_step(case, new_idx):
    """Cache holding every token except `new_idx` (written by the separate cache write),
    then the fused call writes `new_idx` and decodes."""
    g = GpuCase(case, build_cache=False)
    g.cache = g.empty_cache()
    old = np.setdiff1d(np.arange(case.num_tokens), new_idx)
    dev = lambda bits: bits_to_torch_bf16(bits, "cuda")
    api.cache_write(dev(case.latent_bits[old]), dev(case.rope_bits[old]),
                    torch.from_numpy(case.slot_mapping[old]).cuda(), g.cache, g.kv_scale)
    out, lse = api.decode_with_cache_write(
        dev(case.latent_bits[new_idx]), dev(case.rope_bits[new_idx]),
        torch.from_numpy(case.slot_mapping[new_idx]).cuda(), g.q, g.cache, g.block_table, g.seq_lens,
        case.softmax_scale, g.kv_scale, max_seq_len=case.max_seq_len, causal=case.causal,
        workspace=g.workspace)
    torch.cuda.synchronize()
    return g, out, lse


@pytest.mark.parametrize("kv", [BF, F8])
@pytest.mark.parametrize("B,s_q,H,lens", [(4, 1, 16, [100, 2000, 129, 64]), (3, 4, 128, [300, 1000, 5]),
                                          (2, 64, 16, [3000, 4000])])
def test_fused_cache_write_and_decode(kv, B, s_q, H, lens):
    case = synth.make_case(B=B, s_q=s_q, H=H, page_size=64, seq_lens=lens, seed=80 + B + s_q, kv_dtype=kv)
    g, out, lse = fused_step(case, case.step_tokens())
    assert api.decode_check(g.workspace) == (0, 0)
    ref_cache = O.cache_write(case.empty_cache(), case.latent_bits, case.rope_bits, case.slot_mapping,
                              case.page_size, kv, case.kv_scale)
    cache = g.cache_numpy()
    assert np.array_equal(cache, ref_cache)
    ro, rl = oracle_decode(case, cache)
    compare(case, out, lse, ro, rl)


def test_a_whole_batch_written_by_the_fused_call():
    """Every token of the batch as new tokens (the write then needs 128 extra CTAs' strides)."""
    case = synth.make_case(B=2, s_q=1, H=16, page_size=64, seq_lens=[3000, 2500], seed=85, kv_dtype=F8)
    g, out, lse = fused_step(case, np.arange(case.num_tokens))
    assert api.decode_check(g.workspace) == (0, 0)
    ref_cache = O.cache_write(case.empty_cache(), case.latent_bits, case.rope_bits, case.slot_mapping,
                              case.page_size, F8, case.kv_scale)
    assert np.array_equal(g.cache_numpy(), ref_cache)
    ro, rl = oracle_decode(case, g.cache_numpy())
    compare(case, out, lse, ro, rl)


@pytest.mark.parametrize("n_new", [3, 6000])
def test_a_slot_outside_the_pool_is_reported(n_new):
    case = synth.make_case(B=2, s_q=1, H=16, page_size=64, seq_lens=[4000, 3000], seed=86)
    g = GpuCase(case)
    idx = np.arange(n_new)
    slots = torch.from_numpy(case.slot_mapping[idx].copy()).cuda()
    slots[1] = case.num_pages * case.page_size + 3
    dev = lambda bits: bits_to_torch_bf16(bits, "cuda")
    api.decode_with_cache_write(dev(case.latent_bits[idx]), dev(case.rope_bits[idx]), slots, g.q, g.cache,
                                g.block_table, g.seq_lens, case.softmax_scale, max_seq_len=case.max_seq_len,
                                workspace=g.workspace)
    st, bits = api.decode_check(g.workspace)
    assert st == -6 and bits & 0x10
