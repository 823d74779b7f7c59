"""Pins for the float64 decode oracle (oracle/mla_oracle.py).

Each check uses something other than the oracle itself: a pure-Python loop decode that
addresses the cache token by token, torch's scaled_dot_product_attention on a dense
gather built with torch indexing, and invariants of softmax attention. The cases are
chosen so that a dropped term (the 64 rope columns, the scale), a sign error, a wrong
page/offset index or a transposed operand fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden
from mla_paged_decode_02_gb300 import synth
from oracle import fp8_e4m3
from oracle import mla_oracle as O


def build_cache(case):
    return O.cache_write(case.empty_cache(), case.latent_bits, case.rope_bits,
                         case.slot_mapping, case.page_size, case.kv_dtype, case.kv_scale)


def run_oracle(case, cache=None, **kw):
    cache = build_cache(case) if cache is None else cache
    return O.mla_decode(case.q_bits, cache, case.block_table, case.seq_lens, case.page_size,
                        case.softmax_scale, case.kv_dtype, case.kv_scale, case.causal, **kw)


# ------------------------------------------------------------------ brute force
def bf16_to_float(u):
    return float(np.array([int(u) << 16], dtype=np.uint32).view(np.float32)[0])


def brute_force_decode(case, cache):
    """Pure-Python loops: token j of sequence b is read at page block_table[b][j//P],
    row j%P; every dot product, exponential and sum is a Python float operation."""
    P = case.page_size
    out = {}
    for b in range(case.B):
        L = int(case.seq_lens[b])
        keys = []
        for j in range(L):
            page = int(case.block_table[b][j // P])
            row = cache[page, j % P]
            if case.kv_dtype == O.KV_BF16:
                keys.append([bf16_to_float(v) for v in row])
            else:
                keys.append([float(fp8_e4m3.DECODE_TABLE[int(v)]) * case.kv_scale for v in row])
        for i in range(case.s_q):
            n = L - case.s_q + 1 + i if case.causal else L
            for h in range(case.H):
                qv = [bf16_to_float(v) for v in case.q_bits[b, i, h]]
                s = [math.fsum(qv[d] * keys[j][d] for d in range(576)) * case.softmax_scale
                     for j in range(n)]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                tot = math.fsum(e)
                o = [math.fsum(e[j] * keys[j][d] for j in range(n)) / tot for d in range(512)]
                out[(b, i, h)] = (o, m + math.log(tot))
    return out


@pytest.mark.parametrize("kind", ["config1", "causal_sq3", "fp8_noncausal"])
def test_oracle_matches_pure_python_brute_force(kind):
    if kind == "config1":
        case = synth.make_config(1)
    elif kind == "causal_sq3":
        case = synth.make_case(B=2, s_q=3, H=2, page_size=64, seq_lens=[5, 70], seed=7)
    else:
        case = synth.make_case(B=1, s_q=2, H=3, page_size=64, seq_lens=[90], seed=8,
                               kv_dtype=O.KV_FP8_E4M3, causal=False)
    cache = build_cache(case)
    out, lse = run_oracle(case, cache)
    ref = brute_force_decode(case, cache)
    for (b, i, h), (o, l) in ref.items():
        assert np.allclose(out[b, i, h], o, rtol=0, atol=1e-12), (b, i, h)
        assert abs(lse[b, i, h] - l) < 1e-12


# ------------------------------------------------------------------ library case
def sdpa_reference(case, cache):
    """torch float64 SDPA (MQA by expanding the one KV head) over a dense gather
    done with torch indexing of the flattened pool by slot number."""
    P = case.page_size
    pool = torch.from_numpy(O.dequant_rows(cache.reshape(-1, 576), case.kv_dtype, case.kv_scale))
    outs, lses = [], []
    for b in range(case.B):
        L = int(case.seq_lens[b])
        j = torch.arange(L)
        slots = torch.from_numpy(case.block_table[b].astype(np.int64))[j // P] * P + j % P
        K = pool[slots]                                   # [L, 576]
        V = K[:, :512]
        q = torch.from_numpy(O.bf16_bits_to_f64(case.q_bits[b]))     # [s_q, H, 576]
        qh = q.permute(1, 0, 2)                                       # [H, s_q, 576]
        mask = torch.ones(case.s_q, L, dtype=torch.bool)
        if case.causal:
            mask = j[None, :] <= (L - case.s_q + torch.arange(case.s_q))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(
            qh[None], K.expand(case.H, L, 576)[None], V.expand(case.H, L, 512)[None],
            attn_mask=mask, scale=case.softmax_scale)[0]              # [H, s_q, 512]
        s = (qh @ K.T) * case.softmax_scale
        s = s.masked_fill(~mask[None], float("-inf"))
        outs.append(o.permute(1, 0, 2).numpy())
        lses.append(torch.logsumexp(s, dim=-1).permute(1, 0).numpy())
    return np.stack(outs), np.stack(lses)


@pytest.mark.parametrize("B,s_q,H,P,lens,kv,causal", [
    (2, 1, 16, 64, [100, 257], O.KV_BF16, True),
    (3, 4, 8, 64, [4, 129, 300], O.KV_BF16, True),
    (2, 2, 4, 128, [130, 256], O.KV_FP8_E4M3, True),
    (2, 3, 4, 64, [64, 65], O.KV_BF16, False),
])
def test_oracle_matches_torch_sdpa(B, s_q, H, P, lens, kv, causal):
    case = synth.make_case(B=B, s_q=s_q, H=H, page_size=P, seq_lens=lens, seed=11,
                           kv_dtype=kv, causal=causal)
    cache = build_cache(case)
    out, lse = run_oracle(case, cache)
    ro, rl = sdpa_reference(case, cache)
    assert np.allclose(out, ro, rtol=0, atol=1e-10)
    assert np.allclose(lse, rl, rtol=0, atol=1e-10)


# ------------------------------------------------------------------ invariants
def test_attention_weights_sum_to_one_and_are_positive():
    case = synth.make_case(B=1, s_q=2, H=4, page_size=64, seq_lens=[200], seed=3)
    K = O.gather_sequence(build_cache(case), case.block_table[0], 200, 64, O.KV_BF16, None)
    q = O.bf16_bits_to_f64(case.q_bits[0, 1])
    _, _, w = O.attend(q, K, case.softmax_scale)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-14) and (w > 0).all()


def test_constant_value_cache_returns_that_value():
    case = synth.make_case(B=2, s_q=2, H=4, page_size=64, seq_lens=[77, 300], seed=4)
    case.latent_bits[:] = case.latent_bits[0]
    case.rope_bits[:] = case.rope_bits[0]
    out, _ = run_oracle(case)
    v = O.bf16_bits_to_f64(case.latent_bits[0])
    assert np.allclose(out, np.broadcast_to(v, out.shape), atol=1e-13)


def test_single_token_sequence():
    case = synth.make_case(B=1, s_q=1, H=5, page_size=64, seq_lens=[1], seed=5)
    out, lse = run_oracle(case)
    k = np.concatenate([O.bf16_bits_to_f64(case.latent_bits[0]), O.bf16_bits_to_f64(case.rope_bits[0])])
    q = O.bf16_bits_to_f64(case.q_bits[0, 0])
    assert np.array_equal(out[0, 0], np.broadcast_to(k[:512], (5, 512)))
    assert np.allclose(lse[0, 0], (q @ k) * case.softmax_scale, atol=1e-12)


def test_rope_columns_enter_the_scores_but_not_the_output():
    """Changing only the rope part of the cache changes scores (lse); changing q's rope
    part too. The output is a mix of the 512 latent columns only."""
    case = synth.make_case(B=1, s_q=1, H=3, page_size=64, seq_lens=[50], seed=6)
    out0, lse0 = run_oracle(case)
    case.rope_bits[:] = synth.f32_to_bf16_bits(np.zeros_like(O.bf16_bits_to_f32(case.rope_bits)))
    out1, lse1 = run_oracle(case)
    assert np.abs(lse1 - lse0).max() > 1e-3
    # with a zero rope the scores are q_latent . k_latent exactly
    cache = build_cache(case)
    K = O.gather_sequence(cache, case.block_table[0], 50, 64, O.KV_BF16, None)
    q = O.bf16_bits_to_f64(case.q_bits[0, 0])
    s = (q[:, :512] @ K[:, :512].T) * case.softmax_scale
    ref = np.log(np.exp(s).sum(axis=1))
    assert np.allclose(lse1[0, 0], ref, atol=1e-12)


def test_physical_page_permutation_leaves_output_unchanged():
    case = synth.make_case(B=3, s_q=2, H=4, page_size=64, seq_lens=[70, 200, 129], seed=9)
    cache = build_cache(case)
    out0, lse0 = run_oracle(case, cache)
    rng = np.random.default_rng(99)
    perm = rng.permutation(case.num_pages)            # old page p -> new page perm[p]
    cache2 = np.empty_like(cache)
    cache2[perm] = cache
    case.block_table = perm[case.block_table].astype(np.int32)
    out1, lse1 = run_oracle(case, cache2)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_unused_pages_and_tails_are_never_read():
    case = synth.make_case(B=2, s_q=1, H=4, page_size=64, seq_lens=[70, 129], seed=10)
    cache = build_cache(case)
    out0, lse0 = run_oracle(case, cache)
    assert np.isnan(O.bf16_bits_to_f64(cache)).any()   # tails and the spare page are NaN
    clean = cache.copy()
    clean[np.isnan(O.bf16_bits_to_f64(clean))] = 0
    out1, lse1 = run_oracle(case, clean)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)
    assert np.isfinite(out0).all() and np.isfinite(lse0).all()


@pytest.mark.parametrize("cuts", [[0, 1, 300], [0, 128, 256, 300], [0, 17, 18, 250, 300], [0, 299, 300]])
def test_split_kv_with_lse_combine_equals_single_pass(cuts):
    case = synth.make_case(B=1, s_q=1, H=6, page_size=64, seq_lens=[300], seed=12)
    K = O.gather_sequence(build_cache(case), case.block_table[0], 300, 64, O.KV_BF16, None)
    q = O.bf16_bits_to_f64(case.q_bits[0, 0])
    full_o, full_l, _ = O.attend(q, K, case.softmax_scale)
    parts = [O.attend_range(q, K, a, b, case.softmax_scale) for a, b in zip(cuts[:-1], cuts[1:])]
    parts.append(O.attend_range(q, K, 300, 300, case.softmax_scale))     # an empty split
    o, l = O.lse_combine([p[0] for p in parts], [p[1] for p in parts])
    assert np.allclose(o, full_o, atol=1e-12) and np.allclose(l, full_l, atol=1e-12)


def test_scaling_q_equals_scaling_softmax_scale_and_sharpens_to_argmax():
    case = synth.make_case(B=1, s_q=1, H=4, page_size=64, seq_lens=[120], seed=13)
    cache = build_cache(case)
    K = O.gather_sequence(cache, case.block_table[0], 120, 64, O.KV_BF16, None)
    q = O.bf16_bits_to_f64(case.q_bits[0, 0])
    o2, l2, _ = O.attend(2.0 * q, K, case.softmax_scale)
    o2b, l2b, _ = O.attend(q, K, 2.0 * case.softmax_scale)
    assert np.allclose(o2, o2b, atol=1e-13) and np.allclose(l2, l2b, atol=1e-12)
    # lse(c) is convex and increasing for c>0 once the max score is positive
    ls = [O.attend(c * q, K, case.softmax_scale)[1] for c in (1.0, 2.0, 4.0)]
    assert (ls[1] > ls[0]).all() and (ls[2] > ls[1]).all()
    # a very sharp softmax returns the value row of the arg-max score
    s = q @ K.T
    o, _, _ = O.attend(q, K, 200.0)
    for h in range(4):
        srt = np.sort(s[h])
        if (srt[-1] - srt[-2]) * 200.0 > 50:
            assert np.allclose(o[h], K[np.argmax(s[h]), :512], atol=1e-9)


def test_causal_rows_see_the_right_number_of_keys():
    """Row i of s_q new tokens attends to L - s_q + 1 + i keys: replacing the keys it
    must not see with huge values changes nothing for it."""
    case = synth.make_case(B=1, s_q=3, H=2, page_size=64, seq_lens=[66], seed=14)
    cache = build_cache(case)
    out0, _ = run_oracle(case, cache)
    K = O.gather_sequence(cache, case.block_table[0], 66, 64, O.KV_BF16, None)
    q = O.bf16_bits_to_f64(case.q_bits[0])
    for i in range(3):
        n = 66 - 3 + 1 + i
        o, _, _ = O.attend(q[i], K[:n], case.softmax_scale)
        assert np.allclose(out0[0, i], o, atol=1e-14)
        if n < 66:
            o_more, _, _ = O.attend(q[i], K[:n + 1], case.softmax_scale)
            assert not np.allclose(out0[0, i], o_more, atol=1e-6)


# ------------------------------------------------------------------ cache write
def test_cache_write_places_rows_at_their_slots_and_skips_negative_slots():
    case = synth.make_case(B=2, s_q=1, H=1, page_size=64, seq_lens=[10, 70], seed=15)
    slots = case.slot_mapping.copy()
    slots[3] = -1
    cache = O.cache_write(case.empty_cache(), case.latent_bits, case.rope_bits, slots, 64, O.KV_BF16)
    for t, s in enumerate(slots):
        row = cache.reshape(-1, 576)[s] if s >= 0 else None
        if s < 0:
            continue
        assert np.array_equal(row[:512], case.latent_bits[t]) and np.array_equal(row[512:], case.rope_bits[t])
    s3 = case.slot_mapping[3]
    assert (cache.reshape(-1, 576)[s3] == synth.BF16_NAN_BITS).all()


def test_fp8_cache_write_matches_torch_quantisation_in_range():
    case = synth.make_case(B=2, s_q=1, H=1, page_size=64, seq_lens=[33, 64], seed=16,
                           kv_dtype=O.KV_FP8_E4M3)
    cache = build_cache(case)
    rows = np.concatenate([case.latent_bits, case.rope_bits], axis=1)
    x = torch.from_numpy(O.bf16_bits_to_f32(rows))
    q = (x / torch.tensor(case.kv_scale, dtype=torch.float32))       # all |q| <= 448 by the scale choice
    assert float(q.abs().max()) <= 448.0
    ref = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = cache.reshape(-1, 576)[case.slot_mapping]
    assert np.array_equal(got, ref)
    # the largest magnitude maps to +-448 exactly
    assert (np.abs(fp8_e4m3.decode(got)) == 448.0).any()


# ------------------------------------------------------------------ the metric
def test_cos_diff_closed_forms_and_the_logged_failure_value():
    params = dict(read_golden("kernel_test_params.txt"))
    x = np.random.default_rng(0).standard_normal(1000)
    assert O.cos_diff(x, x) == pytest.approx(0.0, abs=1e-15)
    assert O.cos_diff(x, 2 * x) == pytest.approx(1 - 4 / 5, abs=1e-15)
    assert O.cos_diff(x, -x) == pytest.approx(2.0, abs=1e-15)
    # an all-zero output gives exactly the value printed in the failing test log
    assert O.cos_diff(x, np.zeros_like(x)) == float(params["cos_diff_failure_value"])
    assert O.cos_diff(np.zeros(4), np.zeros(4)) == 1.0


def test_flops_closed_form():
    assert O.flops([100, 257], 1, 16) == 2 * 1088 * 16 * 357
    # causal s_q=4: rows see L-3, L-2, L-1, L keys
    assert O.flops([10], 4, 2) == 2 * 1088 * 2 * (7 + 8 + 9 + 10)
    params = dict(read_golden("kernel_test_params.txt"))
    assert int(params["d"]) == O.D_QK and int(params["dv"]) == O.D_V
