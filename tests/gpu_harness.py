"""Shared helpers for the GPU parity tests: upload a synth case, build the cache with the
library's cache write, decode through the C ABI, and compare with the float64 oracle.

Tolerances (the decode contract): bf16 cache — every element |err| <= 2e-2 and relative
L2 <= 5e-3; FP8 cache (against the oracle on the same dequantised bytes) — relative L2
<= 1e-2 and cos_diff < 1e-4; LSE — |err| <= 1e-3 (float32 accumulation of exact
bf16/fp16 products; the reading the pages leave open for the LSE).
"""
from __future__ import annotations

import numpy as np
import torch

from mla_paged_decode_02_gb300 import api, synth
from mla_paged_decode_02_gb300.workload import DeviceWorkload, bits_to_torch_bf16, torch_bf16_to_bits  # noqa: F401
from oracle import mla_oracle as O

BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
FP8_REL_L2 = 1e-2
FP8_COS_DIFF = 1e-4
LSE_ABS = 1e-3


GpuCase = DeviceWorkload


def oracle_decode(case: synth.DecodeCase, cache_np: np.ndarray, rows=None):
    return O.mla_decode(case.q_bits, cache_np, case.block_table, case.seq_lens, case.page_size,
                        case.softmax_scale, case.kv_dtype, case.kv_scale, case.causal, rows=rows)


def compare(case, out_gpu: torch.Tensor, lse_gpu: torch.Tensor, out_ref: np.ndarray,
            lse_ref: np.ndarray, rows=None):
    """Assert the decode contract on all rows (rows=None) or on the sampled (b, i, h)."""
    og = out_gpu.float().cpu().numpy().astype(np.float64)
    lg = lse_gpu.cpu().numpy().astype(np.float64)
    if rows is not None:
        idx = tuple(np.array(rows).T)
        og, lg, out_ref, lse_ref = og[idx], lg[idx], out_ref[idx], lse_ref[idx]
    assert np.isfinite(og).all(), "non-finite output"
    assert np.isfinite(lg).all(), "non-finite lse"
    err = og - out_ref
    rel_l2 = float(np.linalg.norm(err) / max(np.linalg.norm(out_ref), 1e-30))
    max_abs = float(np.abs(err).max())
    lse_err = float(np.abs(lg - lse_ref).max())
    stats = dict(rel_l2=rel_l2, max_abs=max_abs, lse_err=lse_err,
                 cos_diff=O.cos_diff(og, out_ref))
    if case.kv_dtype == synth.KV_BF16:
        assert max_abs <= BF16_MAX_ABS, stats
        assert rel_l2 <= BF16_REL_L2, stats
    else:
        assert rel_l2 <= FP8_REL_L2, stats
        assert stats["cos_diff"] < FP8_COS_DIFF, stats
    assert lse_err <= LSE_ABS, stats
    return stats
