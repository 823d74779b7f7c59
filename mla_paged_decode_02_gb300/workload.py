"""Upload a synthetic workload to the GPU and build its paged cache through the library.

Used by the benchmark and the tests; holds no attention arithmetic (the cache is written
by ``mla_cache_write`` through the C ABI).
"""
from __future__ import annotations

import numpy as np
import torch

from . import api, synth


def bits_to_torch_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def torch_bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


class DeviceWorkload:
    """Device-side tensors of a synth.DecodeCase, with the cache written by mla_cache_write."""

    def __init__(self, case: synth.DecodeCase, device="cuda", build_cache=True):
        self.case = case
        self.device = device
        self.q = bits_to_torch_bf16(case.q_bits, device)
        self.block_table = torch.from_numpy(case.block_table).to(device)
        self.seq_lens = torch.from_numpy(case.seq_lens).to(device)
        self.kv_scale = (torch.tensor([case.kv_scale], dtype=torch.float32, device=device)
                         if case.kv_dtype == synth.KV_FP8_E4M3 else None)
        self.params = api.make_params(case.B, case.s_q, case.H, case.page_size, case.num_pages,
                                      case.max_blocks, case.max_seq_len, case.kv_dtype, case.causal)
        self.workspace = api.alloc_workspace(self.params, device)
        self.cache = None
        if build_cache:
            self.write_cache()

    def empty_cache(self) -> torch.Tensor:
        c = self.case
        if c.kv_dtype == synth.KV_BF16:
            return torch.full((c.num_pages, c.page_size, 576), synth.BF16_NAN_BITS, dtype=torch.int16,
                              device=self.device).view(torch.bfloat16)
        return torch.full((c.num_pages, c.page_size, 576), synth.FP8_NAN_BYTE, dtype=torch.uint8,
                          device=self.device)

    def write_cache(self, chunk_tokens: int = 1 << 20):
        c = self.case
        self.cache = self.empty_cache()
        err = torch.zeros(1, dtype=torch.int32, device=self.device)
        for s in range(0, c.num_tokens, chunk_tokens):
            e = min(c.num_tokens, s + chunk_tokens)
            lat = bits_to_torch_bf16(c.latent_bits[s:e], self.device)
            rope = bits_to_torch_bf16(c.rope_bits[s:e], self.device)
            slots = torch.from_numpy(c.slot_mapping[s:e]).to(self.device)
            api.cache_write(lat, rope, slots, self.cache, self.kv_scale, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0

    def cache_numpy(self) -> np.ndarray:
        if self.case.kv_dtype == synth.KV_BF16:
            return self.cache.cpu().view(torch.int16).numpy().view(np.uint16)
        return self.cache.cpu().numpy()

    def decode(self, out=None, lse=None):
        c = self.case
        return api.decode(self.q, self.cache, self.block_table, self.seq_lens, c.softmax_scale,
                          self.kv_scale, max_seq_len=c.max_seq_len, causal=c.causal, out=out,
                          lse=lse, workspace=self.workspace)
