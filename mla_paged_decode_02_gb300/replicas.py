"""Data-parallel replicas: each GPU decodes its own sequences over its own paged cache.

"[NVIDIA] Add Cutlass MLA backend" serves DeepSeek-V3 with data parallelism (its benchmark
runs DP+EP on 8 GPUs): attention needs no exchange between GPUs, because every sequence's
keys and values live on the GPU that decodes it. This module is the host side of that:

* ``assign`` balances whole sequences over ranks by their lengths (longest first, each to
  the rank with the fewest tokens so far), so the ranks' decode work (linear in the tokens)
  is even;
* ``shard`` gives each rank a page pool of its own (the pages its sequences need plus
  slack), a block table into that pool and the slot of every token it holds;
* ``Replica`` builds a rank's device-side cache from the tokens of its sequences through
  ``mla_cache_write`` and runs ``mla_decode`` on them.

Nothing here communicates: a rank only reads the batch description and its own data. The
outputs of a rank are its sequences' rows, in the order of ``Shard.seq_idx``.
"""
from __future__ import annotations

import heapq
import math
from dataclasses import dataclass

import numpy as np


def assign(seq_lens, world: int) -> list[np.ndarray]:
    """Per rank, the sorted global indices of the sequences it decodes. Longest-first
    greedy: every rank's token count is within one sequence length of the mean."""
    lens = np.asarray(seq_lens, dtype=np.int64)
    if world < 1:
        raise ValueError("world must be at least 1")
    heap = [(0, r) for r in range(world)]
    parts = [[] for _ in range(world)]
    for b in np.argsort(-lens, kind="stable"):
        load, r = heapq.heappop(heap)
        parts[r].append(int(b))
        heapq.heappush(heap, (load + int(lens[b]), r))
    return [np.array(sorted(p), dtype=np.int64) for p in parts]


@dataclass
class Shard:
    """One rank's part of a batch."""
    rank: int
    seq_idx: np.ndarray       # global indices of the rank's sequences (ascending)
    seq_lens: np.ndarray      # [b] int32
    block_table: np.ndarray   # [b, MB] int32 physical pages of the rank's own pool
    num_pages: int
    page_size: int

    def slots(self, b: int) -> np.ndarray:
        """Cache slot of every token of local sequence b (token j -> page j // P, row j % P)."""
        j = np.arange(int(self.seq_lens[b]), dtype=np.int64)
        return self.block_table[b, j // self.page_size].astype(np.int64) * self.page_size + j % self.page_size


def shard(seq_lens, page_size: int, world: int, rank: int, pool_slack: float = 0.10, seed: int = 0) -> Shard:
    """Rank `rank`'s sequences, page pool and block table. The pool holds the pages the
    sequences need plus `pool_slack`, handed out in a seeded random order (so neighbouring
    sequences do not sit in neighbouring pages); table entries past a sequence's last page
    point at its first page (never read)."""
    idx = assign(seq_lens, world)[rank]
    lens = np.asarray(seq_lens, dtype=np.int32)[idx]
    pages = [-(-int(L) // page_size) for L in lens]
    need = sum(pages)
    num_pages = max(1, int(math.ceil((1.0 + pool_slack) * need)))
    perm = np.random.default_rng(seed + 104729 * rank).permutation(num_pages).astype(np.int32)
    mb = max(pages) if pages else 1
    table = np.zeros((len(idx), mb), dtype=np.int32)
    off = 0
    for b, n in enumerate(pages):
        table[b, :n] = perm[off:off + n]
        table[b, n:] = perm[off] if n else 0
        off += n
    return Shard(rank=rank, seq_idx=idx, seq_lens=lens, block_table=table, num_pages=num_pages,
                 page_size=page_size)


def local_token_rows(shard_: Shard, tok_base: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Rows of the global token arrays (latent, rope: tokens laid out sequence after
    sequence, sequence b starting at tok_base[b]) that the rank holds, and their slots in
    the rank's pool."""
    rows, slots = [], []
    for b, g in enumerate(shard_.seq_idx):
        n = int(shard_.seq_lens[b])
        rows.append(int(tok_base[g]) + np.arange(n, dtype=np.int64))
        slots.append(shard_.slots(b))
    if not rows:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    return np.concatenate(rows), np.concatenate(slots)


class Replica:
    """A rank's decode: its own cache, block table and sequences on its own GPU."""

    def __init__(self, shard_: Shard, latent_bits: np.ndarray, rope_bits: np.ndarray, tok_base: np.ndarray,
                 kv_dtype: int, kv_scale: float | None, device):
        import torch

        from . import api
        from .workload import bits_to_torch_bf16
        self.shard = shard_
        self.device = device
        rows, slots = local_token_rows(shard_, tok_base)
        P = shard_.page_size
        if kv_dtype == api.KV_BF16:
            self.cache = torch.full((shard_.num_pages, P, 576), 0x7FC0, dtype=torch.int16,
                                    device=device).view(torch.bfloat16)
            self.kv_scale = None
        else:
            self.cache = torch.full((shard_.num_pages, P, 576), 0x7F, dtype=torch.uint8, device=device)
            self.kv_scale = torch.tensor([kv_scale], dtype=torch.float32, device=device)
        if len(rows):
            api.cache_write(bits_to_torch_bf16(latent_bits[rows], device), bits_to_torch_bf16(rope_bits[rows], device),
                            torch.from_numpy(slots).to(device), self.cache, self.kv_scale)
        self.block_table = torch.from_numpy(shard_.block_table).to(device)
        self.seq_lens = torch.from_numpy(shard_.seq_lens).to(device)

    def decode(self, q_bits_global: np.ndarray, softmax_scale: float, causal: bool = True):
        """Decode the rank's sequences (q rows taken from the global [B, s_q, H, 576] array).
        Returns (out, lse) for the rank's sequences, in the order of shard.seq_idx."""
        from . import api
        from .workload import bits_to_torch_bf16
        q = bits_to_torch_bf16(np.ascontiguousarray(q_bits_global[self.shard.seq_idx]), self.device)
        return api.decode(q, self.cache, self.block_table, self.seq_lens, softmax_scale, self.kv_scale,
                          max_seq_len=int(self.shard.seq_lens.max()), causal=causal)
