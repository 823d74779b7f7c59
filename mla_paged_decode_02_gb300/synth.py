"""Seeded synthetic inputs for paged MLA decode.

This module only draws random numbers and lays out page tables; it holds none of the
attention or quantisation arithmetic, so both the CUDA path and the float64 oracle can
take their inputs from it. Every tensor is a numpy array: bf16 values are carried as
uint16 bit patterns (rounded to nearest-even from float32 draws), integers as int32 /
int64.

Workloads follow the shapes the pages discuss for MLA decode: DeepSeek-V2-Lite style
16 query heads (the kernel test in "[Attention] Blackwell FP8 MLA support with
CUTLASS_MLA backend": b=128, mean_sk=4096, h_q=16, block size 64) and DeepSeek-V3
style 128 heads with page size 128 ("[NVIDIA] Add Cutlass MLA backend": --block-size
128, --max-num-seqs 512), plus a tiny case and a long-context split stress case.

Recipe (fixed so that every run sees the same data):

* ``rng = numpy.random.default_rng(1000 + config_id)`` (or an explicit seed);
* seq_lens drawn first (``rng.integers(lo, hi, endpoint=True)``) unless fixed;
* pages per sequence ``ceil(L_b / P)``; pool ``Np = ceil(1.10 * sum)`` (config 1: the
  exact sum); ``perm = rng.permutation(Np)`` handed out to the sequences in order;
  block-table entries past a sequence's last page point at a spare (never written,
  NaN-poisoned) pool page when one exists, else at the sequence's own first page;
* q, then latent, then rope ~ N(0, 1) drawn as float32 and rounded to bf16;
* the cache starts filled with a NaN pattern (bf16 0x7FC0, E4M3 0x7F) and every
  token is written once through the cache write, token ``j`` of sequence ``b`` at
  slot ``block_table[b, j // P] * P + j % P``;
* FP8: ``kv_scale = float32(max |latent, rope|) / float32(448)``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

D_LATENT = 512
D_ROPE = 64
D_QK = D_LATENT + D_ROPE
D_V = D_LATENT
KV_BF16 = 0
KV_FP8_E4M3 = 1
BF16_NAN_BITS = 0x7FC0
FP8_NAN_BYTE = 0x7F
SOFTMAX_SCALE = float(np.float32(1.0 / math.sqrt(192.0)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) float32 draws rounded to bf16, generated in chunks to bound memory."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


@dataclass
class DecodeCase:
    """One decode workload: everything both the kernels and the oracle consume."""
    name: str
    B: int
    s_q: int
    H: int
    page_size: int
    kv_dtype: int
    causal: bool
    softmax_scale: float
    seq_lens: np.ndarray            # [B] int32
    block_table: np.ndarray         # [B, MB] int32
    num_pages: int
    q_bits: np.ndarray              # [B, s_q, H, 576] uint16 (bf16)
    latent_bits: np.ndarray         # [N, 512] uint16
    rope_bits: np.ndarray           # [N, 64] uint16
    slot_mapping: np.ndarray        # [N] int64
    kv_scale: float | None = None   # float32 value; FP8 only
    meta: dict = field(default_factory=dict)

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max())

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    def empty_cache(self) -> np.ndarray:
        """The pool before any write: every value the NaN pattern."""
        if self.kv_dtype == KV_BF16:
            return np.full((self.num_pages, self.page_size, D_QK), BF16_NAN_BITS, dtype=np.uint16)
        return np.full((self.num_pages, self.page_size, D_QK), FP8_NAN_BYTE, dtype=np.uint8)

    def token_index(self, b: int, j: int) -> int:
        """Row of latent/rope holding token j of sequence b (tokens are batch-major)."""
        return int(self.meta["tok_base"][b]) + j

    def step_tokens(self) -> np.ndarray:
        """Indices (into latent/rope/slot_mapping) of each sequence's last s_q tokens:
        the tokens one decode step appends to the cache."""
        idx = [self.token_index(b, int(self.seq_lens[b]) - self.s_q + i)
               for b in range(self.B) for i in range(self.s_q)]
        return np.asarray(idx, dtype=np.int64)


def make_case(B: int, s_q: int, H: int, page_size: int, seq_lens, kv_dtype: int = KV_BF16,
              seed: int = 0, causal: bool = True, pool_slack: float = 0.10,
              exact_pool: bool = False, softmax_scale: float = SOFTMAX_SCALE,
              name: str = "custom") -> DecodeCase:
    """Build a case. ``seq_lens`` is a list, or a ``(lo, hi)`` tuple drawn uniformly."""
    rng = np.random.default_rng(seed)
    if isinstance(seq_lens, tuple):
        lo, hi = seq_lens
        seq_lens = rng.integers(lo, hi, size=B, endpoint=True)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    assert seq_lens.shape == (B,) and int(seq_lens.min()) >= s_q
    pages = [-(-int(L) // page_size) for L in seq_lens]
    need = sum(pages)
    num_pages = need if exact_pool else int(math.ceil((1.0 + pool_slack) * need))
    perm = rng.permutation(num_pages).astype(np.int32)
    mb = max(pages)
    spare = int(perm[need]) if num_pages > need else None
    block_table = np.empty((B, mb), dtype=np.int32)
    off = 0
    for b, n in enumerate(pages):
        block_table[b, :n] = perm[off:off + n]
        block_table[b, n:] = spare if spare is not None else perm[off]
        off += n
    q_bits = normal_bf16(rng, (B, s_q, H, D_QK))
    n_tok = int(seq_lens.sum())
    latent = normal_bf16(rng, (n_tok, D_LATENT))
    rope = normal_bf16(rng, (n_tok, D_ROPE))
    tok_base = np.zeros(B, dtype=np.int64)
    tok_base[1:] = np.cumsum(seq_lens.astype(np.int64))[:-1]
    slots = np.empty(n_tok, dtype=np.int64)
    for b in range(B):
        L = int(seq_lens[b])
        j = np.arange(L, dtype=np.int64)
        slots[tok_base[b]:tok_base[b] + L] = block_table[b, j // page_size].astype(np.int64) * page_size + j % page_size
    kv_scale = None
    if kv_dtype == KV_FP8_E4M3:
        amax = max(np.abs(_bits_to_f32(latent)).max(initial=0.0),
                   np.abs(_bits_to_f32(rope)).max(initial=0.0))
        kv_scale = float(np.float32(amax) / np.float32(448.0))
    return DecodeCase(name=name, B=B, s_q=s_q, H=H, page_size=page_size, kv_dtype=kv_dtype,
                      causal=causal, softmax_scale=softmax_scale, seq_lens=seq_lens,
                      block_table=block_table, num_pages=num_pages, q_bits=q_bits,
                      latent_bits=latent, rope_bits=rope, slot_mapping=slots,
                      kv_scale=kv_scale, meta={"tok_base": tok_base, "seed": seed})


def _bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


#: The five workloads: name -> (builder kwargs). ``kv`` and ``s_q`` may be overridden.
CONFIGS = {
    1: dict(name="tiny_b2_h16_p64", B=2, s_q=1, H=16, page_size=64, seq_lens=[100, 257],
            exact_pool=True, kv_dtype=KV_BF16),
    2: dict(name="ragged_b128_h16_p64", B=128, s_q=1, H=16, page_size=64, seq_lens=(2048, 6144),
            kv_dtype=KV_BF16),
    3: dict(name="ragged_b128_h16_p64_fp8", B=128, s_q=1, H=16, page_size=64,
            seq_lens=(2048, 6144), kv_dtype=KV_FP8_E4M3),
    4: dict(name="v3_b512_h128_p128", B=512, s_q=1, H=128, page_size=128, seq_lens=(1000, 2000),
            kv_dtype=KV_BF16),
    5: dict(name="long_b4_h128_p64_fp8", B=4, s_q=1, H=128, page_size=64,
            seq_lens=[32768, 65537, 100000, 131072], kv_dtype=KV_FP8_E4M3),
}
#: config 3 is config 2 with an FP8 cache: same seed, same draws.
SEED_OF = {1: 1001, 2: 1002, 3: 1002, 4: 1004, 5: 1005}


def config_name(config_id: int, kv_dtype: int | None = None, s_q: int | None = None) -> str:
    """Name of a workload (no data is drawn)."""
    kw = CONFIGS[config_id]
    kv = kw["kv_dtype"] if kv_dtype is None else kv_dtype
    sq = kw["s_q"] if s_q is None else s_q
    name = kw["name"]
    if kv == KV_FP8_E4M3 and not name.endswith("fp8"):
        name += "_fp8"
    if sq != 1:
        name += f"_sq{sq}"
    return name


def make_config(config_id: int, kv_dtype: int | None = None, s_q: int | None = None) -> DecodeCase:
    kw = dict(CONFIGS[config_id])
    if kv_dtype is not None:
        kw["kv_dtype"] = kv_dtype
    if s_q is not None:
        kw["s_q"] = s_q
    kw.pop("name")
    return make_case(seed=SEED_OF[config_id], name=config_name(config_id, kv_dtype, s_q), **kw)
