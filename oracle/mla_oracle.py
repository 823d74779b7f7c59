"""Float64 reference for paged MLA decode — oracle, test infrastructure only.

What is computed, and where the pages fix it
--------------------------------------------
"[WIP][Attention] FlashAttn MLA" (opening post) computes the decode step of MLA as
"decode MQA": after weight absorption every query head attends over one shared
key/value head. The kernel-test log quoted in "[Attention] Blackwell FP8 MLA support
with CUTLASS_MLA backend" (comment by elvischenv) fixes the shapes:
``h_q`` query heads, ``h_kv = 1``, ``d = 576`` for scores and ``dv = 512`` for the
output, ``s_q`` new query tokens, ``causal = True``, a paged cache (block size 64 in
that test id) and an FP8 E4M3 variant. "[NVIDIA] Add Cutlass MLA backend" (review
thread) adds the page table and the page size (``block_size``).

Per batch ``b``, new-token row ``i`` and head ``h``::

    K_b[j, :]   = dequant(cache[block_table[b, j // P], j % P, 0:576])   j < L_b
    V_b[j, :]   = K_b[j, 0:512]
    s_j         = softmax_scale * <q[b, i, h, :], K_b[j, :]>             j < n_i
    out[b,i,h]  = sum_j softmax(s)_j * V_b[j]
    lse[b,i,h]  = log(sum_j exp(s_j))                                   (natural log)

with ``n_i = L_b - s_q + 1 + i`` when causal (the ``s_q`` new tokens are the last
``s_q`` positions of the sequence; row ``i`` sees itself and everything before it)
and ``n_i = L_b`` otherwise. The pages leave four points open; this file takes the
plainest reading of each: the 576 values of a row are the 512 latent values followed
by the 64 rope values (for q and for the cache alike); the LSE is a natural log; the
causal mask is aligned bottom-right as above; and the FP8 cache has one per-tensor
scale, ``dequant(byte) = e4m3(byte) * kv_scale``.

Representation: bf16 tensors are carried as their uint16 bit patterns (numpy has no
bf16 type); the FP8 cache as uint8 E4M3 bytes. All arithmetic below is float64; the
two matmuls are numpy library calls. Nothing here is blocked, fused or reordered.
"""
from __future__ import annotations

import numpy as np

from . import fp8_e4m3

D_QK = 576          # 512 latent + 64 rope
D_V = 512
KV_BF16 = 0
KV_FP8_E4M3 = 1


# --------------------------------------------------------------------------- values
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 (exact: bf16 is the top half of float32)."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def dequant_rows(rows: np.ndarray, kv_dtype: int, kv_scale: float) -> np.ndarray:
    """Cache rows -> float64. bf16: the value itself. FP8: ``e4m3(byte) * kv_scale``."""
    if kv_dtype == KV_BF16:
        return bf16_bits_to_f64(rows)
    if kv_dtype == KV_FP8_E4M3:
        return fp8_e4m3.decode(rows) * np.float64(np.float32(kv_scale))
    raise ValueError(f"unknown kv_dtype {kv_dtype}")


# --------------------------------------------------------------------- cache write
def cache_write(kv_cache: np.ndarray, latent_bits: np.ndarray, rope_bits: np.ndarray,
                slot_mapping: np.ndarray, page_size: int, kv_dtype: int,
                kv_scale: float | None = None) -> np.ndarray:
    """Return a copy of ``kv_cache`` with token ``t`` written at slot ``slot_mapping[t]``.

    The row is ``concat(latent[t], rope[t])`` (576 values). Slot ``s`` is page
    ``s // page_size``, offset ``s % page_size``; a negative slot is a padding token
    and is skipped. bf16 cache: the bits are copied. FP8 cache ("[Attention]
    Blackwell FP8 MLA support with CUTLASS_MLA backend", Purpose): each value is
    quantised as ``e4m3_rne_satfinite(float32(x) / float32(kv_scale))``, the
    division being IEEE float32 (correctly rounded), as numpy computes it.
    """
    out = np.array(kv_cache, copy=True)
    slot_mapping = np.asarray(slot_mapping, dtype=np.int64)
    keep = slot_mapping >= 0
    page = slot_mapping[keep] // page_size
    off = slot_mapping[keep] % page_size
    rows = np.concatenate([latent_bits[keep], rope_bits[keep]], axis=1)   # [n, 576]
    if kv_dtype == KV_BF16:
        out[page, off, :] = rows
    else:
        x = bf16_bits_to_f32(rows)
        quot = (x / np.float32(kv_scale)).astype(np.float32)   # float32 / float32
        out[page, off, :] = fp8_e4m3.encode_rne_satfinite(quot)
    return out


# -------------------------------------------------------------------------- gather
def gather_sequence(kv_cache: np.ndarray, block_table_row: np.ndarray, seq_len: int,
                    page_size: int, kv_dtype: int, kv_scale: float | None) -> np.ndarray:
    """Walk one block-table row page by page and return K_b [seq_len, 576] float64.

    Logical page ``p`` of the sequence lives in physical page ``block_table_row[p]``;
    only ``ceil(seq_len / page_size)`` entries are read and, of the last page, only
    the ``seq_len - p * page_size`` filled rows.
    """
    pieces = []
    n_pages = -(-seq_len // page_size)
    for p in range(n_pages):
        phys = int(block_table_row[p])
        rows = min(page_size, seq_len - p * page_size)
        pieces.append(dequant_rows(kv_cache[phys, :rows, :], kv_dtype, kv_scale))
    if not pieces:
        return np.zeros((0, D_QK), dtype=np.float64)
    return np.concatenate(pieces, axis=0)


def visible_keys(seq_len: int, s_q: int, i: int, causal: bool) -> int:
    """Number of keys new-token row ``i`` attends to (bottom-right causal alignment)."""
    return seq_len - s_q + 1 + i if causal else seq_len


# -------------------------------------------------------------------------- decode
def attend(q_rows: np.ndarray, K: np.ndarray, softmax_scale: float):
    """Exact softmax attention of float64 query rows [n, 576] over K [T, 576].

    Returns (out [n, 512], lse [n], weights [n, T]). V is K[:, :512].
    """
    s = (q_rows @ K.T) * softmax_scale
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)
    w = e / l[:, None]
    out = w @ K[:, :D_V]
    lse = m + np.log(l)
    return out, lse, w


def mla_decode(q_bits: np.ndarray, kv_cache: np.ndarray, block_table: np.ndarray,
               seq_lens: np.ndarray, page_size: int, softmax_scale: float,
               kv_dtype: int = KV_BF16, kv_scale: float | None = None,
               causal: bool = True, rows=None):
    """Absorbed-MQA paged decode, float64.

    q_bits [B, s_q, H, 576] (bf16 bits); kv_cache [Np, P, 576] (bf16 bits or E4M3
    bytes); block_table [B, MB] int; seq_lens [B] int (each >= s_q).

    Returns ``out`` [B, s_q, H, 512] and ``lse`` [B, s_q, H] (natural log), float64.
    With ``rows`` (an iterable of (b, i, h)) only those rows are computed and the
    rest of ``out``/``lse`` stays NaN: the full-size tests sample rows this way.
    """
    B, s_q, H, d = q_bits.shape
    assert d == D_QK
    out = np.full((B, s_q, H, D_V), np.nan)
    lse = np.full((B, s_q, H), np.nan)
    want = None
    if rows is not None:
        want = {}
        for (b, i, h) in rows:
            want.setdefault(int(b), []).append((int(i), int(h)))
    for b in range(B):
        if want is not None and b not in want:
            continue
        L = int(seq_lens[b])
        K = gather_sequence(kv_cache, block_table[b], L, page_size, kv_dtype, kv_scale)
        qb = bf16_bits_to_f64(q_bits[b])
        pairs = want[b] if want is not None else [(i, h) for i in range(s_q) for h in range(H)]
        for i in sorted({i for i, _ in pairs}):
            hs = [h for (ii, h) in pairs if ii == i]
            n_i = visible_keys(L, s_q, i, causal)
            o, ls, _ = attend(qb[i, hs, :], K[:n_i], softmax_scale)
            out[b, i, hs, :] = o
            lse[b, i, hs] = ls
    return out, lse


# ------------------------------------------------------------------ split / combine
def attend_range(q_rows: np.ndarray, K: np.ndarray, t0: int, t1: int, softmax_scale: float):
    """Attention restricted to keys [t0, t1): the partial (out_s, lse_s) of one split.

    An empty range yields out_s = 0 and lse_s = -inf (it carries no weight).
    """
    if t1 <= t0:
        return np.zeros((q_rows.shape[0], D_V)), np.full(q_rows.shape[0], -np.inf)
    o, l, _ = attend(q_rows, K[t0:t1], softmax_scale)
    return o, l


def lse_combine(outs, lses):
    """Merge per-split normalised outputs by their log-sum-exps.

    ``lse = log(sum_s exp(lse_s))`` and ``out = sum_s exp(lse_s - lse) * out_s``:
    the exact identity that lets a sequence be cut into key ranges (split-KV /
    flash-decoding) and reassembled.
    """
    lses = np.stack([np.asarray(x, dtype=np.float64) for x in lses])   # [S, n]
    outs = np.stack([np.asarray(x, dtype=np.float64) for x in outs])   # [S, n, 512]
    m = lses.max(axis=0)
    w = np.exp(lses - m[None, :])
    tot = w.sum(axis=0)
    lse = m + np.log(tot)
    out = (w[:, :, None] * outs).sum(axis=0) / tot[:, None]
    return out, lse


# ------------------------------------------------------------------------- metric
def cos_diff(x: np.ndarray, y: np.ndarray) -> float:
    """The FP8 kernel test's closeness metric ("[Attention] Blackwell FP8 MLA support
    with CUTLASS_MLA backend", kernel-test log in the comment by elvischenv):
    one minus twice the inner product over the larger of the summed squares and 1e-12.
    0 for identical tensors, 1 for orthogonal ones or when one of them is zero.
    """
    x = np.asarray(x, dtype=np.float64).ravel()
    y = np.asarray(y, dtype=np.float64).ravel()
    return 1.0 - 2.0 * float((x * y).sum()) / max(float((x * x + y * y).sum()), 1e-12)


def flops(seq_lens, s_q: int, num_heads: int, causal: bool = True) -> float:
    """Algorithmic flops: 2 * (576 + 512) per (row, head, visible key)."""
    tot = 0
    for L in seq_lens:
        for i in range(s_q):
            tot += visible_keys(int(L), s_q, i, causal)
    return 2.0 * (D_QK + D_V) * num_heads * tot


def scale_f32(x) -> float:
    """Round a Python float to float32 (the precision the scales travel in)."""
    return float(np.float32(x))
