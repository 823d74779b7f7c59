"""ctypes binding of ``libmla.so`` (declared in ``include/mla.h``) over torch tensors.

Argument marshalling only: every step of the decode runs in the library's kernels.
torch supplies device memory and the current CUDA stream. The library is loaded on
first use; if it is missing this raises — there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

KV_BF16 = 0
KV_FP8_E4M3 = 1
D_QK = 576
D_V = 512

MLA_OK = 0
STATUS = {0: "MLA_OK", -1: "MLA_ERR_INVALID_ARG", -2: "MLA_ERR_UNSUPPORTED",
          -3: "MLA_ERR_WORKSPACE_TOO_SMALL", -4: "MLA_ERR_CUDA", -5: "MLA_ERR_TIMEOUT",
          -6: "MLA_ERR_DEVICE_INDEX"}
EXPORTS = ("mla_abi_version", "mla_status_string", "mla_decode_workspace_size", "mla_decode",
           "mla_decode_check", "mla_cache_write", "mla_decode_noalloc", "mla_decode_noalloc_check",
           "mla_profile_begin", "mla_profile_end", "mla_test_set_hooks", "mla_decode_with_cache_write")
NOALLOC_SCRATCH_BYTES = 32 << 20

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla.so")
_lib = None


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_string(status)})")


class DecodeParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("s_q", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("causal", ctypes.c_int32)]


def lib() -> ctypes.CDLL:
    """The loaded library (loads it on first call; raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build(); "
                               "this package has no non-CUDA implementation")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.mla_abi_version.restype = i32
        L.mla_status_string.restype = ctypes.c_char_p
        L.mla_status_string.argtypes = [i32]
        L.mla_decode_workspace_size.restype = sz
        L.mla_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeParams), i32]
        L.mla_decode.restype = i32
        L.mla_decode.argtypes = [ctypes.POINTER(DecodeParams), vp, vp, vp, vp, ctypes.c_float, vp,
                                 vp, vp, vp, sz, vp]
        L.mla_decode_check.restype = i32
        L.mla_decode_check.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        L.mla_decode_noalloc.restype = i32
        L.mla_decode_noalloc.argtypes = [ctypes.POINTER(DecodeParams), vp, vp, vp, vp, ctypes.c_float,
                                         vp, vp, vp, vp]
        L.mla_decode_noalloc_check.restype = i32
        L.mla_decode_noalloc_check.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        L.mla_cache_write.restype = i32
        L.mla_cache_write.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, vp, vp, vp]
        L.mla_decode_with_cache_write.restype = i32
        L.mla_decode_with_cache_write.argtypes = [ctypes.POINTER(DecodeParams), vp, vp, vp, i32, vp, vp, vp, vp,
                                                  ctypes.c_float, vp, vp, vp, vp, sz, vp]
        L.mla_test_set_hooks.restype = i32
        L.mla_test_set_hooks.argtypes = [ctypes.c_uint64, i32]
        L.mla_profile_begin.restype = i32
        L.mla_profile_begin.argtypes = [i32]
        L.mla_profile_end.restype = i32
        L.mla_profile_end.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i32)]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().mla_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_params(batch, s_q, num_heads, page_size, num_pages, max_blocks_per_seq, max_seq_len,
                kv_dtype, causal=True) -> DecodeParams:
    return DecodeParams(int(batch), int(s_q), int(num_heads), int(page_size), int(num_pages),
                        int(max_blocks_per_seq), int(max_seq_len), int(kv_dtype), int(bool(causal)))


def workspace_size(params: DecodeParams, num_sms: int = 0) -> int:
    n = lib().mla_decode_workspace_size(ctypes.byref(params), int(num_sms))
    if n == 0:
        raise MLAError(-1, "mla_decode_workspace_size")
    return int(n)


def alloc_workspace(params: DecodeParams, device=None) -> torch.Tensor:
    return torch.empty(workspace_size(params), dtype=torch.uint8, device=device or "cuda")


def _kv_dtype_of(kv_cache: torch.Tensor) -> int:
    if kv_cache.dtype == torch.bfloat16:
        return KV_BF16
    if kv_cache.dtype in (torch.uint8, torch.float8_e4m3fn):
        return KV_FP8_E4M3
    raise TypeError(f"kv_cache dtype {kv_cache.dtype}: expected bfloat16, uint8 or float8_e4m3fn")


def _decode_inputs(q, kv_cache, block_table, seq_lens, kv_scale, max_seq_len, causal, out, lse):
    """Check the decode inputs (the library reads them asynchronously, so they are used as
    given: no temporary copies), allocate missing outputs, and build the parameters."""
    B, s_q, H, d = q.shape
    if d != D_QK or q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise ValueError("q must be a contiguous bf16 [B, s_q, H, 576] tensor")
    Np, P, d2 = kv_cache.shape
    if d2 != D_QK or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be a contiguous [Np, P, 576] tensor")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_table and seq_lens must be int32")
    if not block_table.is_contiguous() or not seq_lens.is_contiguous():
        raise ValueError("block_table and seq_lens must be contiguous")
    if block_table.dim() != 2 or block_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("block_table must be [B, MB] and seq_lens [B]")
    kvd = _kv_dtype_of(kv_cache)
    if kvd == KV_FP8_E4M3 and (kv_scale is None or kv_scale.dtype != torch.float32):
        raise ValueError("the FP8 cache needs kv_scale as a float32 device tensor")
    params = make_params(B, s_q, H, P, Np, block_table.shape[1], max_seq_len, kvd, causal)
    if out is None:
        out = torch.empty((B, s_q, H, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, s_q, H), dtype=torch.float32, device=q.device)
    return params, kvd, out, lse


def decode(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
           seq_lens: torch.Tensor, softmax_scale: float, kv_scale: torch.Tensor | None = None,
           *, max_seq_len: int, causal: bool = True, out: torch.Tensor | None = None,
           lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
           stream=None):
    """Paged MLA decode. q [B, s_q, H, 576] bf16; kv_cache [Np, P, 576] (bf16, or uint8 /
    float8_e4m3fn bytes); block_table [B, MB] int32; seq_lens [B] int32; kv_scale a
    1-element float32 device tensor for the FP8 cache. Returns (out, lse)."""
    params, kvd, out, lse = _decode_inputs(q, kv_cache, block_table, seq_lens, kv_scale, max_seq_len,
                                           causal, out, lse)
    if workspace is None:
        workspace = alloc_workspace(params, q.device)
    st = lib().mla_decode(ctypes.byref(params), _ptr(q), _ptr(kv_cache), _ptr(block_table),
                          _ptr(seq_lens), ctypes.c_float(softmax_scale),
                          _ptr(kv_scale) if kvd == KV_FP8_E4M3 else None, _ptr(out), _ptr(lse),
                          _ptr(workspace), workspace.numel(), _stream(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode")
    return out, lse


def decode_with_cache_write(latent: torch.Tensor, rope: torch.Tensor, slot_mapping: torch.Tensor,
                            q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                            seq_lens: torch.Tensor, softmax_scale: float,
                            kv_scale: torch.Tensor | None = None, *, max_seq_len: int,
                            causal: bool = True, out: torch.Tensor | None = None,
                            lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                            stream=None):
    """cache_write() of a step's new tokens followed by decode(), in one launch chain (the
    scheduler kernel writes the new rows). Returns (out, lse)."""
    n = latent.shape[0]
    if latent.shape != (n, 512) or rope.shape != (n, 64) or latent.dtype != torch.bfloat16 \
            or rope.dtype != torch.bfloat16 or not latent.is_contiguous() or not rope.is_contiguous():
        raise ValueError("latent [N,512] and rope [N,64] must be contiguous bf16")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != n or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous int64 [N] tensor")
    params, kvd, out, lse = _decode_inputs(q, kv_cache, block_table, seq_lens, kv_scale, max_seq_len,
                                           causal, out, lse)
    if workspace is None:
        workspace = alloc_workspace(params, q.device)
    st = lib().mla_decode_with_cache_write(ctypes.byref(params), _ptr(latent), _ptr(rope), _ptr(slot_mapping), n,
                                           _ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens),
                                           ctypes.c_float(softmax_scale),
                                           _ptr(kv_scale) if kvd == KV_FP8_E4M3 else None, _ptr(out), _ptr(lse),
                                           _ptr(workspace), workspace.numel(), _stream(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_with_cache_write")
    return out, lse


def decode_noalloc(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                   seq_lens: torch.Tensor, softmax_scale: float, kv_scale: torch.Tensor | None = None,
                   *, max_seq_len: int, causal: bool = True, out: torch.Tensor | None = None,
                   lse: torch.Tensor | None = None, stream=None):
    """decode() without a workspace, for callers that cannot allocate device memory: the
    library's own static scratch array (NOALLOC_SCRATCH_BYTES) is used instead. Calls
    must not overlap on the GPU; pass out and lse to allocate nothing here either."""
    params, kvd, out, lse = _decode_inputs(q, kv_cache, block_table, seq_lens, kv_scale, max_seq_len,
                                           causal, out, lse)
    st = lib().mla_decode_noalloc(ctypes.byref(params), _ptr(q), _ptr(kv_cache), _ptr(block_table),
                                  _ptr(seq_lens), ctypes.c_float(softmax_scale),
                                  _ptr(kv_scale) if kvd == KV_FP8_E4M3 else None, _ptr(out),
                                  _ptr(lse), _stream(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_noalloc")
    return out, lse


def decode_noalloc_check(stream=None):
    """Synchronise and read the device error word of the last decode_noalloc: (status, bits)."""
    bits = ctypes.c_uint32(0)
    st = lib().mla_decode_noalloc_check(_stream(stream), ctypes.byref(bits))
    return int(st), int(bits.value)


def decode_check(workspace: torch.Tensor, stream=None):
    """Synchronise and read the device error word: returns (status, bits)."""
    bits = ctypes.c_uint32(0)
    st = lib().mla_decode_check(_ptr(workspace), _stream(stream), ctypes.byref(bits))
    return int(st), int(bits.value)


def test_set_hooks(wait_limit_ns: int = 0, stall: bool = False) -> None:
    """Tests only: bound of the kernels' pipeline waits (0 = the default 2 s) and the stall
    that makes the first softmax wait run out."""
    st = lib().mla_test_set_hooks(int(wait_limit_ns), int(bool(stall)))
    if st != 0:
        raise MLAError(st, "mla_test_set_hooks")


def profile_begin(max_launches: int) -> None:
    """Time the decode kernel of each of the next `max_launches` decode calls (CUDA events
    around its launch, recorded by the library on the call's stream)."""
    st = lib().mla_profile_begin(int(max_launches))
    if st != 0:
        raise MLAError(st, "mla_profile_begin")


def profile_end():
    """Stop timing; returns (summed decode-kernel milliseconds, number of timed launches)."""
    ms, n = ctypes.c_double(0.0), ctypes.c_int32(0)
    st = lib().mla_profile_end(ctypes.byref(ms), ctypes.byref(n))
    if st != 0:
        raise MLAError(st, "mla_profile_end")
    return float(ms.value), int(n.value)


def cache_write(latent: torch.Tensor, rope: torch.Tensor, slot_mapping: torch.Tensor,
                kv_cache: torch.Tensor, kv_scale: torch.Tensor | None = None,
                device_error: torch.Tensor | None = None, stream=None) -> None:
    """Write token rows concat(latent[t], rope[t]) into the paged cache at slot_mapping[t]."""
    n = latent.shape[0]
    if latent.shape != (n, 512) or rope.shape != (n, 64) or latent.dtype != torch.bfloat16 \
            or rope.dtype != torch.bfloat16 or not latent.is_contiguous() or not rope.is_contiguous():
        raise ValueError("latent [N,512] and rope [N,64] must be contiguous bf16")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != n or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous int64 [N] tensor")
    Np, P, _ = kv_cache.shape
    kvd = _kv_dtype_of(kv_cache)
    st = lib().mla_cache_write(_ptr(latent), _ptr(rope), _ptr(slot_mapping), n,
                               _ptr(kv_cache), Np, P, kvd,
                               _ptr(kv_scale) if kvd == KV_FP8_E4M3 else None,
                               _ptr(device_error), _stream(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_cache_write")
