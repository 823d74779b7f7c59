"""Host-only checks of the C ABI: the library loads, exports every declared symbol, and
rejects bad arguments before touching the GPU. Runs without a GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from mla_paged_decode_02_gb300 import api

HEADER = os.path.join(ROOT, "include", "mla.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(api.LIB_PATH):
        pytest.skip("libmla.so not built")
    return api.lib()


def test_header_declares_the_boundary():
    fns = declared_functions()
    assert set(api.EXPORTS) == set(fns), fns


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.mla_abi_version() == 1


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert api.status_string(code) != "unknown status"
    assert api.status_string(7) == "unknown status"


def test_workspace_size_is_bounded_and_rejects_bad_params(lib):
    p = api.make_params(128, 1, 16, 64, 9000, 100, 6144, api.KV_BF16)
    n = lib.mla_decode_workspace_size(ctypes.byref(p), 148)
    assert 0 < n < 64 << 20
    big = api.make_params(512, 1, 128, 128, 7000, 16, 2000, api.KV_FP8_E4M3)
    assert lib.mla_decode_workspace_size(ctypes.byref(big), 148) < 256 << 20
    for bad in (dict(batch=0), dict(s_q=0), dict(page_size=12), dict(page_size=1), dict(page_size=1032),
                dict(kv_dtype=3), dict(causal=2), dict(max_seq_len=0), dict(num_heads=0)):
        q = api.make_params(2, 1, 16, 64, 10, 5, 300, api.KV_BF16)
        for k, v in bad.items():
            setattr(q, k, v)
        assert lib.mla_decode_workspace_size(ctypes.byref(q), 148) == 0, bad
    # any multiple of 8 up to 1024 rows per page is supported (boxes of gcd(P, 64) rows)
    for P in (8, 16, 24, 48, 1024):
        q = api.make_params(2, 1, 16, P, 10, 5, 300, api.KV_BF16)
        q.max_blocks_per_seq = -(-300 // P)
        assert lib.mla_decode_workspace_size(ctypes.byref(q), 148) > 0, P


def test_decode_rejects_null_and_misaligned_pointers_without_a_gpu(lib):
    p = api.make_params(2, 1, 16, 64, 10, 5, 300, api.KV_BF16)
    vp = ctypes.c_void_p
    good = vp(1 << 20)
    args = [good, good, good, good, ctypes.c_float(0.07), None, good, good, good, 1 << 30, None]
    for i in (0, 1, 2, 3, 6, 7, 8):
        a = list(args)
        a[i] = None
        assert lib.mla_decode(ctypes.byref(p), *a) == -1
    a = list(args)
    a[0] = vp((1 << 20) + 2)          # q not 16-byte aligned
    assert lib.mla_decode(ctypes.byref(p), *a) == -1
    fp8 = api.make_params(2, 1, 16, 64, 10, 5, 300, api.KV_FP8_E4M3)
    assert lib.mla_decode(ctypes.byref(fp8), *args) == -1          # FP8 without kv_scale
    unsup = api.make_params(2, 513, 16, 64, 10, 50, 3000, api.KV_BF16)     # s_q above 512
    assert lib.mla_decode(ctypes.byref(unsup), *args) == -2
    unsup = api.make_params(2, 512, 129, 64, 10, 50, 3000, api.KV_BF16)    # s_q * H above 65536
    assert lib.mla_decode(ctypes.byref(unsup), *args) == -2


def test_test_hooks_reject_a_bad_stall_value(lib):
    assert lib.mla_test_set_hooks(0, 2) == -1
    assert lib.mla_test_set_hooks(0, 0) == 0


def test_profile_window_arguments_without_a_gpu(lib):
    assert lib.mla_profile_begin(0) == -1
    assert lib.mla_profile_begin(4097) == -1
    ms, n = ctypes.c_double(7.0), ctypes.c_int32(7)
    assert lib.mla_profile_end(None, ctypes.byref(n)) == -1
    assert lib.mla_profile_end(ctypes.byref(ms), None) == -1
    assert lib.mla_profile_end(ctypes.byref(ms), ctypes.byref(n)) == 0     # no window open
    assert ms.value == 0.0 and n.value == 0


def test_cache_write_rejects_bad_arguments_without_a_gpu(lib):
    vp = ctypes.c_void_p
    good = vp(1 << 20)
    assert lib.mla_cache_write(good, good, good, 4, good, 10, 64, 1, None, None, None) == -1
    assert lib.mla_cache_write(good, good, good, 4, good, 10, 64, 5, None, None, None) == -1
    assert lib.mla_cache_write(None, good, good, 4, good, 10, 64, 0, None, None, None) == -1
    assert lib.mla_cache_write(None, None, None, 0, None, 10, 64, 0, None, None, None) == 0
