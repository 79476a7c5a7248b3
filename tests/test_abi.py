"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every function include/ckv.h declares, plan records have the declared
sizes, and argument errors are reported before anything is launched."""
import ctypes
import os
import re

import pytest

from compressed_kv_attention_compressplan_gb300 import build as B
from compressed_kv_attention_compressplan_gb300 import ckv

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ckv.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return ckv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ckv_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_record_sizes_match_header():
    text = open(HEADER).read()
    for struct, size in [("ckv_compress_plan", 16), ("ckv_write_plan", 8), ("ckv_decode_plan", 16),
                         ("ckv_online_unit", 16), ("ckv_decode_order", 8)]:
        body = re.search(r"typedef struct %s \{(.*?)\}" % struct, text, flags=re.S).group(1)
        fields = re.findall(r"(u?int32_t)\s+\w+;", body)
        assert 4 * len(fields) == size, struct
    # the prefill hints: three pointers and two 32-bit words
    body = re.search(r"typedef struct ckv_prefill_hints \{(.*?)\}", text, flags=re.S).group(1)
    assert len(re.findall(r"const int64_t\*\s+\w+;", body)) == 3
    assert len(re.findall(r"uint32_t\s+\w+;", body)) == 2
    assert ctypes.sizeof(ckv.PrefillHints) == 32


def test_capacity_bounds(lib):
    assert ckv.capacity_compress(4, 64, 131072) == 131072 // 4 + 64
    assert ckv.capacity_compress(128, 1024, 100) == 100       # never more than the tokens
    assert ckv.capacity_write(4, 64, 10 ** 6) == 64 * 7
    assert ckv.capacity_write(128, 1024, 5000) == 5000
    assert ckv.capacity_compress(5, 1, 1) == 0
    assert ckv.capacity_write_paged(4, 2, 100, 16) == 2 * 7 + 4 * (100 // 16 + 2)
    assert ckv.capacity_write_paged(128, 1024, 5000, 256) == ckv.capacity_write(128, 1024, 5000)
    assert ckv.capacity_online_units(3, 1000) == 1000 // 128 + 6
    assert ckv.capacity_online_units(100, 40) == 40


def test_argument_errors_are_returned_before_any_launch(lib):
    vp = ctypes.c_void_p
    # bad ratio / head_dim / dtype / layout / pointers: rejected on the host
    assert lib.ckv_plan_decode(3, None, None, 1, None, None, None, None) == -1
    # the boundary-row list must be 8-byte aligned
    assert lib.ckv_plan_decode(128, vp(8), vp(8), 1, vp(16), vp(12), None, None) == -4
    assert lib.ckv_plan_prefill(4, None, None, None, 2000, 0, 0, 0, 0, None, None, vp(16), None, None) == -3
    assert lib.ckv_plan_prefill(4, None, None, None, 1, 0, 0, 0, 0, None, None, vp(16), None, None) == -4
    dec = lib.ckv_compress_decode
    assert dec(4, 100, 1, 0, None, 0, None, None, None, None, None, None, 1, None, None, None) == -2
    assert dec(4, 128, 7, 0, None, 0, None, None, None, None, None, None, 1, None, None, None) == -5
    assert dec(4, 128, 1, 0, vp(8), 8, vp(16), vp(16), vp(16), None, None, None, 1, vp(16), None, None) == -4
    # the boundary-row list and the prefetch hints must be 8-byte aligned
    assert dec(128, 512, 1, 0, vp(16), 8, vp(16), vp(16), vp(16), vp(12), None, None, 1, vp(16), None, None) == -4
    assert dec(128, 512, 1, 0, vp(16), 8, vp(16), vp(16), vp(16), None, vp(20), vp(16), 1, vp(16), None, None) == -4
    pool = lib.ckv_compress_pool_prefill
    assert pool(128, 512, 1, 0, None, 0, None, 10, None, None, None, 1, 9, None, None, None, None) == -5
    # prefetch hints: all three arrays or none, 8-byte aligned (checked before anything is launched)
    H = ckv.PrefillHints
    for h in (H(None, 8, 8, 4, 0), H(8, 8, None, 4, 0), H(8, 12, 8, 4, 0)):
        assert pool(128, 512, 1, 0, vp(16), 128, vp(16), 10, vp(16), vp(16), None, 1, 1, vp(16), ctypes.pointer(h),
                    None, None) == -4
    assert lib.ckv_compress_prefill(4, 512, 1, 0, vp(16), 8, vp(16), 10, vp(16), vp(16), vp(16), None, 1, 1, 1,
                                    vp(16), ctypes.pointer(H(8, 8, 12, 4, 0)), None, None) == -4
    assert lib.ckv_compress_write(4, 2048, 1, None, 0, None, 0, None, None, 1, None, None) == -2
    f = ctypes.c_float
    nrd = lib.ckv_norm_rope_store_decode
    assert nrd(4, 512, 64, 0, None, None, 1, None, f(0.0), None, 16, None, 1, None, 16, None, None) == -3  # eps
    assert nrd(4, 512, 30, 0, None, None, 1, None, f(1e-6), None, 16, None, 1, None, 16, None, None) == -2
    assert nrd(4, 512, 64, 7, None, None, 1, None, f(1e-6), None, 16, None, 1, None, 16, None, None) == -5
    assert nrd(4, 512, 64, 0, None, None, 1, None, f(1e-6), None, 16, None, 1, None, 16, None, None) == -4
    assert nrd(4, 512, 64, 0, None, None, 0, None, f(1e-6), None, 16, None, 1, None, 16, None, None) == 0
    assert lib.ckv_plan_decode_paged(128, None, None, 0, 0, None, 0, 256, 256, None, 1, None, None, None,
                                     None) == -3
    assert lib.ckv_plan_prefill_paged(4, None, None, 8, 1, None, 8, 16, 4, None, None, 1, 4, 4, 4, 0, None, None,
                                      None, None, None) == -3  # a 4-row ring
    assert lib.ckv_compress_online_decode(100, 1, 0, None, 0, None, None, None, 1, None, None, None) == -2
    assert lib.ckv_compress_online_prefill(512, 1, 0, None, 1, None, 8, None, None, None, 4, 9, 0, None, None,
                                           None) == -5
    assert lib.ckv_compress_online_prefill(512, 1, 0, None, 1, None, 8, None, None, None, 4, 0, 0, None, None,
                                           None) == -4
    assert lib.ckv_plan_online_prefill(None, None, None, 2000, 0, 0, 0, 0, None, vp(16), None, None) == -3
    fused = lib.ckv_compress_decode_norm_rope_store
    f32 = ctypes.c_float
    ok = dict(state=vp(16), inp=vp(16), ape=vp(16), pd=vp(16), w=vp(16), fr=vp(16), loc=vp(16), cache=vp(16))

    def call(ratio=4, hd=512, rope=64, in_dt=1, eps=1e-6, cache_dt=1, loc=vp(16), batch=3):
        return fused(ratio, hd, rope, in_dt, ok["state"], 64, ok["inp"], ok["ape"], ok["pd"], None, None, batch,
                     ok["w"], f32(eps), ok["fr"], 16, loc, cache_dt, ok["cache"], 16, None, None)
    assert call(ratio=128) == -1      # the C128 decode has no fused form
    assert call(hd=200) == -2
    assert call(rope=30) == -2
    assert call(in_dt=7) == -5
    assert call(cache_dt=7) == -5
    assert call(eps=0.0) == -3
    assert call(loc=vp(12)) == -4     # out_loc must be 8-byte aligned
    assert call(loc=None) == -4
    assert call(batch=0) == 0         # nothing to do, nothing launched
    assert lib.ckv_error_string(-4) != lib.ckv_error_string(0)


def test_binding_rejects_wrong_per_request_arrays():
    """rid / seq_lens / extend_lens reach the library as raw int64 arrays: the
    binding must refuse other dtypes and arrays of different lengths."""
    import torch

    from compressed_kv_attention_compressplan_gb300 import ckv

    i64 = torch.arange(5, dtype=torch.int64)
    assert ckv._lengths(i64, i64.clone(), None) == 5
    with pytest.raises(ValueError):
        ckv._lengths(i64.to(torch.int32), i64)
    with pytest.raises(ValueError):
        ckv._lengths(i64, torch.arange(4, dtype=torch.int64))
    with pytest.raises(ValueError):
        ckv._lengths(i64.view(5, 1))


def test_wait_limit_setter(lib):
    assert lib.ckv_version() >= 220  # ABI 2.20: fused C4 decode + norm (2.10: prefill hints; 2.00: decode lists)
    default = 2_000_000_000
    prev = ckv.set_wait_limit_ns(0)            # whatever was set, back to the default
    assert ckv.set_wait_limit_ns(1234) == default
    assert ckv.set_wait_limit_ns(5) == 1234
    assert ckv.set_wait_limit_ns(0) == 5       # 0 restores the default ...
    assert ckv.set_wait_limit_ns(0) == default
    # limits beyond 10 s come back clamped: every wait stays bounded
    assert ckv.set_wait_limit_ns(2 ** 64 - 1) == default
    assert ckv.set_wait_limit_ns(20_000_000_000) == 10_000_000_000
    assert ckv.set_wait_limit_ns(prev if prev != default else 0) == 10_000_000_000
    with pytest.raises(ValueError):
        ckv.set_wait_limit_ns(-1)
    ckv.set_wait_limit_ns(0)
