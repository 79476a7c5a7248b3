"""CPU oracle for the compressed-KV compressor -- TEST INFRASTRUCTURE ONLY.

The oracle is a plain single-threaded C program (``ckv_oracle.c``) that states
what the GPU library computes: the plan builders, the state write and the
per-channel softmax pool, with the pool carried in double and rounded once.
Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
and never imports it.

Every function takes and returns numpy arrays.  bf16 tensors travel as their
raw ``uint16`` bit patterns, so both sides see identical bytes.

Sources: SGLang ``c_plan.cuh`` (plan builders), ``c4.cuh`` (C4 write + pool),
``compressor_v2.py`` (C128 write + pool).  Each C function names the passage it
follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32 = 0
BF16 = 1
OUT_TOKEN = 0
OUT_COMPACT = 1

OK = 0
BAD_RATIO = -1
BAD_HEAD_DIM = -2
BAD_BATCH = -3
BAD_DTYPE = -5
BAD_LENGTH = -8
BAD_TOTAL = -9
CAPACITY = -10
BAD_INDEX = -11

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ckv_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libckv_oracle.so")
_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what} returned {code}")
        self.code = code


def _compile(src: str, lib: str) -> str:
    tmp = lib + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-Wall", "-shared", "-fPIC", "-o", tmp,
           src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, -O2, no fp contraction)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    return _compile(_SRC, _LIB)


def source() -> str:
    """The oracle's C source (test-only use: the mutation check patches a copy)."""
    return open(_SRC).read()


def build_variant(text: str, tag: str) -> str:
    """Test-only: compile another C source text (a patched copy of the oracle) to its own library under
    _build/; route calls to it with use_library()."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    src = os.path.join(_LIB_DIR, f"ckv_oracle_{tag}.c")
    with open(src, "w") as f:
        f.write(text)
    return _compile(src, os.path.join(_LIB_DIR, f"libckv_oracle_{tag}.so"))


def use_library(path: str | None):
    """Test-only: route the functions of this module to another build (None = the oracle)."""
    global _lib
    with _lock:
        _lib = None
    if path is not None:
        _load(path)


def _load(path: str | None = None):
    global _lib
    with _lock:
        if _lib is None:
            if path is None:
                path = build()
            lib = ctypes.CDLL(path)
            vp, u32, i32, u64 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int, ctypes.c_uint64
            lib.orc_plan_decode.argtypes = [i32, vp, vp, u32, vp]
            lib.orc_plan_prefill.argtypes = [i32, vp, vp, vp, u32, u32, u32, u32, i32, vp, vp, vp]
            lib.orc_compress_pool_prefill.argtypes = [i32, i32, i32, i32, vp, u64, vp, u32, vp, vp, u32, i32, vp]
            lib.orc_compress_write.argtypes = [i32, i32, i32, vp, u64, vp, u32, vp, u32]
            lib.orc_compress_decode.argtypes = [i32, i32, i32, i32, vp, u64, vp, vp, vp, u32, vp]
            lib.orc_compress_history.argtypes = [i32, i32, i32, i32, vp, u32, vp, vp]
            i64 = ctypes.c_int64
            lib.orc_plan_prefill_paged.argtypes = [i32, vp, vp, i64, u32, vp, u64, i32, i32, vp, vp, u32, u32, u32,
                                                   u32, i32, vp, vp, vp]
            lib.orc_plan_decode_paged.argtypes = [i32, vp, vp, i64, u32, vp, u64, i32, i32, vp, u32, vp]
            lib.orc_norm_rope_store.argtypes = [i32, i32, i32, i32, i32, vp, i32, u64, vp, u32, vp, ctypes.c_float,
                                                vp, u32, vp, u64, i32, vp, u64]
            lib.orc_plan_online_prefill.argtypes = [vp, vp, vp, u32, u32, i64, u32, i32, vp, vp]
            lib.orc_online_prefill.argtypes = [i32, i32, i32, vp, u64, vp, u32, vp, vp, u32, i32, u32, vp]
            lib.orc_plan_online_decode.argtypes = [vp, vp, u32, i64, vp]
            lib.orc_online_decode.argtypes = [i32, i32, i32, vp, u64, vp, vp, vp, u32, vp]
            lib.orc_double_to_bf16.argtypes = [ctypes.c_double]
            lib.orc_double_to_bf16.restype = ctypes.c_uint16
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def window(ratio: int) -> int:
    return 8 if ratio == 4 else ratio


def row_width(ratio: int, hd: int) -> int:
    return 4 * hd if ratio == 4 else 2 * hd


def elem_np(dtype: int):
    return np.uint16 if dtype == BF16 else np.float32


# --------------------------------------------------------------------------- plans
def plan_decode(ratio: int, rid, seq_lens) -> np.ndarray:
    """DecodePlan records as a ``[batch, 16]`` uint8 array."""
    rid, sl = _i64(rid), _i64(seq_lens)
    out = np.zeros((len(rid), 16), dtype=np.uint8)
    rc = _load().orc_plan_decode(ratio, _p(rid), _p(sl), len(rid), _p(out))
    if rc:
        raise OracleError(rc, "plan_decode")
    return out


def plan_prefill(ratio: int, rid, seq_lens, extend_lens, num_q_tokens: int | None = None,
                 cap_c: int | None = None, cap_w: int | None = None, pad_invalid: bool = False,
                 check: bool = True):
    """Returns ``(plan_c [cap_c,16] u8, plan_w [cap_w,8] u8, counts (num_c, num_w), rc)``.

    Without capacities, the arrays are sized to the exact counts."""
    rid, sl, el = _i64(rid), _i64(seq_lens), _i64(extend_lens)
    nq = int(el.sum()) if num_q_tokens is None else int(num_q_tokens)
    lib = _load()
    counts = np.zeros(2, dtype=np.uint32)
    if cap_c is None or cap_w is None:
        # first pass: count only
        dummy_c = np.zeros((1, 16), np.uint8)
        dummy_w = np.zeros((1, 8), np.uint8)
        lib.orc_plan_prefill(ratio, _p(rid), _p(sl), _p(el), len(rid), nq, 0, 0, 0, _p(dummy_c), _p(dummy_w),
                             _p(counts))
        cap_c = int(counts[0]) if cap_c is None else cap_c
        cap_w = int(counts[1]) if cap_w is None else cap_w
    pc = np.zeros((max(cap_c, 1), 16), dtype=np.uint8)
    pw = np.zeros((max(cap_w, 1), 8), dtype=np.uint8)
    rc = lib.orc_plan_prefill(ratio, _p(rid), _p(sl), _p(el), len(rid), nq, cap_c, cap_w, int(pad_invalid),
                              _p(pc), _p(pw), _p(counts))
    if check and rc:
        raise OracleError(rc, "plan_prefill")
    return pc[:cap_c], pw[:cap_w], (int(counts[0]), int(counts[1])), rc


def _maps(req_to_token, full_to_state):
    """The two SWA maps as C arrays (C128 reads neither: None stands for none)."""
    if req_to_token is None:
        return np.zeros((1, 1), np.int32), np.zeros(1, np.int64)
    return np.ascontiguousarray(np.asarray(req_to_token, dtype=np.int32)), _i64(full_to_state)


def plan_prefill_paged(ratio: int, rid, req_to_token, full_to_state, swa_page_size: int, ring_size: int, seq_lens,
                       extend_lens, num_q_tokens: int | None = None, cap_c: int | None = None,
                       cap_w: int | None = None, pad_invalid: bool = False, check: bool = True):
    """SWA-paged prefill plans (see ckv_oracle.c); same return value as plan_prefill."""
    rid, sl, el = _i64(rid), _i64(seq_lens), _i64(extend_lens)
    r2t, f2s = _maps(req_to_token, full_to_state)
    nq = int(el.sum()) if num_q_tokens is None else int(num_q_tokens)
    lib = _load()
    counts = np.zeros(2, dtype=np.uint32)
    args = (ratio, _p(rid), _p(r2t), r2t.shape[1], r2t.shape[0], _p(f2s), f2s.size, swa_page_size, ring_size,
            _p(sl), _p(el), len(rid), nq)
    if cap_c is None or cap_w is None:
        dc, dw = np.zeros((1, 16), np.uint8), np.zeros((1, 8), np.uint8)
        lib.orc_plan_prefill_paged(*args, 0, 0, 0, _p(dc), _p(dw), _p(counts))
        cap_c = int(counts[0]) if cap_c is None else cap_c
        cap_w = int(counts[1]) if cap_w is None else cap_w
    pc = np.zeros((max(cap_c, 1), 16), dtype=np.uint8)
    pw = np.zeros((max(cap_w, 1), 8), dtype=np.uint8)
    rc = lib.orc_plan_prefill_paged(*args, cap_c, cap_w, int(pad_invalid), _p(pc), _p(pw), _p(counts))
    if check and rc:
        raise OracleError(rc, "plan_prefill_paged")
    return pc[:cap_c], pw[:cap_w], (int(counts[0]), int(counts[1])), rc


def plan_decode_paged(ratio: int, rid, req_to_token, full_to_state, swa_page_size: int, ring_size: int,
                      seq_lens) -> np.ndarray:
    rid, sl = _i64(rid), _i64(seq_lens)
    r2t, f2s = _maps(req_to_token, full_to_state)
    out = np.zeros((len(rid), 16), dtype=np.uint8)
    rc = _load().orc_plan_decode_paged(ratio, _p(rid), _p(r2t), r2t.shape[1], r2t.shape[0], _p(f2s), f2s.size,
                                       swa_page_size, ring_size, _p(sl), len(rid), _p(out))
    if rc:
        raise OracleError(rc, "plan_decode_paged")
    return out


def decode_plan_fields(plan_c: np.ndarray) -> dict:
    """Unpacks CompressPlan records into named integer columns."""
    w = plan_c.reshape(-1, 16).view(np.uint32).reshape(-1, 4)
    return {
        "seq_len": w[:, 0].astype(np.int64),
        "ragged_id": (w[:, 1] & 0x00FFFFFF).astype(np.int64),
        "buffer_len": (w[:, 1] >> 24).astype(np.int64),
        "read_page_0": w[:, 2].view(np.int32).astype(np.int64),
        "read_page_1": w[:, 3].view(np.int32).astype(np.int64),
    }


# --------------------------------------------------------------------------- compute
def compress_pool_prefill(ratio, hd, in_dtype, out_dtype, state, inp, ape, plan_c, num_c=None,
                          num_q_tokens=None, out_layout=OUT_TOKEN) -> np.ndarray:
    state = np.ascontiguousarray(state)
    inp = np.ascontiguousarray(inp)
    ape = np.ascontiguousarray(ape)
    plan_c = np.ascontiguousarray(plan_c)
    width = row_width(ratio, hd)
    nq = inp.size // width if num_q_tokens is None else int(num_q_tokens)
    nc = plan_c.shape[0] if num_c is None else int(num_c)
    rows = nq if out_layout == OUT_TOKEN else nc
    out = np.zeros((rows, hd), dtype=elem_np(out_dtype))
    state_rows = state.size // width
    rc = _load().orc_compress_pool_prefill(ratio, hd, in_dtype, out_dtype, _p(state), state_rows, _p(inp), nq,
                                           _p(ape), _p(plan_c), nc, out_layout, _p(out))
    if rc:
        raise OracleError(rc, "compress_pool_prefill")
    return out


def compress_write(ratio, hd, dtype, state: np.ndarray, inp, plan_w, num_w=None) -> None:
    """Writes into ``state`` in place."""
    assert state.flags["C_CONTIGUOUS"]
    inp = np.ascontiguousarray(inp)
    plan_w = np.ascontiguousarray(plan_w)
    width = row_width(ratio, hd)
    nw = plan_w.shape[0] if num_w is None else int(num_w)
    rc = _load().orc_compress_write(ratio, hd, dtype, _p(state), state.size // width, _p(inp),
                                    inp.size // width, _p(plan_w), nw)
    if rc:
        raise OracleError(rc, "compress_write")


def compress_decode(ratio, hd, in_dtype, out_dtype, state: np.ndarray, inp, ape, plan_d) -> np.ndarray:
    """Writes the new rows into ``state`` in place and returns the ``[batch, hd]`` output."""
    assert state.flags["C_CONTIGUOUS"]
    inp = np.ascontiguousarray(inp)
    ape = np.ascontiguousarray(ape)
    plan_d = np.ascontiguousarray(plan_d)
    width = row_width(ratio, hd)
    batch = plan_d.shape[0]
    out = np.zeros((batch, hd), dtype=elem_np(out_dtype))
    rc = _load().orc_compress_decode(ratio, hd, in_dtype, out_dtype, _p(state), state.size // width, _p(inp),
                                     _p(ape), _p(plan_d), batch, _p(out))
    if rc:
        raise OracleError(rc, "compress_decode")
    return out


def compress_history(ratio, hd, in_dtype, out_dtype, tokens, ape) -> np.ndarray:
    """Compressed rows of one whole sequence from its token history, token layout."""
    tokens = np.ascontiguousarray(tokens)
    ape = np.ascontiguousarray(ape)
    T = tokens.size // row_width(ratio, hd)
    out = np.zeros((T, hd), dtype=elem_np(out_dtype))
    rc = _load().orc_compress_history(ratio, hd, in_dtype, out_dtype, _p(tokens), T, _p(ape), _p(out))
    if rc:
        raise OracleError(rc, "compress_history")
    return out


def compress_prefill(ratio, hd, in_dtype, out_dtype, state: np.ndarray, inp, ape, rid, seq_lens, extend_lens,
                     out_layout=OUT_TOKEN):
    """Plan, pool, then write (the order of compressor_v2.py's prefill launcher)."""
    pc, pw, (nc, nw), _ = plan_prefill(ratio, rid, seq_lens, extend_lens)
    out = compress_pool_prefill(ratio, hd, in_dtype, out_dtype, state, inp, ape, pc, nc,
                                num_q_tokens=int(_i64(extend_lens).sum()), out_layout=out_layout)
    compress_write(ratio, hd, in_dtype, state, inp, pw, nw)
    return out, pc, pw


def plan_online_prefill(rid, seq_lens, extend_lens, slot_offset: int = 0, num_q_tokens: int | None = None,
                        cap_u: int | None = None, pad_invalid: bool = False, check: bool = True):
    """Online-state prefill units (16 B records); returns (units, (num_units, num_c), rc)."""
    rid, sl, el = _i64(rid), _i64(seq_lens), _i64(extend_lens)
    nq = int(el.sum()) if num_q_tokens is None else int(num_q_tokens)
    lib = _load()
    counts = np.zeros(2, dtype=np.uint32)
    if cap_u is None:
        lib.orc_plan_online_prefill(_p(rid), _p(sl), _p(el), len(rid), nq, slot_offset, 0, 0,
                                    _p(np.zeros((1, 16), np.uint8)), _p(counts))
        cap_u = int(counts[0])
    units = np.zeros((max(cap_u, 1), 16), dtype=np.uint8)
    rc = lib.orc_plan_online_prefill(_p(rid), _p(sl), _p(el), len(rid), nq, slot_offset, cap_u, int(pad_invalid),
                                     _p(units), _p(counts))
    if check and rc:
        raise OracleError(rc, "plan_online_prefill")
    return units[:cap_u], (int(counts[0]), int(counts[1])), rc


def online_prefill(hd, in_dtype, out_dtype, state: np.ndarray, inp, ape, units, out_layout=OUT_TOKEN,
                   out_rows: int | None = None) -> np.ndarray:
    """Runs the units through the online state (float64 ``[slots, 3 hd]``, updated in place)."""
    assert state.dtype == np.float64 and state.flags["C_CONTIGUOUS"]
    inp, ape, units = np.ascontiguousarray(inp), np.ascontiguousarray(ape), np.ascontiguousarray(units)
    nq = inp.size // (2 * hd)
    rows = nq if out_layout == OUT_TOKEN else int(out_rows)
    out = np.zeros((max(rows, 1), hd), dtype=elem_np(out_dtype))
    rc = _load().orc_online_prefill(hd, in_dtype, out_dtype, _p(state), state.size // (3 * hd), _p(inp), nq, _p(ape),
                                    _p(units), units.shape[0], out_layout, rows, _p(out))
    if rc:
        raise OracleError(rc, "online_prefill")
    return out[:rows]


def plan_online_decode(rid, seq_lens, slot_offset: int = 0) -> np.ndarray:
    rid, sl = _i64(rid), _i64(seq_lens)
    out = np.zeros((len(rid), 16), dtype=np.uint8)
    rc = _load().orc_plan_online_decode(_p(rid), _p(sl), len(rid), slot_offset, _p(out))
    if rc:
        raise OracleError(rc, "plan_online_decode")
    return out


def online_decode(hd, in_dtype, out_dtype, state: np.ndarray, inp, ape, plan_d) -> np.ndarray:
    assert state.dtype == np.float64 and state.flags["C_CONTIGUOUS"]
    inp, ape, plan_d = np.ascontiguousarray(inp), np.ascontiguousarray(ape), np.ascontiguousarray(plan_d)
    batch = plan_d.shape[0]
    out = np.zeros((max(batch, 1), hd), dtype=elem_np(out_dtype))
    rc = _load().orc_online_decode(hd, in_dtype, out_dtype, _p(state), state.size // (3 * hd), _p(inp), _p(ape),
                                   _p(plan_d), batch, _p(out))
    if rc:
        raise OracleError(rc, "online_decode")
    return out[:batch]


def norm_rope_store(ratio: int, mode: int, hd: int, rope_dim: int, in_dtype: int, rows, in_layout: int, plan,
                    weight, eps: float, freqs, out_loc, cache_dtype: int, cache: np.ndarray) -> None:
    """RMSNorm + RoPE + store of compressed rows into ``cache`` (in place); mode 0 prefill (plan = CompressPlan
    records), 1 decode (plan = DecodePlan records).  freqs: fp32 ``[max_pos, rope_dim/2, 2]`` (cos, sin)."""
    assert cache.flags["C_CONTIGUOUS"]
    rows = np.ascontiguousarray(rows)
    plan = np.ascontiguousarray(plan).reshape(-1, 16)
    weight = np.ascontiguousarray(weight, dtype=np.float32)
    freqs = np.ascontiguousarray(freqs, dtype=np.float32)
    out_loc = _i64(out_loc)
    n_rows = rows.size // hd
    rc = _load().orc_norm_rope_store(ratio, mode, hd, rope_dim, in_dtype, _p(rows), in_layout, n_rows, _p(plan),
                                     plan.shape[0], _p(weight), float(eps), _p(freqs), freqs.shape[0], _p(out_loc),
                                     out_loc.size, cache_dtype, _p(cache), cache.size // hd)
    if rc:
        raise OracleError(rc, "norm_rope_store")


def double_to_bf16(x: float) -> int:
    return int(_load().orc_double_to_bf16(float(x)))
