"""Python binding of libckv (the GB300 KV compressor) over its C ABI.

Argument marshalling only: every step runs in the library's CUDA kernels.
Functions take CUDA ``torch.Tensor`` arguments, pass their device pointers and
the current CUDA stream to the C entry point of the same name, and raise
``CkvError`` for a non-zero return code.  There is no CPU path: without the
built library (``build()`` / ``__graft_entry__.build()``) every call raises.

Layouts (see include/ckv.h): kv_score rows are C4 ``[kv-ovl|kv|score-ovl|score]``
(4*hd) or C128 ``[kv|score]`` (2*hd); the state is ``[rows, width]`` in the
input dtype with 8 rows per request (C4) or 128 (C128); plans are uint8
tensors of 16-byte (compress, decode) or 8-byte (write) records.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import build as _build

F32 = 0
BF16 = 1
OUT_TOKEN = 0
OUT_COMPACT = 1

STATUS_BAD_LENGTH = 1
STATUS_BAD_TOTAL = 2
STATUS_CAPACITY = 4
STATUS_BAD_INDEX = 8
STATUS_TIMEOUT = 16

_lock = threading.Lock()
_lib = None


class CkvError(RuntimeError):
    def __init__(self, code: int, func: str, msg: str):
        super().__init__(f"{func}: {msg} (code {code})")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load_library():
    """Loads libckv.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libckv.so is not built ({path}); run "
                               "compressed_kv_attention_compressplan_gb300.build.build() first")
        lib = ctypes.CDLL(path)
        vp, u32, i32, u64 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int, ctypes.c_uint64
        lib.ckv_capacity_compress.argtypes = [i32, u32, u32]
        lib.ckv_capacity_compress.restype = u32
        lib.ckv_capacity_write.argtypes = [i32, u32, u32]
        lib.ckv_capacity_write.restype = u32
        lib.ckv_plan_decode.argtypes = [i32, vp, vp, u32, vp, vp, vp, vp]
        i64 = ctypes.c_int64
        lib.ckv_capacity_write_paged.argtypes = [i32, u32, u32, i32]
        lib.ckv_capacity_write_paged.restype = u32
        lib.ckv_plan_prefill_paged.argtypes = [i32, vp, vp, i64, u32, vp, u64, i32, i32, vp, vp, u32, u32, u32, u32,
                                               i32, vp, vp, vp, vp, vp]
        lib.ckv_plan_decode_paged.argtypes = [i32, vp, vp, i64, u32, vp, u64, i32, i32, vp, u32, vp, vp, vp, vp]
        lib.ckv_plan_prefill.argtypes = [i32, vp, vp, vp, u32, u32, u32, u32, i32, vp, vp, vp, vp, vp]
        lib.ckv_compress_write.argtypes = [i32, i32, i32, vp, u64, vp, u32, vp, vp, u32, vp, vp]
        lib.ckv_compress_pool_prefill.argtypes = [i32, i32, i32, i32, vp, u64, vp, u32, vp, vp, vp, u32, i32, vp,
                                                  ctypes.POINTER(PrefillHints), vp, vp]
        lib.ckv_compress_prefill.argtypes = [i32, i32, i32, i32, vp, u64, vp, u32, vp, vp, vp, vp, u32, u32, i32,
                                             vp, ctypes.POINTER(PrefillHints), vp, vp]
        lib.ckv_compress_decode.argtypes = [i32, i32, i32, i32, vp, u64, vp, vp, vp, vp, vp, vp, u32, vp, vp, vp]
        f32 = ctypes.c_float
        lib.ckv_capacity_online_units.argtypes = [u32, u32]
        lib.ckv_capacity_online_units.restype = u32
        lib.ckv_plan_online_prefill.argtypes = [vp, vp, vp, u32, u32, i64, u32, i32, vp, vp, vp, vp]
        lib.ckv_plan_online_decode.argtypes = [vp, vp, u32, i64, vp, vp, vp]
        lib.ckv_compress_online_prefill.argtypes = [i32, i32, i32, vp, u64, vp, u32, vp, vp, vp, u32, i32, u32, vp,
                                                    vp, vp]
        lib.ckv_compress_online_decode.argtypes = [i32, i32, i32, vp, u64, vp, vp, vp, u32, vp, vp, vp]
        lib.ckv_norm_rope_store_prefill.argtypes = [i32, i32, i32, i32, vp, i32, u64, vp, vp, u32, vp, f32, vp, u32,
                                                    vp, u64, i32, vp, u64, vp, vp]
        lib.ckv_norm_rope_store_decode.argtypes = [i32, i32, i32, i32, vp, vp, u32, vp, f32, vp, u32, vp, i32, vp,
                                                   u64, vp, vp]
        lib.ckv_compress_decode_norm_rope_store.argtypes = [i32, i32, i32, i32, vp, u64, vp, vp, vp, vp, vp, u32, vp,
                                                            f32, vp, u32, vp, i32, vp, u64, vp, vp]
        lib.ckv_error_string.argtypes = [i32]
        lib.ckv_error_string.restype = ctypes.c_char_p
        lib.ckv_version.restype = i32
        lib.ckv_set_wait_limit_ns.argtypes = [u64]
        lib.ckv_set_wait_limit_ns.restype = u64
        _lib = lib
        return lib


def _check(rc: int, func: str):
    if rc != 0:
        msg = load_library().ckv_error_string(rc).decode()
        raise CkvError(rc, func, msg)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libckv takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libckv takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _lengths(*ts: Optional[torch.Tensor]) -> int:
    """Checks the per-request arrays (rid, seq_lens, extend_lens): int64, one
    dimension, all of one length (the batch), which is returned.  The library
    reads them as raw int64 arrays, so another dtype would be misread."""
    batch = None
    for t in ts:
        if t is None:
            continue
        if t.dtype != torch.int64 or t.dim() != 1:
            raise ValueError(f"per-request arrays must be 1-D int64 tensors (got {t.dtype}, {t.dim()}-D)")
        if batch is None:
            batch = t.numel()
        elif t.numel() != batch:
            raise ValueError(f"per-request arrays differ in length ({t.numel()} != {batch})")
    return batch or 0


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return F32
    if dt == torch.bfloat16:
        return BF16
    raise ValueError(f"unsupported dtype {dt}")


def width_of(ratio: int, head_dim: int) -> int:
    return 4 * head_dim if ratio == 4 else 2 * head_dim


def window_of(ratio: int) -> int:
    return 8 if ratio == 4 else ratio


def capacity_compress(ratio: int, batch: int, num_q_tokens: int) -> int:
    return int(load_library().ckv_capacity_compress(ratio, batch, num_q_tokens))


def capacity_write(ratio: int, batch: int, num_q_tokens: int) -> int:
    return int(load_library().ckv_capacity_write(ratio, batch, num_q_tokens))


def set_wait_limit_ns(limit_ns: int) -> int:
    """Sets the time limit of the staged kernels' waits on their copies for later launches
    (0 restores the 2 s default) and returns the previous limit."""
    if not 0 <= int(limit_ns) < 1 << 64:
        raise ValueError("limit_ns must fit an unsigned 64-bit integer")
    return int(load_library().ckv_set_wait_limit_ns(int(limit_ns)))


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word (uint32 bits, stored in an int32 tensor)."""
    return torch.zeros(4, dtype=torch.int32, device=device or "cuda")


# ------------------------------------------------------------------------------ plans
def new_decode_order(batch: int, device=None) -> torch.Tensor:
    """Storage for a decode batch's boundary-row list: ``[batch + 1, 8]`` uint8 (``ckv_decode_order_t``)."""
    return torch.empty(batch + 1, 8, dtype=torch.uint8, device=device or "cuda")


def _order(order: Optional[torch.Tensor], batch: int):
    if order is None:
        return None
    if order.dtype != torch.uint8 or order.dim() != 2 or order.shape[1] != 8 or order.shape[0] < batch + 1:
        raise ValueError("a decode order is a uint8 tensor [batch + 1, 8] (new_decode_order)")
    return _ptr(order)


def plan_decode(ratio: int, rid: torch.Tensor, seq_lens: torch.Tensor, plan_d: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None, stream=None, order: Optional[torch.Tensor] = None) -> torch.Tensor:
    """DecodePlan records ``[batch, 16]`` uint8.  With ``order`` (``new_decode_order``), the batch's
    page-boundary rows are also written there, in row order."""
    batch = _lengths(rid, seq_lens)
    if plan_d is None:
        plan_d = torch.empty(max(batch, 1), 16, dtype=torch.uint8, device=rid.device)
    _check(load_library().ckv_plan_decode(ratio, _ptr(rid), _ptr(seq_lens), batch, _ptr(plan_d),
                                          _order(order, batch), _ptr(status), _stream(stream)), "ckv_plan_decode")
    return plan_d[:batch]


def plan_prefill(ratio: int, rid: torch.Tensor, seq_lens: torch.Tensor, extend_lens: torch.Tensor,
                 num_q_tokens: int, capacity_c: Optional[int] = None, capacity_w: Optional[int] = None,
                 pad_invalid: bool = False, plan_c: Optional[torch.Tensor] = None,
                 plan_w: Optional[torch.Tensor] = None, counts: Optional[torch.Tensor] = None,
                 status: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Returns ``(plan_c [cap_c,16] u8, plan_w [cap_w,8] u8, counts [4] int32)``; counts stay on the device:
    ``{num_c, num_w, min extend_len, max extend_len}``."""
    batch = _lengths(rid, seq_lens, extend_lens)
    dev = rid.device
    if capacity_c is None:
        capacity_c = capacity_compress(ratio, batch, num_q_tokens)
    if capacity_w is None:
        capacity_w = capacity_write(ratio, batch, num_q_tokens)
    if plan_c is None:
        plan_c = torch.empty(max(capacity_c, 1), 16, dtype=torch.uint8, device=dev)
    if plan_w is None:
        plan_w = torch.empty(max(capacity_w, 1), 8, dtype=torch.uint8, device=dev)
    if counts is None:
        counts = torch.empty(4, dtype=torch.int32, device=dev)
    _check(load_library().ckv_plan_prefill(ratio, _ptr(rid), _ptr(seq_lens), _ptr(extend_lens), batch, num_q_tokens,
                                           capacity_c, capacity_w, int(pad_invalid), _ptr(plan_c), _ptr(plan_w),
                                           _ptr(counts), _ptr(status), _stream(stream)), "ckv_plan_prefill")
    return plan_c[:capacity_c], plan_w[:capacity_w], counts


def capacity_write_paged(ratio: int, batch: int, num_q_tokens: int, swa_page_size: int) -> int:
    return int(load_library().ckv_capacity_write_paged(ratio, batch, num_q_tokens, swa_page_size))


def _paged_maps(req_to_token: Optional[torch.Tensor], full_to_state: Optional[torch.Tensor]):
    """(pointer, stride, rows) of req_to_token and (pointer, size) of full_to_state; C128 takes None for both."""
    if req_to_token is None:
        return None, 0, 0, None, 0
    if req_to_token.dtype != torch.int32 or full_to_state.dtype != torch.int64 or req_to_token.dim() != 2:
        raise ValueError("req_to_token must be 2-D int32 and full_to_state int64")
    return (_ptr(req_to_token), req_to_token.shape[1], req_to_token.shape[0], _ptr(full_to_state),
            full_to_state.numel())


def plan_prefill_paged(ratio: int, rid: torch.Tensor, req_to_token: torch.Tensor, full_to_state: torch.Tensor,
                       swa_page_size: int, ring_size: int, seq_lens: torch.Tensor, extend_lens: torch.Tensor,
                       num_q_tokens: int, capacity_c: Optional[int] = None, capacity_w: Optional[int] = None,
                       pad_invalid: bool = False, counts: Optional[torch.Tensor] = None,
                       status: Optional[torch.Tensor] = None, stream=None, plan_c: Optional[torch.Tensor] = None,
                       plan_w: Optional[torch.Tensor] = None):
    """SWA-paged prefill plans; req_to_token is ``[num_reqs, stride]`` int32, full_to_state int64."""
    batch = _lengths(rid, seq_lens, extend_lens)
    dev = rid.device
    if capacity_c is None:
        capacity_c = capacity_compress(ratio, batch, num_q_tokens)
    if capacity_w is None:
        capacity_w = capacity_write_paged(ratio, batch, num_q_tokens, swa_page_size)
    if plan_c is None:
        plan_c = torch.empty(max(capacity_c, 1), 16, dtype=torch.uint8, device=dev)
    if plan_w is None:
        plan_w = torch.empty(max(capacity_w, 1), 8, dtype=torch.uint8, device=dev)
    if counts is None:
        counts = torch.empty(4, dtype=torch.int32, device=dev)
    r2t, stride, nreq, f2s, nfull = _paged_maps(req_to_token, full_to_state)
    _check(load_library().ckv_plan_prefill_paged(ratio, _ptr(rid), r2t, stride, nreq, f2s, nfull, swa_page_size,
                                                 ring_size, _ptr(seq_lens), _ptr(extend_lens), batch, num_q_tokens, capacity_c,
                                                 capacity_w, int(pad_invalid), _ptr(plan_c), _ptr(plan_w),
                                                 _ptr(counts), _ptr(status), _stream(stream)),
           "ckv_plan_prefill_paged")
    return plan_c[:capacity_c], plan_w[:capacity_w], counts


def plan_decode_paged(ratio: int, rid: torch.Tensor, req_to_token: torch.Tensor, full_to_state: torch.Tensor,
                      swa_page_size: int, ring_size: int, seq_lens: torch.Tensor,
                      status: Optional[torch.Tensor] = None, stream=None,
                      order: Optional[torch.Tensor] = None) -> torch.Tensor:
    batch = _lengths(rid, seq_lens)
    plan_d = torch.empty(max(batch, 1), 16, dtype=torch.uint8, device=rid.device)
    r2t, stride, nreq, f2s, nfull = _paged_maps(req_to_token, full_to_state)
    _check(load_library().ckv_plan_decode_paged(ratio, _ptr(rid), r2t, stride, nreq, f2s, nfull, swa_page_size,
                                                ring_size, _ptr(seq_lens), batch, _ptr(plan_d), _order(order, batch),
                                                _ptr(status), _stream(stream)),
           "ckv_plan_decode_paged")
    return plan_d[:batch]


# ------------------------------------------------------------------------------ compute
def _state_rows(state: torch.Tensor, ratio: int, head_dim: int) -> int:
    w = width_of(ratio, head_dim)
    if state.numel() % w:
        raise ValueError("state width does not match ratio / head_dim")
    return state.numel() // w


def compress_write(ratio: int, head_dim: int, state: torch.Tensor, kv_score: torch.Tensor, plan_w: torch.Tensor,
                   counts: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None, stream=None) -> None:
    _check(load_library().ckv_compress_write(ratio, head_dim, dtype_code(state.dtype), _ptr(state),
                                             _state_rows(state, ratio, head_dim), _ptr(kv_score),
                                             kv_score.shape[0], _ptr(plan_w), _ptr(counts), plan_w.shape[0],
                                             _ptr(status), _stream(stream)), "ckv_compress_write")


class PrefillHints(ctypes.Structure):
    """ckv_prefill_hints_t: the planner's rid / seq_lens / extend_lens (device pointers) and batch."""
    _fields_ = [("rid", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p), ("extend_lens", ctypes.c_void_p),
                ("batch", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


def _hints(hints):
    """``None`` or ``(rid, seq_lens, extend_lens)`` device tensors -> a ctypes pointer (or None)."""
    if hints is None:
        return None
    rid, sl, el = hints
    batch = _lengths(rid, sl, el)
    return ctypes.pointer(PrefillHints(_ptr(rid), _ptr(sl), _ptr(el), batch, 0))


def compress_pool_prefill(ratio: int, head_dim: int, state: torch.Tensor, kv_score: torch.Tensor, ape: torch.Tensor,
                          plan_c: torch.Tensor, counts: Optional[torch.Tensor] = None,
                          out_layout: int = OUT_TOKEN, out_dtype: torch.dtype = torch.float32,
                          out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                          stream=None, hints=None) -> torch.Tensor:
    """``hints``: ``None`` or the ``(rid, seq_lens, extend_lens)`` the planner read (prefetch only)."""
    nq = kv_score.shape[0]
    rows = nq if out_layout == OUT_TOKEN else plan_c.shape[0]
    if out is None:
        out = torch.empty(max(rows, 1), head_dim, dtype=out_dtype, device=kv_score.device)
    _check(load_library().ckv_compress_pool_prefill(ratio, head_dim, dtype_code(kv_score.dtype), dtype_code(out.dtype),
                                                    _ptr(state), _state_rows(state, ratio, head_dim), _ptr(kv_score),
                                                    nq, _ptr(ape), _ptr(plan_c), _ptr(counts), plan_c.shape[0],
                                                    out_layout, _ptr(out), _hints(hints), _ptr(status),
                                                    _stream(stream)),
           "ckv_compress_pool_prefill")
    return out[:rows]


def compress_prefill(ratio: int, head_dim: int, state: torch.Tensor, kv_score: torch.Tensor, ape: torch.Tensor,
                     plan_c: torch.Tensor, plan_w: torch.Tensor, counts: Optional[torch.Tensor] = None,
                     out_layout: int = OUT_TOKEN, out_dtype: torch.dtype = torch.float32,
                     out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                     stream=None, hints=None) -> torch.Tensor:
    """Pool, then write the state (one stream, in that order).  ``hints`` as compress_pool_prefill."""
    nq = kv_score.shape[0]
    rows = nq if out_layout == OUT_TOKEN else plan_c.shape[0]
    if out is None:
        out = torch.empty(max(rows, 1), head_dim, dtype=out_dtype, device=kv_score.device)
    _check(load_library().ckv_compress_prefill(ratio, head_dim, dtype_code(kv_score.dtype), dtype_code(out.dtype),
                                               _ptr(state), _state_rows(state, ratio, head_dim), _ptr(kv_score), nq,
                                               _ptr(ape), _ptr(plan_c), _ptr(plan_w), _ptr(counts), plan_c.shape[0],
                                               plan_w.shape[0], out_layout, _ptr(out), _hints(hints), _ptr(status),
                                               _stream(stream)), "ckv_compress_prefill")
    return out[:rows]


def compress_decode(ratio: int, head_dim: int, state: torch.Tensor, kv_score: torch.Tensor, ape: torch.Tensor,
                    plan_d: torch.Tensor, out_dtype: torch.dtype = torch.float32, out: Optional[torch.Tensor] = None,
                    status: Optional[torch.Tensor] = None, stream=None, order: Optional[torch.Tensor] = None,
                    rid_hint: Optional[torch.Tensor] = None, seq_lens_hint: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Decode step over ``plan_d``; ``order`` is the boundary-row list plan_decode wrote for it (optional);
    ``rid_hint`` / ``seq_lens_hint`` are the arrays plan_decode read (optional, both or neither): the decode
    prefetches its windows from them before its dependency wait."""
    batch = plan_d.shape[0]
    if (rid_hint is None) != (seq_lens_hint is None):
        raise ValueError("rid_hint and seq_lens_hint go together")
    if rid_hint is not None and _lengths(rid_hint, seq_lens_hint) != batch:
        raise ValueError("the hints need one entry per batch row")
    if out is None:
        out = torch.empty(max(batch, 1), head_dim, dtype=out_dtype, device=kv_score.device)
    _check(load_library().ckv_compress_decode(ratio, head_dim, dtype_code(kv_score.dtype), dtype_code(out.dtype),
                                              _ptr(state), _state_rows(state, ratio, head_dim), _ptr(kv_score),
                                              _ptr(ape), _ptr(plan_d), _order(order, batch), _ptr(rid_hint),
                                              _ptr(seq_lens_hint), batch, _ptr(out), _ptr(status), _stream(stream)),
           "ckv_compress_decode")
    return out[:batch]


# ------------------------------------------------------------------------------ online C128 state
def capacity_online_units(batch: int, num_q_tokens: int) -> int:
    return int(load_library().ckv_capacity_online_units(batch, num_q_tokens))


def plan_online_prefill(rid: torch.Tensor, seq_lens: torch.Tensor, extend_lens: torch.Tensor, num_q_tokens: int,
                        slot_offset: int = 0, capacity_u: Optional[int] = None, pad_invalid: bool = False,
                        units: Optional[torch.Tensor] = None, counts: Optional[torch.Tensor] = None,
                        status: Optional[torch.Tensor] = None, stream=None):
    """Returns ``(units [cap_u, 16] u8, counts [4] int32)``; counts = {num_c, num_units, min el, max el}."""
    batch = _lengths(rid, seq_lens, extend_lens)
    if capacity_u is None:
        capacity_u = capacity_online_units(batch, num_q_tokens)
    if units is None:
        units = torch.empty(max(capacity_u, 1), 16, dtype=torch.uint8, device=rid.device)
    if counts is None:
        counts = torch.empty(4, dtype=torch.int32, device=rid.device)
    _check(load_library().ckv_plan_online_prefill(_ptr(rid), _ptr(seq_lens), _ptr(extend_lens), batch, num_q_tokens,
                                                  slot_offset, capacity_u, int(pad_invalid), _ptr(units),
                                                  _ptr(counts), _ptr(status), _stream(stream)),
           "ckv_plan_online_prefill")
    return units[:capacity_u], counts


def plan_online_decode(rid: torch.Tensor, seq_lens: torch.Tensor, slot_offset: int = 0,
                       plan_d: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    batch = _lengths(rid, seq_lens)
    if plan_d is None:
        plan_d = torch.empty(max(batch, 1), 16, dtype=torch.uint8, device=rid.device)
    _check(load_library().ckv_plan_online_decode(_ptr(rid), _ptr(seq_lens), batch, slot_offset, _ptr(plan_d),
                                                 _ptr(status), _stream(stream)), "ckv_plan_online_decode")
    return plan_d[:batch]


def _online_state(state: torch.Tensor, head_dim: int) -> int:
    if state.dtype != torch.float32 or state.numel() % (3 * head_dim):
        raise ValueError("the online state is fp32 [slots, 3 * head_dim]")
    return state.numel() // (3 * head_dim)


def compress_online_prefill(head_dim: int, state: torch.Tensor, kv_score: torch.Tensor, ape: torch.Tensor,
                            units: torch.Tensor, counts: Optional[torch.Tensor], out_layout: int = OUT_TOKEN,
                            out_dtype: torch.dtype = torch.float32, out_rows: Optional[int] = None,
                            out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """Folds the units' tokens into the state; token layout out [num_q_tokens, hd], compact [out_rows, hd]."""
    nq = kv_score.shape[0]
    if out is None:
        rows = nq if out_layout == OUT_TOKEN else int(out_rows)
        out = torch.empty(max(rows, 1), head_dim, dtype=out_dtype, device=kv_score.device)
    rows = out.shape[0] if out_layout == OUT_COMPACT else nq
    _check(load_library().ckv_compress_online_prefill(head_dim, dtype_code(kv_score.dtype), dtype_code(out.dtype),
                                                      _ptr(state), _online_state(state, head_dim), _ptr(kv_score),
                                                      nq, _ptr(ape), _ptr(units), _ptr(counts), units.shape[0],
                                                      out_layout, rows, _ptr(out), _ptr(status), _stream(stream)),
           "ckv_compress_online_prefill")
    return out


def compress_online_decode(head_dim: int, state: torch.Tensor, kv_score: torch.Tensor, ape: torch.Tensor,
                           plan_d: torch.Tensor, out_dtype: torch.dtype = torch.float32,
                           out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                           stream=None) -> torch.Tensor:
    batch = plan_d.shape[0]
    if out is None:
        out = torch.empty(max(batch, 1), head_dim, dtype=out_dtype, device=kv_score.device)
    _check(load_library().ckv_compress_online_decode(head_dim, dtype_code(kv_score.dtype), dtype_code(out.dtype),
                                                     _ptr(state), _online_state(state, head_dim), _ptr(kv_score),
                                                     _ptr(ape), _ptr(plan_d), batch, _ptr(out), _ptr(status),
                                                     _stream(stream)), "ckv_compress_online_decode")
    return out[:batch]


# ------------------------------------------------------------------------------ norm, RoPE, store
def _nr_common(rows: torch.Tensor, norm_weight: torch.Tensor, freqs: torch.Tensor, kv_cache: torch.Tensor):
    if norm_weight.dtype != torch.float32 or freqs.dtype != torch.float32 or freqs.dim() != 3 or freqs.shape[2] != 2:
        raise ValueError("norm_weight must be fp32 [head_dim] and freqs fp32 [max_pos, rope_dim/2, 2]")
    head_dim = kv_cache.shape[-1]
    return head_dim, 2 * freqs.shape[1], dtype_code(rows.dtype), dtype_code(kv_cache.dtype)


def norm_rope_store_prefill(ratio: int, rows: torch.Tensor, plan_c: torch.Tensor, counts: Optional[torch.Tensor],
                            norm_weight: torch.Tensor, eps: float, freqs: torch.Tensor, out_loc: torch.Tensor,
                            kv_cache: torch.Tensor, in_layout: int = OUT_COMPACT, status: Optional[torch.Tensor] = None,
                            stream=None) -> None:
    """RMSNorm + RoPE of the pooled prefill rows, stored into ``kv_cache`` at ``out_loc[ragged_id]``."""
    hd, rope_dim, ci, cc = _nr_common(rows, norm_weight, freqs, kv_cache)
    _check(load_library().ckv_norm_rope_store_prefill(ratio, hd, rope_dim, ci, _ptr(rows), in_layout, rows.shape[0],
                                                      _ptr(plan_c), _ptr(counts), plan_c.shape[0], _ptr(norm_weight),
                                                      float(eps), _ptr(freqs), freqs.shape[0], _ptr(out_loc),
                                                      out_loc.numel(), cc, _ptr(kv_cache), kv_cache.shape[0],
                                                      _ptr(status), _stream(stream)),
           "ckv_norm_rope_store_prefill")


def norm_rope_store_decode(ratio: int, rows: torch.Tensor, plan_d: torch.Tensor, norm_weight: torch.Tensor,
                           eps: float, freqs: torch.Tensor, out_loc: torch.Tensor, kv_cache: torch.Tensor,
                           status: Optional[torch.Tensor] = None, stream=None) -> None:
    """RMSNorm + RoPE of the decode output rows (non-boundary rows stored as zeros) at ``out_loc[b]``."""
    hd, rope_dim, ci, cc = _nr_common(rows, norm_weight, freqs, kv_cache)
    if out_loc.numel() < plan_d.shape[0]:
        raise ValueError("out_loc needs one entry per batch row")
    _check(load_library().ckv_norm_rope_store_decode(ratio, hd, rope_dim, ci, _ptr(rows), _ptr(plan_d),
                                                     plan_d.shape[0], _ptr(norm_weight), float(eps), _ptr(freqs),
                                                     freqs.shape[0], _ptr(out_loc), cc, _ptr(kv_cache),
                                                     kv_cache.shape[0], _ptr(status), _stream(stream)),
           "ckv_norm_rope_store_decode")


def compress_decode_norm_rope_store(head_dim: int, state: torch.Tensor, kv_score: torch.Tensor, ape: torch.Tensor,
                                    plan_d: torch.Tensor, norm_weight: torch.Tensor, eps: float, freqs: torch.Tensor,
                                    out_loc: torch.Tensor, kv_cache: torch.Tensor,
                                    status: Optional[torch.Tensor] = None, stream=None,
                                    rid_hint: Optional[torch.Tensor] = None,
                                    seq_lens_hint: Optional[torch.Tensor] = None) -> None:
    """The C4 decode fused with norm + RoPE + store: the state write, and each row's pooled row (+0.0 off a
    group boundary) normalised, rotated and stored into ``kv_cache`` at ``out_loc[b]``."""
    if norm_weight.dtype != torch.float32 or freqs.dtype != torch.float32 or freqs.dim() != 3 or freqs.shape[2] != 2:
        raise ValueError("norm_weight must be fp32 [head_dim] and freqs fp32 [max_pos, rope_dim/2, 2]")
    if (rid_hint is None) != (seq_lens_hint is None):
        raise ValueError("rid_hint and seq_lens_hint go together")
    batch = plan_d.shape[0]
    if out_loc.dtype != torch.int64 or out_loc.numel() < batch:
        raise ValueError("out_loc must be int64 with one entry per batch row")
    _lengths(rid_hint, seq_lens_hint)
    _check(load_library().ckv_compress_decode_norm_rope_store(
        4, head_dim, 2 * freqs.shape[1], dtype_code(kv_score.dtype), _ptr(state), _state_rows(state, 4, head_dim),
        _ptr(kv_score), _ptr(ape), _ptr(plan_d), _ptr(rid_hint), _ptr(seq_lens_hint), batch, _ptr(norm_weight),
        float(eps), _ptr(freqs), freqs.shape[0], _ptr(out_loc), dtype_code(kv_cache.dtype), _ptr(kv_cache),
        kv_cache.shape[0], _ptr(status), _stream(stream)), "ckv_compress_decode_norm_rope_store")


# ------------------------------------------------------------------------------ convenience
def prefill_step(ratio: int, head_dim: int, state: torch.Tensor, kv_score: torch.Tensor, ape: torch.Tensor,
                 rid: torch.Tensor, seq_lens: torch.Tensor, extend_lens: torch.Tensor, out_layout: int = OUT_TOKEN,
                 out_dtype: torch.dtype = torch.float32, status: Optional[torch.Tensor] = None, stream=None):
    """plan_prefill -> pool -> write.  Returns ``(out, plan_c, plan_w, counts)`` (all on the device)."""
    plan_c, plan_w, counts = plan_prefill(ratio, rid, seq_lens, extend_lens, kv_score.shape[0], status=status,
                                          stream=stream)
    out = compress_prefill(ratio, head_dim, state, kv_score, ape, plan_c, plan_w, counts, out_layout, out_dtype,
                           status=status, stream=stream, hints=(rid, seq_lens, extend_lens))
    return out, plan_c, plan_w, counts


def decode_step(ratio: int, head_dim: int, state: torch.Tensor, kv_score: torch.Tensor, ape: torch.Tensor,
                rid: torch.Tensor, seq_lens: torch.Tensor, out_dtype: torch.dtype = torch.float32,
                status: Optional[torch.Tensor] = None, stream=None):
    """plan_decode (with the boundary-row list) -> decode.  Returns ``(out, plan_d)``."""
    order = new_decode_order(rid.numel(), rid.device)
    plan_d = plan_decode(ratio, rid, seq_lens, status=status, stream=stream, order=order)
    out = compress_decode(ratio, head_dim, state, kv_score, ape, plan_d, out_dtype, status=status, stream=stream,
                          order=order, rid_hint=rid, seq_lens_hint=seq_lens)
    return out, plan_d
