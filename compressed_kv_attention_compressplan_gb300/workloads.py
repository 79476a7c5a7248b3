"""Seeded synthetic inputs for the compressor -- shared by tests and the benchmark.

This module only draws numbers: request lengths, request pool indices, the
``kv_score`` rows, the ``ape`` bias and the prior state contents.  It holds none
of the compressor's arithmetic.  Everything is generated on the CPU from a
``torch.Generator`` seeded per tensor, so the GPU library and the CPU oracle
receive byte-identical inputs (bf16 values are drawn in fp32 and rounded to
nearest-even by ``Tensor.to``).

The five named workloads follow the shapes, value distributions and length
mixes of the compressor's serving regimes:

* ``c4_prefill_small``  C4 ragged prefill, one request, prefix 0, extend 64,
  head_dim 128, fp32 in/out, token-layout output, sentinel-filled 8-slot ring.
* ``c4_decode``         C4 decode, batch 256, seq_len ~ U[1, 8192], head_dim 512,
  bf16 input, fp32 output, ring pre-filled N(0,1).
* ``c128_decode``       C128 decode, batch 512, seq_len ~ U[1, 32768] with a
  seeded 25 % subset forced to multiples of 128, head_dim 512, bf16 -> fp32.
* ``c4_prefill``        C4 ragged prefill, batch 64, prefix ~ U[0, 4096],
  extend ~ U[1, 4096], head_dim 512, bf16 in/out, token layout.
* ``c128_prefill``      C128 ragged prefill, batch 1024: 896 requests extend by 4
  (speculative-decoding verify shape), 128 requests extend by U[128, 16384],
  prefix ~ U[0, 65536], head_dim 512, bf16 input with 1 % of the score entries
  set to +8, fp32 compact output.
* ``c4_prefill_mtp`` / ``c128_prefill_mtp``  the speculative-decoding verify
  step: batch 1024, every request extends by 4, prefix ~ U[0, 65536], head_dim
  512, bf16 input (C4: bf16 token-layout output; C128: fp32 compact output).
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import os
from typing import Optional

import torch

# Bit patterns used to fill state slots that no step has written: a quiet NaN
# with a payload, so a read of such a slot by a pooled window is visible.
SENTINEL_F32 = 0x7FC0DEAD
SENTINEL_BF16 = 0x7FDE

TOKEN = "token"
COMPACT = "compact"


@dataclasses.dataclass
class Workload:
    name: str
    mode: str                     # "prefill" or "decode"
    ratio: int                    # 4 or 128
    head_dim: int
    in_dtype: torch.dtype         # torch.float32 or torch.bfloat16
    out_dtype: torch.dtype
    out_layout: str               # TOKEN or COMPACT (prefill only)
    rid: torch.Tensor             # [B] int64 request pool index
    seq_lens: torch.Tensor        # [B] int64, length after this step
    extend_lens: Optional[torch.Tensor]  # [B] int64 (prefill) or None (decode: 1 each)
    kv_score: torch.Tensor        # [N, width] in_dtype, ragged rows (decode: N = B)
    ape: torch.Tensor             # [window, head_dim] in_dtype
    state: torch.Tensor           # [rows, width] in_dtype (C4: 8 rows per ring, C128: 128 per page)

    @property
    def batch(self) -> int:
        return int(self.rid.numel())

    @property
    def num_q_tokens(self) -> int:
        return int(self.kv_score.shape[0])

    @property
    def width(self) -> int:
        return int(self.kv_score.shape[1])

    @property
    def window(self) -> int:
        return 8 if self.ratio == 4 else self.ratio

    def describe(self) -> dict:
        d = {"workload": self.name, "mode": self.mode, "ratio": self.ratio, "head_dim": self.head_dim,
             "batch": self.batch, "num_q_tokens": self.num_q_tokens,
             "in_dtype": str(self.in_dtype).replace("torch.", ""),
             "out_dtype": str(self.out_dtype).replace("torch.", "")}
        if self.mode == "prefill":
            d["out_layout"] = self.out_layout
        return d


def width_of(ratio: int, head_dim: int) -> int:
    """Columns of one kv_score row: C4 |kv-ovl|kv|score-ovl|score|, C128 |kv|score|."""
    return 4 * head_dim if ratio == 4 else 2 * head_dim


def slots_of(ratio: int) -> int:
    """State rows owned by one request: an 8-slot ring (C4) or a 128-slot page (C128)."""
    return 8 if ratio == 4 else 128


def _seed(seed: int, k: int) -> int:
    return int(seed) * 1_000_003 + int(k)


def _gen(seed: int, k: int) -> torch.Generator:
    return torch.Generator().manual_seed(_seed(seed, k))


def normal(shape, dtype: torch.dtype, std: float, gen_seed: int, chunk: int = 1 << 22) -> torch.Tensor:
    """N(0, std^2) draws in fp32, rounded to ``dtype``.  The tensor is filled in
    fixed chunks, each from its own generator seeded by (gen_seed, chunk index),
    so the values do not depend on how many threads fill it."""
    out = torch.empty(shape, dtype=dtype)
    flat = out.view(-1)
    n = flat.numel()

    def fill(ci):
        s = ci * chunk
        e = min(n, s + chunk)
        g = torch.Generator().manual_seed(int(gen_seed) * 7919 + ci)
        t = torch.empty(e - s, dtype=torch.float32)
        t.normal_(0.0, std, generator=g)
        flat[s:e].copy_(t)

    nchunks = (n + chunk - 1) // chunk
    if nchunks <= 1:
        for ci in range(nchunks):
            fill(ci)
    else:
        with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def sentinel(shape, dtype: torch.dtype) -> torch.Tensor:
    if dtype == torch.bfloat16:
        return torch.full(shape, SENTINEL_BF16, dtype=torch.int16).view(torch.bfloat16)
    return torch.full(shape, SENTINEL_F32, dtype=torch.int32).view(torch.float32)


def set_score_outliers(kv_score: torch.Tensor, ratio: int, head_dim: int, frac: float, value: float,
                       gen: torch.Generator) -> None:
    """Sets ``value`` at round(frac * #score entries) seeded positions of the score
    columns (positions are drawn with replacement, so a few may repeat)."""
    c0 = 2 * head_dim if ratio == 4 else head_dim
    ncols = kv_score.shape[1] - c0
    n = kv_score.shape[0]
    k = int(round(frac * n * ncols))
    if k == 0:
        return
    idx = torch.randint(0, n * ncols, (k,), generator=gen, dtype=torch.int64)
    kv_score[idx // ncols, c0 + idx % ncols] = value


def make(name: str, mode: str, ratio: int, head_dim: int, in_dtype, out_dtype, out_layout, rid, seq_lens,
         extend_lens, seed: int, num_requests_state: Optional[int] = None, state_fill: str = "normal",
         outlier_frac: float = 0.0) -> Workload:
    """Builds the tensors of one workload from its lengths."""
    rid = torch.as_tensor(rid, dtype=torch.int64)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int64)
    if extend_lens is not None:
        extend_lens = torch.as_tensor(extend_lens, dtype=torch.int64)
        n = int(extend_lens.sum())
    else:
        n = int(rid.numel())
    width = width_of(ratio, head_dim)
    window = 8 if ratio == 4 else ratio
    kv_score = normal((n, width), in_dtype, 1.0, _seed(seed, 11))
    if outlier_frac > 0:
        set_score_outliers(kv_score, ratio, head_dim, outlier_frac, 8.0, _gen(seed, 12))
    ape = normal((window, head_dim), in_dtype, 0.1, _seed(seed, 13))
    nreq = int(num_requests_state if num_requests_state is not None else (int(rid.max()) + 1 if rid.numel() else 1))
    rows = nreq * slots_of(ratio)
    if state_fill == "normal":
        state = normal((rows, width), in_dtype, 1.0, _seed(seed, 14))
    else:
        state = sentinel((rows, width), in_dtype)
    return Workload(name, mode, ratio, head_dim, in_dtype, out_dtype, out_layout, rid, seq_lens, extend_lens,
                    kv_score, ape, state)


# ----------------------------------------------------------------------------- named workloads
def c4_prefill_small(seed: int = 0) -> Workload:
    return make("c4_prefill_small", "prefill", 4, 128, torch.float32, torch.float32, TOKEN,
                rid=[0], seq_lens=[64], extend_lens=[64], seed=seed, num_requests_state=1, state_fill="sentinel")


def c4_decode(seed: int = 0, batch: int = 256, head_dim: int = 512) -> Workload:
    g = _gen(seed, 1)
    seq_lens = torch.randint(1, 8192 + 1, (batch,), generator=g, dtype=torch.int64)
    rid = torch.randperm(batch, generator=_gen(seed, 2))
    return make("c4_decode", "decode", 4, head_dim, torch.bfloat16, torch.float32, TOKEN, rid, seq_lens, None,
                seed, num_requests_state=batch)


def c128_decode_lengths(seed: int = 0, batch: int = 512):
    """(rid, seq_lens) of the C128 decode workload: seq_len ~ U[1, 32768], a quarter on page boundaries."""
    g = _gen(seed, 1)
    seq_lens = torch.randint(1, 32768 + 1, (batch,), generator=g, dtype=torch.int64)
    forced = torch.randperm(batch, generator=_gen(seed, 3))[: batch // 4]
    seq_lens[forced] = 128 * torch.randint(1, 256 + 1, (forced.numel(),), generator=_gen(seed, 4),
                                           dtype=torch.int64)
    rid = torch.randperm(batch, generator=_gen(seed, 2))
    return rid, seq_lens


def c128_decode(seed: int = 0, batch: int = 512, head_dim: int = 512) -> Workload:
    rid, seq_lens = c128_decode_lengths(seed, batch)
    return make("c128_decode", "decode", 128, head_dim, torch.bfloat16, torch.float32, TOKEN, rid, seq_lens,
                None, seed, num_requests_state=batch)


def c4_prefill_lengths(seed: int = 0, batch: int = 64, max_prefix: int = 4096, max_extend: int = 4096):
    """(rid, seq_lens, extend_lens) of the C4 prefill workload."""
    pl = torch.randint(0, max_prefix + 1, (batch,), generator=_gen(seed, 1), dtype=torch.int64)
    el = torch.randint(1, max_extend + 1, (batch,), generator=_gen(seed, 5), dtype=torch.int64)
    rid = torch.randperm(batch, generator=_gen(seed, 2))
    return rid, pl + el, el


def c4_prefill(seed: int = 0, batch: int = 64, head_dim: int = 512, **lengths) -> Workload:
    rid, sl, el = c4_prefill_lengths(seed, batch, **lengths)
    return make("c4_prefill", "prefill", 4, head_dim, torch.bfloat16, torch.bfloat16, TOKEN, rid, sl, el,
                seed, num_requests_state=batch)


def c128_prefill_lengths(seed: int = 0, batch: int = 1024, num_long: int = 128, short_extend: int = 4,
                         long_extend=(128, 16384), max_prefix: int = 65536):
    """(rid, seq_lens, extend_lens) of the C128 prefill workload."""
    el = torch.full((batch,), short_extend, dtype=torch.int64)
    long_ids = torch.randperm(batch, generator=_gen(seed, 6))[:num_long]
    el[long_ids] = torch.randint(long_extend[0], long_extend[1] + 1, (num_long,), generator=_gen(seed, 5),
                                 dtype=torch.int64)
    pl = torch.randint(0, max_prefix + 1, (batch,), generator=_gen(seed, 1), dtype=torch.int64)
    rid = torch.randperm(batch, generator=_gen(seed, 2))
    return rid, pl + el, el


def c128_prefill(seed: int = 0, batch: int = 1024, head_dim: int = 512, **lengths) -> Workload:
    rid, sl, el = c128_prefill_lengths(seed, batch, **lengths)
    return make("c128_prefill", "prefill", 128, head_dim, torch.bfloat16, torch.float32, COMPACT, rid, sl, el,
                seed, num_requests_state=batch, outlier_frac=0.01)


def c128_prefill_mtp(seed: int = 0, batch: int = 1024, extend: int = 4, head_dim: int = 512,
                     max_prefix: int = 65536) -> Workload:
    """Speculative-decoding verify step: every request extends by the same few tokens."""
    el = torch.full((batch,), extend, dtype=torch.int64)
    pl = torch.randint(0, max_prefix + 1, (batch,), generator=_gen(seed, 1), dtype=torch.int64)
    rid = torch.randperm(batch, generator=_gen(seed, 2))
    return make("c128_prefill_mtp", "prefill", 128, head_dim, torch.bfloat16, torch.float32, COMPACT, rid, pl + el,
                el, seed, num_requests_state=batch)


def c4_prefill_mtp(seed: int = 0, batch: int = 1024, extend: int = 4, head_dim: int = 512,
                   max_prefix: int = 65536) -> Workload:
    el = torch.full((batch,), extend, dtype=torch.int64)
    pl = torch.randint(0, max_prefix + 1, (batch,), generator=_gen(seed, 1), dtype=torch.int64)
    rid = torch.randperm(batch, generator=_gen(seed, 2))
    return make("c4_prefill_mtp", "prefill", 4, head_dim, torch.bfloat16, torch.bfloat16, TOKEN, rid, pl + el, el,
                seed, num_requests_state=batch)


NAMED = {
    "c4_prefill_small": c4_prefill_small,
    "c4_decode": c4_decode,
    "c128_decode": c128_decode,
    "c4_prefill": c4_prefill,
    "c128_prefill": c128_prefill,
    "c4_prefill_mtp": c4_prefill_mtp,
    "c128_prefill_mtp": c128_prefill_mtp,
}


# ----------------------------------------------------------------------------- SWA-paged state
@dataclasses.dataclass
class PagedMaps:
    """The token maps of an SWA-paged pool, as the paged planners read them."""
    swa_page_size: int
    ring_size: int
    req_to_token: torch.Tensor   # int32 [num_requests, stride]: full-pool slot of each position
    full_to_state: torch.Tensor  # int64 [num_full_slots]: SWA slot of each full-pool slot
    num_pages: int


def swa_paged_maps(rid, seq_lens, num_requests: int, swa_page_size: int, ring_size: int, seed: int) -> PagedMaps:
    """A seeded page-granular allocation: position p of request rid gets a full-pool slot (a seeded
    permutation) and the SWA slot at offset p % swa_page_size of the request's (p // swa_page_size)-th
    SWA page; the pages are handed out in seeded random order."""
    sl = [int(x) for x in seq_lens]
    stride = max(sl) if sl else 1
    npages = [(x + swa_page_size - 1) // swa_page_size for x in sl]
    num_pages = max(1, sum(npages))
    pages = torch.randperm(num_pages, generator=_gen(seed, 41))
    num_full = max(1, sum(sl))
    full = torch.randperm(num_full, generator=_gen(seed, 42))
    r2t = torch.full((num_requests, stride), -1, dtype=torch.int32)
    f2s = torch.full((num_full,), -1, dtype=torch.int64)
    fo = po = 0
    for r, n, npg in zip([int(x) for x in rid], sl, npages):
        p = torch.arange(n, dtype=torch.int64)
        slots = full[fo:fo + n]
        r2t[r, :n] = slots.to(torch.int32)
        f2s[slots] = pages[po + p // swa_page_size] * swa_page_size + p % swa_page_size
        fo += n
        po += npg
    return PagedMaps(swa_page_size, ring_size, r2t, f2s, num_pages)


def c4_prefill_paged(seed: int = 0, head_dim: int = 512, swa_page_size: int = 128, ring_size: int = 8):
    """The C4 prefill workload over SWA-paged state (128-token SWA pages, 8-row rings): (Workload, PagedMaps)."""
    rid, sl, el = c4_prefill_lengths(seed)
    maps = swa_paged_maps(rid, sl, rid.numel(), swa_page_size, ring_size, seed)
    w = make("c4_prefill_paged", "prefill", 4, head_dim, torch.bfloat16, torch.bfloat16, TOKEN, rid, sl, el, seed,
             num_requests_state=1, state_fill="sentinel")
    w.state = normal((maps.num_pages * ring_size, width_of(4, head_dim)), torch.bfloat16, 1.0, _seed(seed, 14))
    return w, maps


PAGED = {"c4_prefill_paged": c4_prefill_paged}


# ----------------------------------------------------------------------------- norm + RoPE + store inputs
def rope_table(max_pos: int, rope_dim: int, base: float = 10000.0) -> torch.Tensor:
    """fp32 [max_pos, rope_dim/2, 2]: cos / sin of pos * base^(-2i/rope_dim), formed in float64."""
    inv = base ** (-torch.arange(0, rope_dim, 2, dtype=torch.float64) / rope_dim)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.stack([torch.cos(ang), torch.sin(ang)], dim=-1).to(torch.float32)


@dataclasses.dataclass
class NormRopeInputs:
    """Inputs of the norm + RoPE + store step over the compressed rows of a workload."""
    name: str
    ratio: int
    head_dim: int
    rope_dim: int
    rid: torch.Tensor
    seq_lens: torch.Tensor
    extend_lens: Optional[torch.Tensor]   # None: decode
    rows: torch.Tensor        # fp32 [num_rows, head_dim] (prefill: compact, one per compress record)
    weight: torch.Tensor      # fp32 [head_dim]
    eps: float
    freqs: torch.Tensor       # fp32 [max_pos, rope_dim/2, 2]
    out_loc: torch.Tensor     # int64, one cache row per token (prefill) or per batch row (decode)
    cache_rows: int
    cache_dtype: torch.dtype


def norm_rope_c128_prefill(seed: int = 0, head_dim: int = 512, rope_dim: int = 64) -> NormRopeInputs:
    """The compressed rows of the C128 prefill workload (compact fp32) into a bf16 cache."""
    rid, sl, el = c128_prefill_lengths(seed)
    nq = int(el.sum())
    # at least one row per compress record (a request adds at most extend_len / 128 + 1)
    rows = normal((nq // 128 + rid.numel(), head_dim), torch.float32, 1.0, _seed(seed, 21))
    weight = 1.0 + normal((head_dim,), torch.float32, 0.1, _seed(seed, 22))
    cache_rows = nq  # every token owns a distinct cache row
    out_loc = torch.randperm(cache_rows, generator=_gen(seed, 23)).to(torch.int64)
    return NormRopeInputs("norm_rope_c128_prefill", 128, head_dim, rope_dim, rid, sl, el, rows, weight, 1e-6,
                          rope_table(int(sl.max()) + 1, rope_dim), out_loc, cache_rows, torch.bfloat16)


def norm_rope_c128_decode(seed: int = 0, head_dim: int = 512, rope_dim: int = 64) -> NormRopeInputs:
    """The decode output rows of the C128 decode workload into a bf16 cache."""
    rid, sl = c128_decode_lengths(seed)
    batch = rid.numel()
    rows = normal((batch, head_dim), torch.float32, 1.0, _seed(seed, 21))
    weight = 1.0 + normal((head_dim,), torch.float32, 0.1, _seed(seed, 22))
    cache_rows = 4 * batch
    out_loc = torch.randperm(cache_rows, generator=_gen(seed, 23))[:batch].to(torch.int64)
    return NormRopeInputs("norm_rope_c128_decode", 128, head_dim, rope_dim, rid, sl, None, rows, weight, 1e-6,
                          rope_table(int(sl.max()) + 1, rope_dim), out_loc, cache_rows, torch.bfloat16)


NORM_ROPE = {"norm_rope_c128_prefill": norm_rope_c128_prefill, "norm_rope_c128_decode": norm_rope_c128_decode}


@dataclasses.dataclass
class DecodeNormInputs:
    """A decode workload plus the norm + RoPE + store inputs of its output rows."""
    w: "Workload"
    rope_dim: int
    weight: torch.Tensor      # fp32 [head_dim]
    eps: float
    freqs: torch.Tensor       # fp32 [max_pos, rope_dim/2, 2]
    out_loc: torch.Tensor     # int64 [batch]
    cache_rows: int
    cache_dtype: torch.dtype


def c4_decode_norm_rope(seed: int = 0, rope_dim: int = 64) -> DecodeNormInputs:
    """The C4 decode workload whose output rows go through norm + RoPE into a bf16 cache."""
    w = c4_decode(seed)
    hd, batch = w.head_dim, w.batch
    weight = 1.0 + normal((hd,), torch.float32, 0.1, _seed(seed, 22))
    cache_rows = 4 * batch
    out_loc = torch.randperm(cache_rows, generator=_gen(seed, 23))[:batch].to(torch.int64)
    return DecodeNormInputs(w, rope_dim, weight, 1e-6, rope_table(int(w.seq_lens.max()) + 1, rope_dim), out_loc,
                            cache_rows, torch.bfloat16)


DECODE_NORM = {"c4_decode_norm_rope": c4_decode_norm_rope}


# ----------------------------------------------------------------------------- online C128 state inputs
@dataclasses.dataclass
class OnlineInputs:
    """A C128 step through the online state.  The state of each request's
    current group is not drawn: the earlier tokens of that group are
    (prefix_rows, prefix_lens tokens per request, batch order), and the caller
    folds them into the state before the step."""
    name: str
    mode: str                # "prefill" | "decode"
    head_dim: int
    rid: torch.Tensor
    seq_lens: torch.Tensor
    extend_lens: Optional[torch.Tensor]
    kv_score: torch.Tensor   # bf16 [num_q_tokens or batch, 2 * head_dim]
    ape: torch.Tensor        # bf16 [128, head_dim]
    prefix_rows: torch.Tensor
    prefix_lens: torch.Tensor
    out_dtype: torch.dtype
    out_layout: str


def c128_online_prefill(seed: int = 0, head_dim: int = 512, num_long: int = 128, lengths=None) -> OnlineInputs:
    """The C128 prefill workload's lengths and inputs, through the online state (or the given
    ``(rid, seq_lens, extend_lens)``)."""
    rid, sl, el = c128_prefill_lengths(seed, num_long=num_long) if lengths is None else lengths
    nq = int(el.sum())
    kv = normal((nq, 2 * head_dim), torch.bfloat16, 1.0, _seed(seed, 11))
    set_score_outliers(kv, 128, head_dim, 0.01, 8.0, _gen(seed, 12))
    ape = normal((128, head_dim), torch.bfloat16, 0.1, _seed(seed, 13))
    part = (sl - el) % 128
    prefix = normal((int(part.sum()), 2 * head_dim), torch.bfloat16, 1.0, _seed(seed, 31))
    return OnlineInputs("c128_online_prefill", "prefill", head_dim, rid, sl, el, kv, ape, prefix, part,
                        torch.float32, COMPACT)


def c128_online_decode(seed: int = 0, head_dim: int = 512) -> OnlineInputs:
    """The C128 decode workload's lengths and inputs, through the online state."""
    rid, sl = c128_decode_lengths(seed)
    kv = normal((rid.numel(), 2 * head_dim), torch.bfloat16, 1.0, _seed(seed, 11))
    ape = normal((128, head_dim), torch.bfloat16, 0.1, _seed(seed, 13))
    part = (sl - 1) % 128
    prefix = normal((int(part.sum()), 2 * head_dim), torch.bfloat16, 1.0, _seed(seed, 31))
    return OnlineInputs("c128_online_decode", "decode", head_dim, rid, sl, None, kv, ape, prefix, part,
                        torch.float32, TOKEN)


ONLINE = {"c128_online_prefill": c128_online_prefill, "c128_online_decode": c128_online_decode}


def random_prefill(ratio: int, head_dim: int, in_dtype, out_dtype, out_layout: str, prefix_lens, extend_lens,
                   seed: int, num_requests_state: Optional[int] = None, rid=None,
                   state_fill: str = "normal", outlier_frac: float = 0.0) -> Workload:
    """A prefill workload with the given per-request lengths (rid = seeded permutation by default)."""
    pl = torch.as_tensor(prefix_lens, dtype=torch.int64)
    el = torch.as_tensor(extend_lens, dtype=torch.int64)
    if rid is None:
        nreq = num_requests_state if num_requests_state is not None else len(pl)
        rid = torch.randperm(nreq, generator=_gen(seed, 2))[: len(pl)]
    rid = torch.as_tensor(rid, dtype=torch.int64)
    return make("random_prefill", "prefill", ratio, head_dim, in_dtype, out_dtype, out_layout, rid, pl + el, el,
                seed, num_requests_state=num_requests_state, state_fill=state_fill, outlier_frac=outlier_frac)


def random_decode(ratio: int, head_dim: int, in_dtype, out_dtype, seq_lens, seed: int,
                  num_requests_state: Optional[int] = None, rid=None) -> Workload:
    sl = torch.as_tensor(seq_lens, dtype=torch.int64)
    if rid is None:
        nreq = num_requests_state if num_requests_state is not None else len(sl)
        rid = torch.randperm(nreq, generator=_gen(seed, 2))[: len(sl)]
    return make("random_decode", "decode", ratio, head_dim, in_dtype, out_dtype, TOKEN, rid, sl, None, seed,
                num_requests_state=num_requests_state)


def bits(t: torch.Tensor):
    """numpy view of a CPU tensor as the oracle takes it (bf16 -> uint16 bit patterns)."""
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
