"""Test helpers: brute-force plan enumeration, bit-distance metrics, and the
multi-step (prefill / chunked prefill / decode) schedule driver used by the
mode-equivalence tests on both the oracle and the GPU library."""
from __future__ import annotations

import numpy as np
import torch


def window(ratio: int) -> int:
    return 8 if ratio == 4 else ratio


def slots(ratio: int) -> int:
    return 8 if ratio == 4 else 128


def brute_plan(ratio, rid, seq_lens, extend_lens):
    """Enumerates every extend position of every request and derives the plan
    from what the windows need, not from the planner's closed forms:

    * an emission happens at position p when (p+1) % ratio == 0;
    * buffer_len = number of window positions that precede the extend (held by
      the prefix state, or -- C4 first group -- before position 0);
    * a position is written to the state iff a later emission's window (one
      ending at q >= seq_len) still covers it;
    * a position's state row is rid*slots + p % slots (an 8-slot ring for C4, a
      128-slot page for C128).
    Returns (compress records [seq_len, ragged, buffer_len, state rows of the
    state-held entries], write records [ragged, write_loc])."""
    W = window(ratio)
    S = slots(ratio)
    comp, wr = [], []
    base = 0
    for b in range(len(rid)):
        sl, el, r = int(seq_lens[b]), int(extend_lens[b]), int(rid[b])
        pl = sl - el
        future = [q for q in range(sl, sl + W + ratio + 1) if (q + 1) % ratio == 0]
        for p in range(pl, sl):
            ragged = base + (p - pl)
            if (p + 1) % ratio == 0:
                win = list(range(p - W + 1, p + 1))
                held = [q for q in win if q < pl]
                rows = [r * S + q % S if q >= 0 else None for q in held]
                comp.append((p + 1, ragged, len(held), rows))
            if any(q - W + 1 <= p <= q for q in future):
                wr.append((ragged, r * S + p % S))
        base += el
    return comp, wr


def plan_c_fields(plan_c: np.ndarray) -> dict:
    w = np.ascontiguousarray(plan_c).reshape(-1, 16).view(np.uint32).reshape(-1, 4)
    return {
        "seq_len": w[:, 0].astype(np.int64),
        "ragged_id": (w[:, 1] & 0x00FFFFFF).astype(np.int64),
        "buffer_len": (w[:, 1] >> 24).astype(np.int64),
        "read_page_0": w[:, 2].view(np.int32).astype(np.int64),
        "read_page_1": w[:, 3].view(np.int32).astype(np.int64),
    }


def plan_w_fields(plan_w: np.ndarray) -> dict:
    w = np.ascontiguousarray(plan_w).reshape(-1, 8).view(np.uint32).reshape(-1, 2)
    return {"ragged_id": w[:, 0].astype(np.int64), "write_loc": w[:, 1].view(np.int32).astype(np.int64)}


def plan_d_fields(plan_d: np.ndarray) -> dict:
    w = np.ascontiguousarray(plan_d).reshape(-1, 16).view(np.uint32).reshape(-1, 4)
    return {"seq_len": w[:, 0].astype(np.int64), "write_loc": w[:, 1].view(np.int32).astype(np.int64),
            "read_page_0": w[:, 2].view(np.int32).astype(np.int64),
            "read_page_1": w[:, 3].view(np.int32).astype(np.int64)}


def expected_decode_order(plan_d: np.ndarray, ratio: int) -> np.ndarray:
    """The boundary-row list of a decode plan, derived from the oracle's records:
    rows whose record is valid and whose seq_len is a multiple of the ratio, in
    row order, as {row, read_page_0}; row 0 of the result is {count, 0}."""
    f = plan_d_fields(plan_d)
    valid = f["seq_len"] != 0xFFFFFFFF
    rows = np.nonzero(valid & (f["seq_len"] % ratio == 0))[0]
    out = np.zeros((len(rows) + 1, 2), np.uint32)
    out[0, 0] = len(rows)
    out[1:, 0] = rows
    out[1:, 1] = f["read_page_0"][rows].astype(np.int32).view(np.uint32)
    return out


def decode_order_entries(order) -> np.ndarray:
    """The written part of a device boundary-row list ([batch + 1, 8] uint8) as {row, page} uint32 pairs."""
    a = order.cpu().numpy().reshape(-1, 8).view(np.uint32).reshape(-1, 2)
    return a[: int(a[0, 0]) + 1]


def state_row_of_entry(ratio: int, i: int, rp0: int, rp1: int) -> int:
    """State row a plan record names for window entry i (C4: half-ring pages of 4
    slots, entries 0..3 in read_page_0; C128: one 128-slot page)."""
    if ratio == 4:
        return (rp0 if i < 4 else rp1) * 4 + i % 4
    return rp0 * 128 + i


# --------------------------------------------------------------------------- numeric comparisons
def ordered_int(a: np.ndarray) -> np.ndarray:
    """Maps float bit patterns to integers whose order is the float order."""
    if a.dtype == np.float32:
        i = a.view(np.int32).astype(np.int64)
        return np.where(i < 0, -(i & 0x7FFFFFFF), i)
    if a.dtype == np.uint16:  # bf16 bits
        i = a.astype(np.int64)
        return np.where(i >= 0x8000, -(i & 0x7FFF), i)
    raise TypeError(a.dtype)


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(ordered_int(a) - ordered_int(b))


def bf16_to_f32(bits16: np.ndarray) -> np.ndarray:
    return (bits16.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- schedules
def split_schedule(total: int, rng: np.random.Generator, max_chunk: int, decode_prob: float):
    """A random sequence of ('prefill', n) / ('decode', 1) steps covering ``total`` tokens."""
    steps, done = [], 0
    while done < total:
        if done > 0 and rng.random() < decode_prob:
            steps.append(("decode", 1))
            done += 1
        else:
            n = int(rng.integers(1, max_chunk + 1))
            n = min(n, total - done)
            steps.append(("prefill", n))
            done += n
    return steps


def run_schedule(backend, ratio, hd, in_dt, out_dt, histories, rids, schedules, ape, state, start=None):
    """Feeds every request's token history through its schedule.

    Each round takes, for every request, its next step; all requests whose next
    step is a prefill go into one ragged prefill call, those whose next step is
    a decode go into one decode call.  Returns per-request [T, hd] outputs in
    token layout (rows of positions that emit nothing are zero).  ``backend``
    supplies prefill(...) and decode(...).  ``start`` gives, per request, the
    number of leading positions whose state is already in place (a cached
    prefix); their output rows stay zero."""
    nreq = len(histories)
    pos = [0] * nreq if start is None else list(start)
    cursor = [0] * nreq
    outs = [np.zeros((h.shape[0], hd), dtype=np.uint16 if out_dt == 1 else np.float32) for h in histories]
    while any(cursor[b] < len(schedules[b]) for b in range(nreq)):
        pre, dec = [], []
        for b in range(nreq):
            if cursor[b] < len(schedules[b]):
                kind, n = schedules[b][cursor[b]]
                (pre if kind == "prefill" else dec).append((b, n))
        if pre:
            rows = np.concatenate([histories[b][pos[b]:pos[b] + n] for b, n in pre])
            sl = [pos[b] + n for b, n in pre]
            el = [n for b, n in pre]
            out = backend.prefill(ratio, hd, in_dt, out_dt, state, rows, ape, [rids[b] for b, _ in pre], sl, el)
            r = 0
            for b, n in pre:
                outs[b][pos[b]:pos[b] + n] = out[r:r + n]
                r += n
                pos[b] += n
                cursor[b] += 1
        if dec:
            rows = np.stack([histories[b][pos[b]] for b, _ in dec])
            sl = [pos[b] + 1 for b, _ in dec]
            out = backend.decode(ratio, hd, in_dt, out_dt, state, rows, ape, [rids[b] for b, _ in dec], sl)
            for k, (b, _) in enumerate(dec):
                outs[b][pos[b]] = out[k]
                pos[b] += 1
                cursor[b] += 1
    return outs


class OracleBackend:
    """Prefill / decode steps through the CPU oracle (state: numpy, updated in place)."""

    def __init__(self, oracle):
        self.o = oracle

    def prefill(self, ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl, el):
        out, _, _ = self.o.compress_prefill(ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl, el,
                                            out_layout=self.o.OUT_TOKEN)
        return out

    def decode(self, ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl):
        plan = self.o.plan_decode(ratio, rid, sl)
        return self.o.compress_decode(ratio, hd, in_dt, out_dt, state, rows, ape, plan)


class SwaPagedPool:
    """Token maps of an SWA-paged KV pool, as the paged planners read them.

    Every position of a request gets a slot of the full pool (req_to_token) and
    an SWA slot (full_to_state).  SWA slots come in pages of swa_page_size
    consecutive slots handed out in random order; position p of a request sits
    at offset p % swa_page_size of its (p // swa_page_size)-th page.  Full slots
    are a random permutation.  ``share`` lets a request reuse another's first
    pages, as a prefix-cache hit does."""

    def __init__(self, num_reqs: int, stride: int, swa_page_size: int, num_swa_pages: int,
                 rng: np.random.Generator):
        self.S = swa_page_size
        self.r2t = np.full((num_reqs, stride), -1, np.int32)
        self.num_full = num_reqs * stride + 5
        self.f2s = np.full(self.num_full, -1, np.int64)
        self.free_full = [int(x) for x in rng.permutation(self.num_full)]
        self.free_pages = [int(x) for x in rng.permutation(num_swa_pages)]
        self.num_swa_pages = num_swa_pages
        self.page_of = {}
        self.upto = [0] * num_reqs

    def ensure(self, rid: int, n: int) -> None:
        """Maps positions upto[rid] .. n-1 of request rid."""
        for p in range(self.upto[rid], n):
            full = self.free_full.pop()
            k = p // self.S
            if (rid, k) not in self.page_of:
                self.page_of[(rid, k)] = self.free_pages.pop()
            self.r2t[rid, p] = full
            self.f2s[full] = self.page_of[(rid, k)] * self.S + p % self.S
        self.upto[rid] = max(self.upto[rid], n)

    def share(self, rid_b: int, rid_a: int, n: int) -> None:
        """Request rid_b takes over the first n positions (whole pages) of rid_a."""
        assert n % self.S == 0 and self.upto[rid_a] >= n
        self.r2t[rid_b, :n] = self.r2t[rid_a, :n]
        for k in range(n // self.S):
            self.page_of[(rid_b, k)] = self.page_of[(rid_a, k)]
        self.upto[rid_b] = n


class PagedOracleBackend:
    """Prefill / decode steps through the oracle with SWA-paged plans."""

    def __init__(self, oracle, pool: SwaPagedPool, ring: int):
        self.o, self.pool, self.ring = oracle, pool, ring

    def prefill(self, ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl, el):
        o, pool = self.o, self.pool
        for r, s in zip(rid, sl):
            pool.ensure(r, s)
        pc, pw, (nc, nw), _ = o.plan_prefill_paged(ratio, rid, pool.r2t, pool.f2s, pool.S, self.ring, sl, el)
        out = o.compress_pool_prefill(ratio, hd, in_dt, out_dt, state, rows, ape, pc, nc, len(rows), o.OUT_TOKEN)
        o.compress_write(ratio, hd, in_dt, state, rows, pw, nw)
        return out

    def decode(self, ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl):
        o, pool = self.o, self.pool
        for r, s in zip(rid, sl):
            pool.ensure(r, s)
        plan = o.plan_decode_paged(ratio, rid, pool.r2t, pool.f2s, pool.S, self.ring, sl)
        return o.compress_decode(ratio, hd, in_dt, out_dt, state, rows, ape, plan)


def np_bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


# --------------------------------------------------------------------------- GPU-side helpers
def torch_dtype(code: int):
    return torch.bfloat16 if code == 1 else torch.float32


def to_torch(a: np.ndarray, code: int) -> torch.Tensor:
    """numpy array (bf16 as uint16 bits, or float32) -> CPU torch tensor of that dtype."""
    a = np.ascontiguousarray(a)
    if code == 1:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


def as_f32(a: np.ndarray) -> np.ndarray:
    return bf16_to_f32(a) if a.dtype == np.uint16 else a.astype(np.float32)


def window_kv_absmax_loop(ratio, hd, state, inp, seq_len, ragged, bl, rp0, rp1):
    """max_i |kv_i[c]| over each event's window (masked entries excluded): [n, hd] float64, one entry at a
    time (the plain statement of window_kv_absmax, kept to check it).  ``state`` / ``inp`` are numpy row
    arrays (bf16 bits or fp32) of the kv_score layout."""
    W = window(ratio)
    n = len(seq_len)
    out = np.zeros((n, hd))
    for k in range(n):
        first = 4 if (ratio == 4 and int(seq_len[k]) == 4) else 0
        m = np.zeros(hd)
        for i in range(first, W):
            off = (0 if i < 4 else hd) if ratio == 4 else 0
            if i < bl[k]:
                row = state[state_row_of_entry(ratio, i, int(rp0[k]), int(rp1[k]))]
            else:
                row = inp[int(ragged[k]) - (W - 1) + i]
            m = np.maximum(m, np.abs(as_f32(row[off:off + hd]).astype(np.float64)))
        out[k] = m
    return out


def window_kv_absmax(ratio, hd, state, inp, seq_len, ragged, bl, rp0, rp1, chunk: int = 64):
    """The same as window_kv_absmax_loop, gathered a chunk of events at a time (full-size workloads)."""
    W = window(ratio)
    seq_len, ragged, bl = (np.asarray(x, np.int64) for x in (seq_len, ragged, bl))
    rp0, rp1 = np.asarray(rp0, np.int64), np.asarray(rp1, np.int64)
    n = len(seq_len)
    out = np.zeros((n, hd))
    i = np.arange(W)[None, :]
    for s in range(0, n, chunk):
        e = slice(s, min(n, s + chunk))
        from_state = i < bl[e, None]
        first = np.where((ratio == 4) & (seq_len[e] == 4), 4, 0)[:, None]
        live = i >= first
        if ratio == 4:
            srow = np.where(i < 4, rp0[e, None], rp1[e, None]) * 4 + i % 4
        else:
            srow = rp0[e, None] * 128 + i
        irow = ragged[e, None] - (W - 1) + i
        # unused indices are clipped into range; their rows are masked out below
        vs = state[np.clip(np.where(from_state & live, srow, 0), 0, len(state) - 1)]
        vi = inp[np.clip(np.where(~from_state & live, irow, 0), 0, len(inp) - 1)]
        rows = np.where(from_state[..., None], vs, vi)                     # [c, W, width]
        if ratio == 4:
            kv = np.where((i < 4)[..., None], rows[..., :hd], rows[..., hd:2 * hd])
        else:
            kv = rows[..., :hd]
        a = np.abs(as_f32(kv).astype(np.float64))
        out[e] = np.where(live[..., None], a, 0.0).max(1)
    return out


def assert_pool_close(got: np.ndarray, want: np.ndarray, out_code: int, kvmax: np.ndarray = None, what=""):
    """The parity bar.  fp32 outputs: |got - want| <= 2e-6 * max|kv| of the
    window, per channel.  bf16 outputs: at most 1 ulp apart (ordered-integer
    distance of the bit patterns) -- except where the output is so much smaller
    than its window's kv that the fp32 accumulation error alone exceeds a bf16
    ulp of it (cancellation, e.g. an output of 1e-5 from kv values of ~2); there
    the fp32 bar applies to the bf16 values."""
    assert got.shape == want.shape, (got.shape, want.shape, what)
    if out_code == 1:
        d = ulp_distance(got, want)
        err = np.abs(bf16_to_f32(got).astype(np.float64) - bf16_to_f32(want).astype(np.float64))
        bad = (d > 1) & (err > 2e-6 * kvmax)
        if bad.any():
            k = tuple(np.argwhere(bad)[0])
            raise AssertionError(f"{what}: {bad.sum()} bf16 values off by >1 ulp and > 2e-6 max|kv|; first at "
                                 f"{k}: got {bf16_to_f32(got)[k]} want {bf16_to_f32(want)[k]} kvmax {kvmax[k]}")
    else:
        err = np.abs(got.astype(np.float64) - want.astype(np.float64))
        tol = 2e-6 * kvmax
        bad = err > tol
        if bad.any():
            k = tuple(np.argwhere(bad)[0])
            raise AssertionError(f"{what}: {bad.sum()} channels over tolerance, worst err/kvmax "
                                 f"{(err / np.maximum(kvmax, 1e-30)).max():.3e}; first at {k}: got {got[k]} "
                                 f"want {want[k]} kvmax {kvmax[k]}")


class GpuBackend:
    """Prefill / decode steps through libckv (state: a CUDA tensor, updated in place)."""

    def __init__(self, device="cuda"):
        from compressed_kv_attention_compressplan_gb300 import ckv

        self.ckv = ckv
        self.dev = torch.device(device)
        self.status = ckv.new_status(self.dev)

    def prefill(self, ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl, el):
        c = self.ckv
        d = self.dev
        out, _, _, _ = c.prefill_step(ratio, hd, state, to_torch(rows, in_dt).to(d), to_torch(ape, in_dt).to(d),
                                      torch.tensor(rid, dtype=torch.int64, device=d),
                                      torch.tensor(sl, dtype=torch.int64, device=d),
                                      torch.tensor(el, dtype=torch.int64, device=d), c.OUT_TOKEN,
                                      torch_dtype(out_dt), status=self.status)
        return np_bits(out)

    def decode(self, ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl):
        c = self.ckv
        d = self.dev
        out, _ = c.decode_step(ratio, hd, state, to_torch(rows, in_dt).to(d), to_torch(ape, in_dt).to(d),
                               torch.tensor(rid, dtype=torch.int64, device=d),
                               torch.tensor(sl, dtype=torch.int64, device=d), torch_dtype(out_dt),
                               status=self.status)
        return np_bits(out)


class PagedGpuBackend:
    """Prefill / decode steps through libckv with SWA-paged plans built on the GPU."""

    def __init__(self, pool: SwaPagedPool, ring: int, device="cuda"):
        from compressed_kv_attention_compressplan_gb300 import ckv

        self.ckv, self.pool, self.ring = ckv, pool, ring
        self.dev = torch.device(device)
        self.status = ckv.new_status(self.dev)

    def _maps(self):
        d = self.dev
        return torch.from_numpy(self.pool.r2t).to(d), torch.from_numpy(self.pool.f2s).to(d)

    def prefill(self, ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl, el):
        c, d, pool = self.ckv, self.dev, self.pool
        for r, s in zip(rid, sl):
            pool.ensure(r, s)
        r2t, f2s = self._maps()
        nq = len(rows)
        i64 = dict(dtype=torch.int64, device=d)
        rid_t, sl_t, el_t = torch.tensor(rid, **i64), torch.tensor(sl, **i64), torch.tensor(el, **i64)
        cap_c = c.capacity_compress(ratio, len(rid), nq)
        cap_w = c.capacity_write_paged(ratio, len(rid), nq, pool.S)
        pc, pw, counts = c.plan_prefill_paged(ratio, rid_t, r2t, f2s, pool.S, self.ring, sl_t, el_t, nq, cap_c,
                                              cap_w, status=self.status)
        out = c.compress_prefill(ratio, hd, state, to_torch(rows, in_dt).to(d), to_torch(ape, in_dt).to(d), pc, pw,
                                 counts, c.OUT_TOKEN, torch_dtype(out_dt), status=self.status)
        return np_bits(out)

    def decode(self, ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl):
        c, d, pool = self.ckv, self.dev, self.pool
        for r, s in zip(rid, sl):
            pool.ensure(r, s)
        r2t, f2s = self._maps()
        i64 = dict(dtype=torch.int64, device=d)
        pd = c.plan_decode_paged(ratio, torch.tensor(rid, **i64), r2t, f2s, pool.S, self.ring,
                                 torch.tensor(sl, **i64), status=self.status)
        out = c.compress_decode(ratio, hd, state, to_torch(rows, in_dt).to(d), to_torch(ape, in_dt).to(d), pd,
                                torch_dtype(out_dt), status=self.status)
        return np_bits(out)
