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


def run_schedule(backend, ratio, hd, in_dt, out_dt, histories, rids, schedules, ape, state):
    """Feeds every request's token history through its schedule.

    Each round takes, for every request, its next step; all requests whose next
    step is a prefill go into one ragged prefill call, those whose next step is
    a decode go into one decode call.  Returns per-request [T, hd] outputs in
    token layout (rows of positions that emit nothing are zero).  ``backend``
    supplies prefill(...) and decode(...)."""
    nreq = len(histories)
    pos = [0] * nreq
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


def window_kv_absmax(ratio, hd, state, inp, seq_len, ragged, bl, rp0, rp1):
    """max_i |kv_i[c]| over each event's window (masked entries excluded): [n, hd] float64.
    ``state`` / ``inp`` are numpy row arrays (bf16 bits or fp32) of the kv_score layout."""
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
