"""Pins of the oracle's online C128 state (a running softmax per request slot,
reset at every 128-group start; compressor_v2.py's online compression, whose
kernels are off-page -- the recurrence is derived in ckv_oracle.c).

Anchors outside the recurrence: the whole-history window definition
(compress_history) for one prefill, chunked prefills, token-by-token decode
and mixed schedules; the window-mean and dominant-entry closed forms; a
hand-derived unit plan; unit plans rebuilt by classifying every token.
"""
import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H

HD = 128


class OnlineOracleBackend:
    """Prefill / decode steps through the oracle's online state (float64 [slots, 3 hd])."""

    def __init__(self, o, slot_offset=0):
        self.o, self.off = o, slot_offset

    def prefill(self, ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl, el):
        units, _, _ = self.o.plan_online_prefill(rid, sl, el, self.off)
        return self.o.online_prefill(hd, in_dt, out_dt, state, rows, ape, units)

    def decode(self, ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl):
        plan = self.o.plan_online_decode(rid, sl, self.off)
        return self.o.online_decode(hd, in_dt, out_dt, state, rows, ape, plan)


def _close(got, want, kvmax, what):
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    assert (err <= 2.0 ** -22 * kvmax).all(), (what, float(err.max()))


@pytest.mark.parametrize("seed", [0, 1])
def test_online_schedules_equal_window_definition(oracle_mod, seed):
    o = oracle_mod
    rng = np.random.default_rng(40 + seed)
    nreq = 4
    lens = [int(rng.integers(1, 3 * 128 + 60)) for _ in range(nreq)]
    rids = [int(x) for x in rng.permutation(6)[:nreq]]
    in_dt, out_dt = (1, 0) if seed == 0 else (0, 0)
    tdt = torch.bfloat16 if in_dt else torch.float32
    g = torch.Generator().manual_seed(70 + seed)
    hist = [wl.bits(torch.randn(n, 2 * HD, generator=g).to(tdt)).copy() for n in lens]
    ape = wl.bits((torch.randn(128, HD, generator=g) * 0.5).to(tdt)).copy()
    want = [o.compress_history(128, HD, in_dt, out_dt, h, ape) for h in hist]
    kvmax = [np.abs(H.as_f32(h[:, :HD])).max() for h in hist]
    backend = OnlineOracleBackend(o, slot_offset=2)
    for mode in ["oneshot", "chunked", "decode", "mixed"]:
        if mode == "oneshot":
            sched = [[("prefill", n)] for n in lens]
        elif mode == "chunked":
            sched = [H.split_schedule(n, rng, 150, 0.0) for n in lens]
        elif mode == "decode":
            sched = [[("decode", 1)] * n for n in lens]
        else:
            sched = [H.split_schedule(n, rng, 70, 0.5) for n in lens]
        state = np.full((8 + 2, 3 * HD), np.nan)  # never-written slots poison a wrong load
        got = H.run_schedule(backend, 128, HD, in_dt, out_dt, hist, rids, sched, ape, state)
        for b in range(nreq):
            _close(got[b], want[b], kvmax[b], (mode, b))


def test_online_closed_forms(oracle_mod):
    o = oracle_mod
    T = 256
    kv = np.arange(T * HD, dtype=np.float64).reshape(T, HD) % 7 - 3
    tok = np.zeros((T, 2 * HD), np.float32)
    tok[:, :HD] = kv
    ape0 = np.zeros((128, HD), np.float32)
    state = np.zeros((1, 3 * HD))
    units, _, _ = o.plan_online_prefill([0], [T], [T])
    out = o.online_prefill(HD, 0, 0, state, tok, ape0, units)
    for g in range(2):  # equal scores: the group mean
        np.testing.assert_allclose(out[128 * g + 127], kv[128 * g:128 * g + 128].mean(0), rtol=0, atol=1e-6)
    tok[200, HD:] = 200.0  # a dominant score selects its token's kv
    state[:] = 0
    out = o.online_prefill(HD, 0, 0, state, tok, ape0, units)
    assert (out[255] == kv[200].astype(np.float32)).all()
    assert (np.delete(out, [127, 255], axis=0) == 0).all()


def test_online_plan_worked_example(oracle_mod):
    """Request rid 3 prefills 300 tokens from scratch; request rid 0 extends
    positions 5..9 (slot offset 2): units (position, ragged, count, slot,
    output row, flags LOAD=1 EMIT=2 STORE=4) worked out by hand."""
    o = oracle_mod
    units, (nu, nc), _ = o.plan_online_prefill([3, 0], [300, 10], [300, 5], slot_offset=2)
    w = units.view(np.uint32).reshape(-1, 4)
    got = [(int(r[0]), int(r[1] & 0xFFFFFF), int(r[1] >> 24), int(r[2]), int(r[3] & 0xFFFFFF), int(r[3] >> 24))
           for r in w]
    assert (nu, nc) == (4, 2)
    assert got == [(0, 0, 128, 5, 0, 2), (128, 128, 128, 5, 1, 2), (256, 256, 44, 5, 0xFFFFFF, 4),
                   (5, 300, 5, 2, 0xFFFFFF, 5)]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_online_plan_bruteforce(oracle_mod, seed):
    """Every extend token, classified on its own, groups into exactly the units."""
    o = oracle_mod
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 9))
    sl = rng.integers(1, 700, B)
    el = np.array([int(rng.integers(1, s + 1)) for s in sl])
    rid = rng.permutation(B)
    units, (nu, nc), _ = o.plan_online_prefill(rid, sl, el, slot_offset=1)
    w = units.view(np.uint32).reshape(-1, 4)
    want, base, row = [], 0, 0
    for b in range(B):
        pl = int(sl[b] - el[b])
        groups = {}
        for j in range(int(el[b])):
            groups.setdefault((pl + j) // 128, []).append(pl + j)
        for gi in sorted(groups):
            ps = groups[gi]
            emit = ps[-1] % 128 == 127
            flags = (1 if ps[0] % 128 else 0) | (2 if emit else 0) | (4 if ps[-1] == sl[b] - 1 else 0)
            want.append((ps[0], base + ps[0] - pl, len(ps), int(rid[b]) + 1, row if emit else 0xFFFFFF, flags))
            row += emit
        base += int(el[b])
    got = [(int(r[0]), int(r[1] & 0xFFFFFF), int(r[1] >> 24), int(r[2]), int(r[3] & 0xFFFFFF), int(r[3] >> 24))
           for r in w]
    assert got == want and nu == len(want) and nc == row
    # padding: the tail of a larger buffer is the invalid record
    padded, _, _ = o.plan_online_prefill(rid, sl, el, 1, cap_u=nu + 3, pad_invalid=True)
    assert (padded[:nu] == units).all() and (padded[nu:] == 0xFF).all()
