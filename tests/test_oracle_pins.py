"""Pins of the CPU oracle against facts that c_plan.cuh, compressor_v2.py,
c4.cuh and the mathematics fix.

Nothing here compares the oracle with itself: the plan is checked against a
hand-worked example and a brute-force enumeration of what the windows need,
the pool against closed forms (window mean, dominant entry, tagged columns),
against float64 ``torch.softmax`` on tiny shapes, and the drivers against the
stateless whole-history definition (one prefill == chunked prefill == decode).
"""
import json
import os

import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ----------------------------------------------------------------------------- plans
def test_plan_worked_examples(oracle_mod):
    o = oracle_mod
    g = json.load(open(os.path.join(GOLDEN, "plans_worked.json")))
    for case in g["prefill"]:
        pc, pw, (nc, nw), _ = o.plan_prefill(case["ratio"], case["rid"], case["seq_lens"], case["extend_lens"])
        f = H.plan_c_fields(pc)
        got = np.stack([f["seq_len"], f["ragged_id"], f["buffer_len"], f["read_page_0"], f["read_page_1"]], 1)
        assert got.tolist() == case["compress"], case["name"]
        fw = H.plan_w_fields(pw)
        if "write" in case:
            assert np.stack([fw["ragged_id"], fw["write_loc"]], 1).tolist() == case["write"], case["name"]
        else:
            rule = case["write_rule"]
            assert nw == rule["count"]
            assert fw["ragged_id"].tolist() == list(range(rule["ragged_first"], rule["ragged_first"] + nw))
            assert fw["write_loc"].tolist() == list(range(rule["write_loc_first"], rule["write_loc_first"] + nw))
    for case in g["decode"]:
        pd = o.plan_decode(case["ratio"], [case["rid"]], [case["seq_len"]])
        f = H.plan_d_fields(pd)
        got = [int(f["seq_len"][0]), int(f["write_loc"][0]), int(f["read_page_0"][0]), int(f["read_page_1"][0])]
        assert got == case["plan"], case


@pytest.mark.parametrize("ratio", [4, 128])
@pytest.mark.parametrize("seed", range(6))
def test_plan_bruteforce(oracle_mod, ratio, seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 24))
    span = 3 * ratio + 20
    pl = rng.integers(0, span, B)
    el = rng.integers(1, span, B)
    if seed == 0:
        el[:] = 1  # decode-like prefill steps
    rid = rng.permutation(64)[:B]
    sl = pl + el
    pc, pw, (nc, nw), _ = oracle_mod.plan_prefill(ratio, rid, sl, el)
    comp, wr = H.brute_plan(ratio, rid, sl, el)
    assert nc == len(comp) and nw == len(wr)
    f = H.plan_c_fields(pc)
    for k, (seq_len, ragged, held, rows) in enumerate(comp):
        assert f["seq_len"][k] == seq_len and f["ragged_id"][k] == ragged and f["buffer_len"][k] == held
        for i, row in enumerate(rows):
            if row is not None:
                assert H.state_row_of_entry(ratio, i, f["read_page_0"][k], f["read_page_1"][k]) == row
    fw = H.plan_w_fields(pw)
    assert list(zip(fw["ragged_id"].tolist(), fw["write_loc"].tolist())) == wr


def test_plan_padding_capacity_and_validation(oracle_mod):
    o = oracle_mod
    pc, pw, (nc, nw), rc = o.plan_prefill(4, [0, 1], [9, 12], [9, 4], cap_c=8, cap_w=16, pad_invalid=True)
    assert rc == 0 and (nc, nw) == (3, 9)  # (p=3,7 | p=11); writes p=4..8 | p=8..11
    assert (pc[nc:] == 0xFF).all() and (pw[nw:] == 0xFF).all()
    _, _, _, rc = o.plan_prefill(4, [0, 1], [9, 12], [9, 4], cap_c=2, cap_w=16, check=False)
    assert rc == o.CAPACITY
    _, _, _, rc = o.plan_prefill(4, [0], [9], [0], num_q_tokens=0, cap_c=4, cap_w=4, check=False)
    assert rc == o.BAD_LENGTH
    _, _, _, rc = o.plan_prefill(4, [0], [9], [10], num_q_tokens=10, cap_c=4, cap_w=4, check=False)
    assert rc == o.BAD_LENGTH
    _, _, _, rc = o.plan_prefill(4, [0], [9], [5], num_q_tokens=6, cap_c=4, cap_w=8, check=False)
    assert rc == o.BAD_TOTAL
    _, _, _, rc = o.plan_prefill(3, [0], [9], [5], check=False)
    assert rc == o.BAD_RATIO


# ----------------------------------------------------------------------------- bf16 rounding
def test_bf16_round_once(oracle_mod):
    o = oracle_mod
    # ties go to the even neighbour; a value just above a tie rounds up (a second
    # rounding through fp32 would lose the 2^-40 and round down)
    assert o.double_to_bf16(1.0 + 2 ** -8) == 0x3F80
    assert o.double_to_bf16(1.0 + 3 * 2 ** -8) == 0x3F82
    assert o.double_to_bf16(1.0 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert o.double_to_bf16(-2.0) == 0xC000
    assert o.double_to_bf16(0.0) == 0 and o.double_to_bf16(-0.0) == 0x8000
    assert o.double_to_bf16(3.5e38) == 0x7F80  # above the largest finite bf16 after rounding
    assert o.double_to_bf16(2.0 ** -133) == 0x0001  # smallest subnormal
    # for fp32 inputs a single rounding is what torch's fp32 -> bf16 conversion does
    x = torch.randn(20000, generator=torch.Generator().manual_seed(7)) * torch.logspace(-30, 30, 20000)
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([o.double_to_bf16(float(v)) for v in x.tolist()], dtype=np.uint16)
    assert (ref == got).all()


# ----------------------------------------------------------------------------- pool closed forms
def _one_request(ratio, hd, dtype, T, seed, state_fill="sentinel"):
    w = wl.random_prefill(ratio, hd, dtype, torch.float32, wl.TOKEN, [0], [T], seed, num_requests_state=1,
                          rid=[0], state_fill=state_fill)
    return w


@pytest.mark.parametrize("ratio", [4, 128])
def test_equal_scores_give_window_mean(oracle_mod, ratio):
    o = oracle_mod
    hd = 128
    W = H.window(ratio)
    T = 2 * W if ratio == 128 else 24
    rng = np.random.default_rng(1)
    width = wl.width_of(ratio, hd)
    tok = np.zeros((T, width), np.float32)
    kvcols = [slice(0, 2 * hd)] if ratio == 4 else [slice(0, hd)]
    for c in kvcols:
        tok[:, c] = rng.integers(-50, 51, (T, c.stop - c.start))
    tok[:, 2 * hd if ratio == 4 else hd:] = 0.75  # all scores equal
    ape = np.zeros((W, hd), np.float32)
    out = o.compress_history(ratio, hd, o.F32, o.F32, tok, ape)
    for p in range(T):
        if (p + 1) % ratio:
            assert (out[p] == 0).all()
            continue
        if ratio == 4:
            ent = [(q, 0 if i < 4 else hd) for i, q in enumerate(range(p - 7, p + 1)) if q >= 0]
        else:
            ent = [(q, 0) for q in range(p - 127, p + 1)]
        want = np.zeros(hd)
        for q, off in ent:
            want += tok[q, off:off + hd]
        want /= len(ent)  # divisions by 4, 8, 128: exact
        assert (out[p] == want.astype(np.float32)).all(), p


@pytest.mark.parametrize("ratio", [4, 128])
def test_dominant_ape_selects_entry_and_column(oracle_mod, ratio):
    """ape[i][c] = +60 for one window index i per channel (others 0), equal scores:
    channel c must return exactly kv of window entry i(c), from the right column half."""
    o = oracle_mod
    hd = 128
    W = H.window(ratio)
    T = 3 * ratio if ratio == 128 else 20
    width = wl.width_of(ratio, hd)
    tok = np.zeros((T, width), np.float32)
    q = np.arange(T, dtype=np.float32)[:, None]
    ch = np.arange(hd, dtype=np.float32)[None, :]
    if ratio == 4:
        tok[:, 0:hd] = 1000.0 + q + ch / 256.0      # kv overlap half: tag 1000 + position
        tok[:, hd:2 * hd] = q + ch / 256.0          # kv main half: tag = position
    else:
        tok[:, 0:hd] = q + ch / 256.0
    pick = (np.arange(hd) * 7 + 3) % W
    ape = np.zeros((W, hd), np.float32)
    ape[pick, np.arange(hd)] = 60.0
    out = o.compress_history(ratio, hd, o.F32, o.F32, tok, ape)
    for p in range(W - 1, T, ratio):
        for c in range(hd):
            i = pick[c]
            pos = p - (W - 1) + i
            tag = (1000.0 + pos if i < 4 else pos) if ratio == 4 else pos
            assert out[p, c] == np.float32(tag + c / 256.0), (p, c, i)


def test_c4_first_group_masks_previous_group(oracle_mod):
    """seq_len == 4: there is no previous group; the window is positions 0..3 only
    and a NaN in the (never written) state must not reach the output."""
    o = oracle_mod
    hd = 128
    w = _one_request(4, hd, torch.float32, 4, seed=3)
    tok = wl.bits(w.kv_score)
    state = wl.bits(w.state).copy()
    out = o.compress_pool_prefill(4, hd, o.F32, o.F32, state, tok,
                                  np.zeros((8, hd), np.float32),
                                  o.plan_prefill(4, [0], [4], [4])[0])
    assert np.isfinite(out).all()
    tokz = tok.copy()
    tokz[:, 3 * hd:] = 0.0  # equal main scores -> mean of main kv of positions 0..3
    out = o.compress_history(4, hd, o.F32, o.F32, tokz, np.zeros((8, hd), np.float32))
    want = tokz[0:4, hd:2 * hd].astype(np.float64).mean(0)
    assert np.allclose(out[3], want, rtol=0, atol=1e-6)


@pytest.mark.parametrize("ratio,in_dt,out_dt", [(4, 0, 0), (4, 1, 1), (128, 1, 0), (128, 0, 1)])
def test_pool_matches_float64_torch_softmax(oracle_mod, ratio, in_dt, out_dt):
    o = oracle_mod
    hd = 128
    W = H.window(ratio)
    T = 2 * W + 4
    tdt = torch.bfloat16 if in_dt else torch.float32
    g = torch.Generator().manual_seed(5)
    width = wl.width_of(ratio, hd)
    tok = (torch.randn(T, width, generator=g) * 2).to(tdt)
    ape = (torch.randn(W, hd, generator=g) * 0.5).to(tdt)
    out = o.compress_history(ratio, hd, in_dt, out_dt, wl.bits(tok), wl.bits(ape))
    for p in range(T):
        if (p + 1) % ratio:
            continue
        kv_rows, sc_rows, idx = [], [], []
        for i in range(W):
            q = p - (W - 1) + i
            if q < 0:
                continue
            if ratio == 4:
                kv_rows.append(tok[q, (0 if i < 4 else hd):(0 if i < 4 else hd) + hd])
                sc_rows.append(tok[q, (2 * hd if i < 4 else 3 * hd):(2 * hd if i < 4 else 3 * hd) + hd])
            else:
                kv_rows.append(tok[q, :hd])
                sc_rows.append(tok[q, hd:])
            idx.append(i)
        kv = torch.stack(kv_rows).double()
        s = (torch.stack(sc_rows).float() + ape[idx].float()).double()   # fp32 score + bias
        want = (torch.softmax(s, dim=0) * kv).sum(0)
        if out_dt:
            want_bits = want.float().to(torch.bfloat16)  # two roundings: allow 1 ulp
            d = H.ulp_distance(out[p], wl.bits(want_bits))
        else:
            d = H.ulp_distance(out[p], want.float().numpy())
        assert d.max() <= 1, (p, d.max())


# ----------------------------------------------------------------------------- drivers
@pytest.mark.parametrize("ratio", [4, 128])
@pytest.mark.parametrize("seed", range(3))
def test_modes_equal_history(oracle_mod, ratio, seed):
    """One prefill, random chunked prefills and token-by-token decode over the same
    token streams give exactly the rows of the stateless whole-history definition.
    A wrong write set, buffer_len or page would read a NaN sentinel or a stale slot."""
    o = oracle_mod
    hd = 128
    rng = np.random.default_rng(seed)
    nreq = 5
    lens = [int(rng.integers(1, 3 * ratio + 30)) for _ in range(nreq)]
    rids = list(rng.permutation(8)[:nreq])
    in_dt, out_dt = (1, 0) if seed % 2 == 0 else (0, 1)
    tdt = torch.bfloat16 if in_dt else torch.float32
    g = torch.Generator().manual_seed(50 + seed)
    width = wl.width_of(ratio, hd)
    hist = [wl.bits((torch.randn(n, width, generator=g)).to(tdt)).copy() for n in lens]
    ape = wl.bits((torch.randn(H.window(ratio), hd, generator=g) * 0.1).to(tdt)).copy()
    want = [o.compress_history(ratio, hd, in_dt, out_dt, h, ape) for h in hist]
    backend = H.OracleBackend(o)
    for mode in ["oneshot", "chunked", "decode", "mixed"]:
        if mode == "oneshot":
            sched = [[("prefill", n)] for n in lens]
        elif mode == "chunked":
            sched = [H.split_schedule(n, rng, max(1, ratio + 5), 0.0) for n in lens]
        elif mode == "decode":
            sched = [[("decode", 1)] * n for n in lens]
        else:
            sched = [H.split_schedule(n, rng, max(2, ratio // 2 + 3), 0.5) for n in lens]
        state = wl.bits(wl.sentinel((8 * H.slots(ratio), width), tdt)).copy()
        got = H.run_schedule(backend, ratio, hd, in_dt, out_dt, hist, rids, sched, ape, state)
        for b in range(nreq):
            assert (got[b].view(np.uint32 if got[b].dtype == np.float32 else np.uint16)
                    == want[b].view(np.uint32 if want[b].dtype == np.float32 else np.uint16)).all(), (mode, b)


def test_decode_nonboundary_rows_are_zero(oracle_mod):
    o = oracle_mod
    for ratio in (4, 128):
        w = wl.random_decode(ratio, 128, torch.bfloat16, torch.float32, [1, 2, 3, 5, 4, 8, 129, 256], seed=2,
                             num_requests_state=8)
        plan = o.plan_decode(ratio, w.rid.numpy(), w.seq_lens.numpy())
        state = wl.bits(w.state).copy()
        out = o.compress_decode(ratio, 128, 1, 0, state, wl.bits(w.kv_score), wl.bits(w.ape), plan)
        for b, sl in enumerate(w.seq_lens.tolist()):
            if sl % ratio:
                assert (out[b].view(np.uint32) == 0).all()
            else:
                assert np.abs(out[b]).max() > 0


def test_prefill_token_layout_zero_rows_and_compact_order(oracle_mod):
    o = oracle_mod
    w = wl.random_prefill(4, 128, torch.bfloat16, torch.float32, wl.TOKEN, [5, 0, 2], [4, 3, 6], seed=4,
                          num_requests_state=4, rid=[1, 0, 2])
    pc, pw, (nc, nw), _ = o.plan_prefill(4, w.rid, w.seq_lens, w.extend_lens)
    st = wl.bits(w.state)
    tok = o.compress_pool_prefill(4, 128, 1, 0, st, wl.bits(w.kv_score), wl.bits(w.ape), pc, nc,
                                  out_layout=o.OUT_TOKEN)
    cmp_ = o.compress_pool_prefill(4, 128, 1, 0, st, wl.bits(w.kv_score), wl.bits(w.ape), pc, nc,
                                   out_layout=o.OUT_COMPACT)
    rag = H.plan_c_fields(pc)["ragged_id"]
    assert (tok[rag] == cmp_).all()
    others = np.setdiff1d(np.arange(tok.shape[0]), rag)
    assert (tok[others].view(np.uint32) == 0).all()
