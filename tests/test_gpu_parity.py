"""GPU parity: libckv (through its C ABI) against the CPU oracle.

Bar: plans, write locations and state buffers bit-exact; fp32 outputs within
2e-6 * max|kv| of the window per channel; bf16 outputs within 1 ulp.  Sizes
span several tiles / grid-stride rounds and ragged tails; the edge cases
(empty batch, maximum batch, first C4 group, capacity overflow, bad lengths,
out-of-range plan records) are covered here too.
"""
import zlib

import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H

pytestmark = pytest.mark.gpu

DT = {"f32": 0, "bf16": 1}


@pytest.fixture(scope="module")
def env(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_attention_compressplan_gb300 import build as B
    from compressed_kv_attention_compressplan_gb300 import ckv

    B.build()
    ckv.load_library()
    return oracle_mod, ckv, torch.device("cuda")


def _dev_i64(x, dev):
    return torch.as_tensor(np.asarray(x), dtype=torch.int64).to(dev)


# ----------------------------------------------------------------------------- plans
@pytest.mark.parametrize("ratio", [4, 128])
@pytest.mark.parametrize("B", [777, 1024, 1500, 5000])
def test_plan_decode_bit_exact(env, ratio, B):
    """Records bit-exact against the oracle, with and without the boundary-row
    list; the list (one CTA, chunks of 1024 or 4096 rows) equals the rows the
    oracle's records mark as emitting, in row order."""
    o, ckv, dev = env
    rng = np.random.default_rng(ratio + B)
    rid = rng.permutation(8192)[:B]
    sl = rng.integers(1, 70000, B)
    sl[:40] = np.arange(1, 41)
    sl[40:80] = ratio * rng.integers(1, 300, 40)
    sl[-3:] = ratio  # boundary rows at the tail of the last chunk
    want = o.plan_decode(ratio, rid, sl)
    got = ckv.plan_decode(ratio, _dev_i64(rid, dev), _dev_i64(sl, dev)).cpu().numpy()
    assert (got == want).all()
    order = ckv.new_decode_order(B, dev)
    order.fill_(0xAB)
    got = ckv.plan_decode(ratio, _dev_i64(rid, dev), _dev_i64(sl, dev), order=order).cpu().numpy()
    assert (got == want).all()
    assert (H.decode_order_entries(order) == H.expected_decode_order(want, ratio)).all()


def test_plan_decode_order_skips_bad_rows_and_empty_batches(env):
    o, ckv, dev = env
    status = ckv.new_status(dev)
    rid, sl = [0, -1, 2, 3], [128, 128, 0, 256]
    order = ckv.new_decode_order(4, dev)
    pd = ckv.plan_decode(128, _dev_i64(rid, dev), _dev_i64(sl, dev), status=status, order=order).cpu().numpy()
    torch.cuda.synchronize()
    assert int(status[0]) & ckv.STATUS_BAD_LENGTH
    ent = H.decode_order_entries(order)
    assert ent[:, 0].tolist() == [2, 0, 3] and ent[1:, 1].tolist() == [0, 3]
    assert (ent == H.expected_decode_order(pd, 128)).all()
    empty = ckv.new_decode_order(0, dev)
    empty.fill_(0xAB)
    ckv.plan_decode(128, _dev_i64([], dev), _dev_i64([], dev), order=empty)
    assert H.decode_order_entries(empty).tolist() == [[0, 0]]


def _prefill_case(name, ratio, rng):
    if name == "random":
        B = 37
        pl = rng.integers(0, 3 * ratio + 50, B)
        el = rng.integers(1, 5 * ratio + 40, B)
    elif name == "mtp_uniform":
        B = 1024
        pl = rng.integers(0, 70000, B)
        el = np.full(B, 4)
    elif name == "decode_like":
        B = 1000
        pl = rng.integers(0, 5000, B)
        el = np.ones(B, np.int64)
    elif name in ("uniform_32", "uniform_33"):  # the largest uniform extend of the per-request path, and one past it
        B = 700
        pl = rng.integers(0, 9000, B)
        el = np.full(B, int(name[-2:]))
    elif name == "one_long":
        B = 1
        pl = np.array([rng.integers(0, 1000)])
        el = np.array([20000 + int(rng.integers(0, 999))])
    elif name == "max_batch_mixed":
        B = 1024
        pl = rng.integers(0, 65536, B)
        el = np.where(rng.random(B) < 0.875, 4, rng.integers(128, 2000, B))
    elif name == "max_tokens":  # the largest step the 24-bit ragged ids allow: 2^24 - 1 tokens, 1024 requests
        B = 1024
        pl = rng.integers(0, 65536, B)
        total = (1 << 24) - 1
        el = np.full(B, total // B)
        el[: total - int(el.sum())] += 1
        assert int(el.sum()) == total
    else:
        raise ValueError(name)
    rid = rng.permutation(max(B, 2048))[:B]
    return rid, pl + el, el


@pytest.mark.parametrize("ratio", [4, 128])
@pytest.mark.parametrize("case", ["random", "mtp_uniform", "decode_like", "uniform_32", "uniform_33", "one_long",
                                  "max_batch_mixed", "max_tokens"])
@pytest.mark.parametrize("pad", [False, True])
def test_plan_prefill_bit_exact(env, ratio, case, pad):
    o, ckv, dev = env
    rng = np.random.default_rng(zlib.crc32(f"{ratio}-{case}".encode()))
    rid, sl, el = _prefill_case(case, ratio, rng)
    nq = int(el.sum())
    cap_c = ckv.capacity_compress(ratio, len(rid), nq)
    cap_w = ckv.capacity_write(ratio, len(rid), nq)
    status = ckv.new_status(dev)
    pc, pw, counts = ckv.plan_prefill(ratio, _dev_i64(rid, dev), _dev_i64(sl, dev), _dev_i64(el, dev), nq, cap_c,
                                      cap_w, pad_invalid=pad, status=status)
    torch.cuda.synchronize()
    wc, ww, (nc, nw), rc = o.plan_prefill(ratio, rid, sl, el, nq, cap_c, cap_w, pad_invalid=pad)
    assert rc == 0 and int(status[0]) == 0
    cnt = counts.cpu().numpy()
    assert (cnt[0], cnt[1]) == (nc, nw)
    assert (cnt[2], cnt[3]) == (el.min(), el.max())
    n_c = cap_c if pad else nc
    n_w = cap_w if pad else nw
    assert (pc[:n_c].cpu().numpy() == wc[:n_c]).all()
    assert (pw[:n_w].cpu().numpy() == ww[:n_w]).all()


def test_plan_prefill_empty_and_errors(env):
    o, ckv, dev = env
    status = ckv.new_status(dev)
    e = torch.empty(0, dtype=torch.int64, device=dev)
    pc, pw, counts = ckv.plan_prefill(4, e, e, e, 0, 4, 4, pad_invalid=True, status=status)
    torch.cuda.synchronize()
    assert counts[:2].tolist() == [0, 0] and int(status[0]) == 0
    assert (pc.cpu().numpy() == 0xFF).all() and (pw.cpu().numpy() == 0xFF).all()
    # capacity overflow: true counts reported, CAPACITY set, no record past the buffer
    rid, sl, el = [0, 1], [9, 12], [9, 4]
    pc, pw, counts = ckv.plan_prefill(4, _dev_i64(rid, dev), _dev_i64(sl, dev), _dev_i64(el, dev), 13, 2, 3,
                                      status=status)
    torch.cuda.synchronize()
    assert counts[:2].tolist() == [3, 9] and int(status[0]) & ckv.STATUS_CAPACITY
    wc, ww, _, _ = o.plan_prefill(4, rid, sl, el, 13, 2, 3, check=False)
    assert (pc.cpu().numpy() == wc).all() and (pw.cpu().numpy() == ww).all()
    # the same with equal extends (the per-request emission of uniform batches), padded
    rid, sl, el = [0, 1, 2], [8, 12, 7], [4, 4, 4]
    status.zero_()
    pc, pw, counts = ckv.plan_prefill(4, _dev_i64(rid, dev), _dev_i64(sl, dev), _dev_i64(el, dev), 12, 2, 5,
                                      pad_invalid=True, status=status)
    torch.cuda.synchronize()
    assert counts[:2].tolist() == [3, 12] and int(status[0]) & ckv.STATUS_CAPACITY
    wc, ww, _, _ = o.plan_prefill(4, rid, sl, el, 12, 2, 5, pad_invalid=True, check=False)
    assert (pc.cpu().numpy() == wc).all() and (pw.cpu().numpy() == ww).all()
    # bad lengths and a wrong token total: flagged, nothing emitted, no fault
    for sl_, el_, nq, bit in [([9, 5], [9, 6], 15, ckv.STATUS_BAD_LENGTH), ([9, 5], [9, 0], 9, ckv.STATUS_BAD_LENGTH),
                              ([9, 5], [9, 5], 13, ckv.STATUS_BAD_TOTAL)]:
        status.zero_()
        pc, pw, counts = ckv.plan_prefill(128, _dev_i64([0, 1], dev), _dev_i64(sl_, dev), _dev_i64(el_, dev), nq, 8,
                                          8, pad_invalid=True, status=status)
        torch.cuda.synchronize()
        assert int(status[0]) & bit
    # decode plan: a bad row is invalid, the rest are fine
    status.zero_()
    pd = ckv.plan_decode(4, _dev_i64([0, -1, 2], dev), _dev_i64([5, 5, 0], dev), status=status).cpu().numpy()
    torch.cuda.synchronize()
    assert int(status[0]) & ckv.STATUS_BAD_LENGTH
    assert (pd[1] == 0xFF).all() and (pd[2] == 0xFF).all()
    assert (pd[0] == o.plan_decode(4, [0], [5])[0]).all()


# ----------------------------------------------------------------------------- prefill pool + write
def _run_prefill_parity(env, ratio, hd, in_dt, out_dt, layout, pl, el, seed, state_fill="normal", outliers=0.0):
    o, ckv, dev = env
    w = wl.random_prefill(ratio, hd, H.torch_dtype(in_dt), H.torch_dtype(out_dt),
                          wl.TOKEN if layout == 0 else wl.COMPACT, pl, el, seed,
                          num_requests_state=len(pl) + 3, state_fill=state_fill, outlier_frac=outliers)
    nq = w.num_q_tokens
    state_d = w.state.to(dev)
    status = ckv.new_status(dev)
    lens = (w.rid.to(dev), w.seq_lens.to(dev), w.extend_lens.to(dev))
    pc, pw, counts = ckv.plan_prefill(ratio, *lens, nq, status=status)
    # about half of the cases also hand the pool the planner's inputs as prefetch hints
    hinted = zlib.crc32(f"{ratio},{hd},{in_dt},{out_dt},{layout},{seed}".encode()) & 1
    out = ckv.compress_prefill(ratio, hd, state_d, w.kv_score.to(dev), w.ape.to(dev), pc, pw, counts, layout,
                               H.torch_dtype(out_dt), status=status, hints=lens if hinted else None)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    st = wl.bits(w.state).copy()
    inp = wl.bits(w.kv_score)
    wc, ww, (nc, nw), _ = o.plan_prefill(ratio, w.rid, w.seq_lens, w.extend_lens)
    want = o.compress_pool_prefill(ratio, hd, in_dt, out_dt, st, inp, wl.bits(w.ape), wc, nc, nq, layout)
    f = H.plan_c_fields(wc)
    kvmax = H.window_kv_absmax(ratio, hd, st, inp, f["seq_len"], f["ragged_id"], f["buffer_len"],
                               f["read_page_0"], f["read_page_1"])
    got = H.np_bits(out)
    if layout == 0:
        rows = f["ragged_id"]
        H.assert_pool_close(got[rows], want[rows], out_dt, kvmax, "compress rows")
        others = np.setdiff1d(np.arange(nq), rows)
        assert (got[others].view(np.uint16 if out_dt else np.uint32) == 0).all(), "non-compress rows not zero"
    else:
        H.assert_pool_close(got[:nc], want, out_dt, kvmax, "compact rows")
    o.compress_write(ratio, hd, in_dt, st, inp, ww, nw)
    assert (H.np_bits(state_d).view(np.uint8) == st.view(np.uint8)).all(), "state after write"


# head_dim 640 and 1024 give the C4 pool its other widths (128-channel blocks,
# five per quarter; 1 KB-wide fp32 rows).  Steps this small take the direct
# kernel, except fp32 at 640 and 1024 (one record fills a stage); each launch
# shape of the pool has its own cases in test_gpu_pool_shapes.py.
@pytest.mark.parametrize("hd", [128, 384, 512, 640, 1024])
@pytest.mark.parametrize("dts", [("bf16", "f32"), ("bf16", "bf16"), ("f32", "f32"), ("f32", "bf16")])
@pytest.mark.parametrize("layout", [0, 1])
def test_c4_prefill_parity(env, hd, dts, layout):
    rng = np.random.default_rng(hd + 7 * layout)
    pl = list(rng.integers(0, 40, 9)) + [0, 2, 5, 0]
    el = list(rng.integers(1, 70, 9)) + [4, 2, 4, 1]
    _run_prefill_parity(env, 4, hd, DT[dts[0]], DT[dts[1]], layout, pl, el, seed=hd + layout)


@pytest.mark.parametrize("hd", [128, 384, 512, 1024])
@pytest.mark.parametrize("dts", [("bf16", "f32"), ("bf16", "bf16"), ("f32", "f32"), ("f32", "bf16")])
@pytest.mark.parametrize("layout", [0, 1])
def test_c128_prefill_parity(env, hd, dts, layout):
    rng = np.random.default_rng(hd + 11 * layout)
    pl = list(rng.integers(0, 400, 5)) + [0, 127, 1]
    el = list(rng.integers(1, 420, 5)) + [128, 1, 300]
    _run_prefill_parity(env, 128, hd, DT[dts[0]], DT[dts[1]], layout, pl, el, seed=hd + layout, outliers=0.01)


def test_c4_prefill_first_group_ignores_nan_state(env):
    # sentinel-filled (NaN) ring: the first group of each request must not read it
    _run_prefill_parity(env, 4, 128, 0, 0, 0, [0, 0, 1, 2], [4, 64, 3, 9], seed=3, state_fill="sentinel")


# ----------------------------------------------------------------------------- decode
def decode_through(ckv, ordered, ratio, hd, state_d, w, out_dtype, status, dev):
    """plan_decode -> compress_decode, with the boundary-row list (decode_step) or without it."""
    if ordered:
        return ckv.decode_step(ratio, hd, state_d, w.kv_score.to(dev), w.ape.to(dev), w.rid.to(dev),
                               w.seq_lens.to(dev), out_dtype, status=status)
    pd = ckv.plan_decode(ratio, w.rid.to(dev), w.seq_lens.to(dev), status=status)
    out = ckv.compress_decode(ratio, hd, state_d, w.kv_score.to(dev), w.ape.to(dev), pd, out_dtype, status=status)
    return out, pd


@pytest.mark.parametrize("ratio", [4, 128])
@pytest.mark.parametrize("hd", [128, 512])
@pytest.mark.parametrize("dts", [("bf16", "f32"), ("bf16", "bf16"), ("f32", "f32")])
@pytest.mark.parametrize("ordered", [True, False])
def test_decode_parity(env, ratio, hd, dts, ordered):
    o, ckv, dev = env
    in_dt, out_dt = DT[dts[0]], DT[dts[1]]
    rng = np.random.default_rng(ratio + hd)
    B = 203
    sl = rng.integers(1, 5000, B)
    sl[:60] = ratio * rng.integers(1, 30, 60)
    sl[60:64] = [1, 4, 8, ratio]
    w = wl.random_decode(ratio, hd, H.torch_dtype(in_dt), H.torch_dtype(out_dt), sl, seed=ratio + hd,
                         num_requests_state=256)
    state_d = w.state.to(dev)
    status = ckv.new_status(dev)
    out, pd = decode_through(ckv, ordered, ratio, hd, state_d, w, H.torch_dtype(out_dt), status, dev)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    st0 = wl.bits(w.state).copy()
    st = st0.copy()
    wpd = o.plan_decode(ratio, w.rid, w.seq_lens)
    assert (pd.cpu().numpy() == wpd).all()
    inp = wl.bits(w.kv_score)
    want = o.compress_decode(ratio, hd, in_dt, out_dt, st, inp, wl.bits(w.ape), wpd)
    got = H.np_bits(out)
    f = H.plan_d_fields(wpd)
    bnd = np.nonzero(f["seq_len"] % ratio == 0)[0]
    W = H.window(ratio)
    kvmax = H.window_kv_absmax(ratio, hd, st0, inp, f["seq_len"][bnd], bnd, np.full(len(bnd), W - 1),
                               f["read_page_0"][bnd], f["read_page_1"][bnd])
    H.assert_pool_close(got[bnd], want[bnd], out_dt, kvmax, "decode boundary rows")
    nb = np.setdiff1d(np.arange(B), bnd)
    assert (got[nb].view(np.uint16 if out_dt else np.uint32) == 0).all()
    assert (H.np_bits(state_d).view(np.uint8) == st.view(np.uint8)).all(), "state after decode"


def test_out_of_range_records_are_flagged_not_faulted(env):
    """Plan records that point outside the state or the input are skipped by the
    kernels' own bounds checks and reported in the status word."""
    o, ckv, dev = env
    for ratio in (4, 128):
        hd = 128
        w = wl.random_decode(ratio, hd, torch.bfloat16, torch.float32, [ratio, 3], seed=1, num_requests_state=2)
        status = ckv.new_status(dev)
        bad = torch.tensor([[ratio, 10 ** 6, 10 ** 6, 10 ** 6], [3, 1, 0, 0]], dtype=torch.int32)
        pd = bad.view(torch.uint8).reshape(2, 16).to(dev)
        out = ckv.compress_decode(ratio, hd, w.state.to(dev), w.kv_score.to(dev), w.ape.to(dev), pd,
                                  status=status)
        torch.cuda.synchronize()
        assert int(status[0]) & ckv.STATUS_BAD_INDEX
        assert (out[0] == 0).all()
        # prefill: a compress record whose page is outside the state, one whose
        # window reaches before input row 0
        W = H.window(ratio)
        recs = torch.tensor([[2 * ratio, (W - 1) | (3 << 24), 10 ** 6, 10 ** 6],
                             [ratio, 2 | (0 << 24), 0, 0]], dtype=torch.int32)
        pc = recs.view(torch.uint8).reshape(2, 16).to(dev)
        kv = torch.randn(W + 2, wl.width_of(ratio, hd)).to(torch.bfloat16).to(dev)
        status.zero_()
        ckv.compress_pool_prefill(ratio, hd, w.state.to(dev), kv, w.ape.to(dev), pc, None, ckv.OUT_COMPACT,
                                  status=status)
        torch.cuda.synchronize()
        assert int(status[0]) & ckv.STATUS_BAD_INDEX
        # write records outside the state / input
        pw = torch.tensor([[0, 10 ** 7], [10 ** 6, 0]], dtype=torch.int32).view(torch.uint8).reshape(2, 8).to(dev)
        status.zero_()
        ckv.compress_write(ratio, hd, w.state.to(dev), kv, pw, None, status=status)
        torch.cuda.synchronize()
        assert int(status[0]) & ckv.STATUS_BAD_INDEX


@pytest.mark.parametrize("ratio", [4, 128])
@pytest.mark.parametrize("padded", [False, True])
def test_prefill_step_without_compress_records(env, ratio, padded):
    """A step in which no request reaches a multiple of the ratio: no compress
    record (padded plans: all records invalid).  Token layout: every output row
    is +0.0; compact layout: the output is left as it was; the state write
    still happens, bit for bit."""
    o, ckv, dev = env
    hd = 256
    pl = [1, 130, 260, 5] if ratio == 128 else [1, 5, 9, 13]
    el = [2, 3, 1, 2] if ratio == 128 else [2, 2, 1, 2]
    w = wl.random_prefill(ratio, hd, torch.bfloat16, torch.float32, wl.TOKEN, pl, el, seed=9 + ratio,
                          num_requests_state=6)
    nq = w.num_q_tokens
    lens = (w.rid.to(dev), w.seq_lens.to(dev), w.extend_lens.to(dev))
    cap_c = nq if padded else ckv.capacity_compress(ratio, 4, nq)
    cap_w = nq if padded else ckv.capacity_write(ratio, 4, nq)
    for layout in (ckv.OUT_TOKEN, ckv.OUT_COMPACT):
        status = ckv.new_status(dev)
        state_d = w.state.to(dev)
        pc, pw, counts = ckv.plan_prefill(ratio, *lens, nq, cap_c, cap_w, pad_invalid=padded, status=status)
        rows = nq if layout == ckv.OUT_TOKEN else cap_c
        out = torch.full((rows, hd), float("nan"), dtype=torch.float32, device=dev)
        ckv.compress_prefill(ratio, hd, state_d, w.kv_score.to(dev), w.ape.to(dev), pc, pw, counts, layout,
                             torch.float32, out=out, status=status, hints=lens)
        torch.cuda.synchronize()
        assert int(status[0]) == 0 and int(counts[0]) == 0
        if layout == ckv.OUT_TOKEN:
            assert (H.np_bits(out).view(np.uint32) == 0).all()
        else:
            assert torch.isnan(out).all()
        st = wl.bits(w.state).copy()
        _, ww, (nc, nw), _ = o.plan_prefill(ratio, w.rid, w.seq_lens, w.extend_lens)
        assert nc == 0
        o.compress_write(ratio, hd, 1, st, wl.bits(w.kv_score), ww, nw)
        assert (H.np_bits(state_d).view(np.uint8) == st.view(np.uint8)).all()


@pytest.mark.parametrize("ratio", [4, 128])
def test_decode_prefetch_hints_only_steer_prefetches(env, ratio):
    """The rid / seq_lens hints are read before the decode's dependency wait,
    so they may be stale: hints that name other rows, other pages, pages past
    the state and negative ids leave every output and state byte as without
    hints (and as the oracle's)."""
    o, ckv, dev = env
    hd = 512
    rng = np.random.default_rng(ratio + 5)
    B = 300
    sl = rng.integers(1, 9000, B)
    sl[:90] = ratio * rng.integers(1, 60, 90)
    w = wl.random_decode(ratio, hd, torch.bfloat16, torch.float32, sl, seed=ratio + 5, num_requests_state=320)
    order = ckv.new_decode_order(B, dev)
    pd = ckv.plan_decode(ratio, w.rid.to(dev), w.seq_lens.to(dev), order=order)
    outs = {}
    for name, hints in [("none", None),
                        ("right", (w.rid, w.seq_lens)),
                        ("stale", (torch.from_numpy(rng.permutation(320)[:B]).to(torch.int64),
                                   torch.from_numpy(ratio * rng.integers(1, 99, B)).to(torch.int64))),
                        ("outside", (torch.full((B,), 10 ** 9, dtype=torch.int64), torch.full((B,), 128, dtype=torch.int64))),
                        ("negative", (torch.full((B,), -5, dtype=torch.int64), torch.full((B,), -128, dtype=torch.int64)))]:
        state_d = w.state.to(dev)
        status = ckv.new_status(dev)
        kw = {} if hints is None else {"rid_hint": hints[0].to(dev), "seq_lens_hint": hints[1].to(dev)}
        out = ckv.compress_decode(ratio, hd, state_d, w.kv_score.to(dev), w.ape.to(dev), pd, torch.float32,
                                  status=status, order=order, **kw)
        torch.cuda.synchronize()
        assert int(status[0]) == 0, name
        outs[name] = (H.np_bits(out).copy(), H.np_bits(state_d).copy())
    for name in ("right", "stale", "outside", "negative"):
        assert (outs[name][0].view(np.uint32) == outs["none"][0].view(np.uint32)).all(), name
        assert (outs[name][1].view(np.uint8) == outs["none"][1].view(np.uint8)).all(), name
    st = wl.bits(w.state).copy()
    want = o.compress_decode(ratio, hd, 1, 0, st, wl.bits(w.kv_score), wl.bits(w.ape), o.plan_decode(ratio, w.rid, w.seq_lens))
    f = H.plan_d_fields(pd.cpu().numpy())
    bnd = np.nonzero(f["seq_len"] % ratio == 0)[0]
    kvmax = H.window_kv_absmax(ratio, hd, wl.bits(w.state), wl.bits(w.kv_score), f["seq_len"][bnd], bnd,
                               np.full(len(bnd), H.window(ratio) - 1), f["read_page_0"][bnd], f["read_page_1"][bnd])
    H.assert_pool_close(outs["none"][0][bnd], want[bnd], 0, kvmax, "decode with hints")
    assert (outs["none"][1].view(np.uint8) == st.view(np.uint8)).all()


@pytest.mark.parametrize("ratio", [4, 128])
def test_prefill_prefetch_hints_only_steer_prefetches(env, ratio):
    """The prefill pool reads the planner's rid / seq_lens / extend_lens before
    its dependency wait, only to prefetch windows: hints that name other
    requests, rows past the state, negative ids or lengths, or extends longer
    than the sequence leave every output byte as without hints (and within the
    bar of the oracle's)."""
    o, ckv, dev = env
    B = 300
    w = (wl.c4_prefill_mtp if ratio == 4 else wl.c128_prefill_mtp)(ratio + 11, batch=B)
    hd, nq = w.head_dim, w.num_q_tokens
    ci, co = (1 if w.in_dtype == torch.bfloat16 else 0), (1 if w.out_dtype == torch.bfloat16 else 0)
    layout = ckv.OUT_TOKEN if w.out_layout == wl.TOKEN else ckv.OUT_COMPACT
    pc, pw, counts = ckv.plan_prefill(ratio, w.rid.to(dev), w.seq_lens.to(dev), w.extend_lens.to(dev), nq)
    rng = np.random.default_rng(ratio)
    i64 = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.int64)
    cases = [("none", None),
             ("right", (w.rid, w.seq_lens, w.extend_lens)),
             ("stale", (i64(rng.permutation(B)), i64(rng.integers(1, 70000, B)), i64(rng.integers(1, 300, B)))),
             ("outside", (i64(np.full(B, 10 ** 12)), w.seq_lens, w.extend_lens)),
             ("negative", (i64(np.full(B, -3)), i64(np.full(B, -130)), i64(np.full(B, -4)))),
             ("long_extend", (w.rid, w.seq_lens, w.seq_lens + 5))]
    outs = {}
    for name, hints in cases:
        status = ckv.new_status(dev)
        hk = None if hints is None else tuple(t.to(dev) for t in hints)
        out = ckv.compress_pool_prefill(ratio, hd, w.state.to(dev), w.kv_score.to(dev), w.ape.to(dev), pc, counts,
                                        layout, w.out_dtype, status=status, hints=hk)
        torch.cuda.synchronize()
        assert int(status[0]) == 0, name
        outs[name] = H.np_bits(out).copy()
    wc, _, (nc, _), _ = o.plan_prefill(ratio, w.rid, w.seq_lens, w.extend_lens)
    written = slice(None) if layout == ckv.OUT_TOKEN else slice(0, nc)  # compact rows past the count stay as they were
    for name, _ in cases[1:]:
        assert (outs[name][written].view(np.uint8) == outs["none"][written].view(np.uint8)).all(), name
    st = wl.bits(w.state)
    inp = wl.bits(w.kv_score)
    want = o.compress_pool_prefill(ratio, hd, ci, co, st.copy(), inp, wl.bits(w.ape), np.ascontiguousarray(wc), nc,
                                   nq, o.OUT_COMPACT)
    f = H.plan_c_fields(wc)
    kvmax = H.window_kv_absmax(ratio, hd, st, inp, f["seq_len"], f["ragged_id"], f["buffer_len"], f["read_page_0"],
                               f["read_page_1"])
    rows = f["ragged_id"] if layout == ckv.OUT_TOKEN else np.arange(nc)
    H.assert_pool_close(outs["none"][rows], want, co, kvmax, "prefill pool with hints")


@pytest.mark.parametrize("B", [3000, 28000])
def test_c128_decode_large_batch_through_the_list(env, B):
    """Large batches through the boundary-row list and the prefetch hints: at
    28000 rows each persistent CTA owns ~370 list entries (more than its 352
    threads, so its prologue takes two passes) and ~185 rows without a window;
    every output row and state byte is compared with the oracle."""
    o, ckv, dev = env
    hd = 128
    rng = np.random.default_rng(B)
    sl = rng.integers(1, 4000, B)
    sl[rng.permutation(B)[: B // 4]] = 128 * rng.integers(1, 30, B // 4)
    w = wl.random_decode(128, hd, torch.bfloat16, torch.float32, sl, seed=B, num_requests_state=B + 3)
    state_d = w.state.to(dev)
    status = ckv.new_status(dev)
    out, pd = ckv.decode_step(128, hd, state_d, w.kv_score.to(dev), w.ape.to(dev), w.rid.to(dev),
                              w.seq_lens.to(dev), torch.float32, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    st0 = wl.bits(w.state).copy()
    st = st0.copy()
    wpd = o.plan_decode(128, w.rid, w.seq_lens)
    assert (pd.cpu().numpy() == wpd).all()
    want = o.compress_decode(128, hd, 1, 0, st, wl.bits(w.kv_score), wl.bits(w.ape), wpd)
    got = H.np_bits(out)
    f = H.plan_d_fields(wpd)
    bnd = np.nonzero(f["seq_len"] % 128 == 0)[0]
    kvmax = H.window_kv_absmax(128, hd, st0, wl.bits(w.kv_score), f["seq_len"][bnd], bnd, np.full(len(bnd), 127),
                               f["read_page_0"][bnd], f["read_page_1"][bnd])
    H.assert_pool_close(got[bnd], want[bnd], 0, kvmax, "large-batch decode boundary rows")
    nb = np.setdiff1d(np.arange(B), bnd)
    assert (got[nb].view(np.uint32) == 0).all()
    assert (H.np_bits(state_d).view(np.uint8) == st.view(np.uint8)).all()


def test_bad_order_entries_are_flagged_not_faulted(env):
    """A boundary-row list that does not match the plan (a row past the batch, a
    page outside the state, a count larger than the batch) is bounds-checked by
    the C128 decode: those entries are skipped and reported, nothing faults, and
    the rows the list does name correctly are pooled as usual."""
    o, ckv, dev = env
    hd = 128
    w = wl.random_decode(128, hd, torch.bfloat16, torch.float32, [128, 256, 384, 5], seed=2, num_requests_state=4)
    pd = ckv.plan_decode(128, w.rid.to(dev), w.seq_lens.to(dev))
    good = ckv.new_decode_order(4, dev)
    ckv.plan_decode(128, w.rid.to(dev), w.seq_lens.to(dev), order=good)
    want = ckv.compress_decode(128, hd, w.state.to(dev), w.kv_score.to(dev), w.ape.to(dev), pd, order=good)
    # count past the batch; row 0 and row 1 named correctly; a row past the batch; row 2 with a page
    # outside the state (so row 2 is not pooled: its output is unspecified)
    ent = torch.tensor([[100, 0], [0, int(w.rid[0])], [9, 0], [2, 10 ** 6], [1, int(w.rid[1])]], dtype=torch.int32)
    bad = ent.view(torch.uint8).reshape(5, 8).to(dev)
    status = ckv.new_status(dev)
    state_d = w.state.to(dev)
    out = ckv.compress_decode(128, hd, state_d, w.kv_score.to(dev), w.ape.to(dev), pd, status=status, order=bad)
    torch.cuda.synchronize()
    assert int(status[0]) & ckv.STATUS_BAD_INDEX
    assert torch.equal(out[0], want[0]) and torch.equal(out[1], want[1])
    assert (out[3] == 0).all()               # not a boundary row: zeroed by its own record


# ----------------------------------------------------------------------------- invariants on the GPU
@pytest.mark.parametrize("ratio", [4, 128])
def test_modes_bitwise_identical_on_gpu(env, ratio):
    """One prefill, chunked prefills, token-by-token decode and a random mix of
    both produce bit-identical rows on the GPU, and match the oracle's
    whole-history definition within the parity bar."""
    o, ckv, dev = env
    hd = 512 if ratio == 4 else 256
    rng = np.random.default_rng(ratio)
    nreq = 6
    lens = [int(rng.integers(1, 3 * ratio + 40)) for _ in range(nreq)]
    rids = list(rng.permutation(8)[:nreq])
    g = torch.Generator().manual_seed(ratio)
    width = wl.width_of(ratio, hd)
    hist = [wl.bits(torch.randn(n, width, generator=g).to(torch.bfloat16)).copy() for n in lens]
    ape = wl.bits((torch.randn(H.window(ratio), hd, generator=g) * 0.1).to(torch.bfloat16)).copy()
    want = [o.compress_history(ratio, hd, 1, 0, h, ape) for h in hist]
    backend = H.GpuBackend(dev)
    results = {}
    for mode in ["oneshot", "chunked", "decode", "mixed"]:
        if mode == "oneshot":
            sched = [[("prefill", n)] for n in lens]
        elif mode == "chunked":
            sched = [H.split_schedule(n, rng, ratio + 5, 0.0) for n in lens]
        elif mode == "decode":
            sched = [[("decode", 1)] * n for n in lens]
        else:
            sched = [H.split_schedule(n, rng, ratio // 2 + 3, 0.5) for n in lens]
        state = wl.sentinel((8 * H.slots(ratio), width), torch.bfloat16).to(dev)
        results[mode] = H.run_schedule(backend, ratio, hd, 1, 0, hist, rids, sched, ape, state)
        assert int(backend.status[0]) == 0
    for b in range(nreq):
        ref = results["oneshot"][b]
        for mode in ["chunked", "decode", "mixed"]:
            assert (results[mode][b].view(np.uint32) == ref.view(np.uint32)).all(), (mode, b)
        emit = [p for p in range(lens[b]) if (p + 1) % ratio == 0]
        if emit:
            seq = np.array(emit) + 1
            tok = hist[b]
            # the window of a whole-history row: all from the token history
            kvmax = H.window_kv_absmax(ratio, hd, tok, tok, seq, np.array(emit),
                                       np.zeros(len(emit), np.int64), np.zeros(len(emit)), np.zeros(len(emit)))
            H.assert_pool_close(ref[emit], want[b][emit], 0, kvmax, f"history b={b}")


@pytest.mark.parametrize("ratio", [4, 128])
def test_closed_forms_on_gpu(env, ratio):
    """Equal scores + zero ape -> the exact window mean, bit for bit (the score
    0.5 is a power of two, so max*log2(e) is exact and every weight is exactly
    1); a dominant ape entry -> that entry's kv (within the parity bar)."""
    o, ckv, dev = env
    hd = 128
    W = H.window(ratio)
    T = 3 * ratio + 8
    width = wl.width_of(ratio, hd)
    rng = np.random.default_rng(3)
    ncol = 2 * hd if ratio == 4 else hd
    tok = np.zeros((T, width), np.float32)
    tok[:, :ncol] = rng.integers(-50, 51, (T, ncol))
    tok[:, ncol:] = 0.5
    ape0 = np.zeros((W, hd), np.float32)
    backend = H.GpuBackend(dev)
    state = wl.sentinel((H.slots(ratio), width), torch.float32).to(dev)
    got = H.run_schedule(backend, ratio, hd, 0, 0, [tok], [0], [[("prefill", T)]], ape0, state)[0]
    want = o.compress_history(ratio, hd, 0, 0, tok, ape0)
    assert (got.view(np.uint32) == want.view(np.uint32)).all()
    q = np.arange(T, dtype=np.float32)[:, None]
    ch = np.arange(hd, dtype=np.float32)[None, :] / 256.0
    tok[:, :hd] = (1000.0 + q + ch) if ratio == 4 else (1.0 + q + ch)
    if ratio == 4:
        tok[:, hd:2 * hd] = 1.0 + q + ch
    pick = (np.arange(hd) * 5 + 1) % W
    ape = np.zeros((W, hd), np.float32)
    ape[pick, np.arange(hd)] = 60.0
    state = wl.sentinel((H.slots(ratio), width), torch.float32).to(dev)
    got = H.run_schedule(backend, ratio, hd, 0, 0, [tok], [0], [[("prefill", T)]], ape, state)[0]
    want = o.compress_history(ratio, hd, 0, 0, tok, ape)
    for p in range(W - 1, T, ratio):
        i = pick
        pos = p - (W - 1) + i
        tag = np.where(i < 4, 1000.0 + pos, 1.0 + pos) if ratio == 4 else 1.0 + pos
        tag = (tag + np.arange(hd) / 256.0).astype(np.float32)
        assert (want[p] == tag).all()
        assert np.abs(got[p] - tag).max() <= 2e-6 * np.abs(tag).max(), p


def test_c128_decode_large_batch_path_matches(env):
    """A decode batch too large for the persistent kernel's per-CTA row list
    (here 40000 rows, almost all invalid records) takes the one-CTA-per-(row,
    slice) kernel; its rows must be bit-identical to the same rows decoded in a
    small batch, and the invalid rows must be zero."""
    o, ckv, dev = env
    hd = 512
    sl = [128, 256, 5, 384, 1280, 7, 512, 130]
    w = wl.random_decode(128, hd, torch.bfloat16, torch.float32, sl, seed=9, num_requests_state=8)
    small_state = w.state.to(dev)
    out_small, pd_small = ckv.decode_step(128, hd, small_state, w.kv_score.to(dev), w.ape.to(dev), w.rid.to(dev),
                                          w.seq_lens.to(dev), torch.float32)
    B = 40000
    pos = np.sort(np.random.default_rng(1).choice(B, len(sl), replace=False))
    plan = torch.full((B, 16), 0xFF, dtype=torch.uint8, device=dev)
    plan[torch.as_tensor(pos, device=dev)] = pd_small
    kv = torch.zeros(B, 2 * hd, dtype=torch.bfloat16, device=dev)
    kv[torch.as_tensor(pos, device=dev)] = w.kv_score.to(dev)
    big_state = w.state.to(dev)
    status = ckv.new_status(dev)
    out_big = ckv.compress_decode(128, hd, big_state, kv, w.ape.to(dev), plan, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    assert torch.equal(out_big[torch.as_tensor(pos, device=dev)].view(torch.int32), out_small.view(torch.int32))
    mask = torch.ones(B, dtype=torch.bool, device=dev)
    mask[torch.as_tensor(pos, device=dev)] = False
    assert (out_big[mask].view(torch.int32) == 0).all()
    assert torch.equal(big_state.view(torch.int16), small_state.view(torch.int16))


@pytest.mark.parametrize("ratio,dts", [(128, ("bf16", "f32")), (128, ("f32", "bf16")), (4, ("bf16", "bf16")),
                                       (4, ("f32", "f32"))])
def test_prefill_every_buffer_len(env, ratio, dts):
    """Windows that start in the state with every possible number of state
    entries: request r has prefix r and extends to the first boundary, so its
    window holds r state entries (C128: 1 .. 127, every split of the state
    and input row ranges into copies; C4: prefixes 1 .. 7 and later groups)."""
    if ratio == 128:
        pl = list(range(1, 128))
        el = [128 - r for r in pl]
    else:
        pl = [1, 2, 3, 4, 5, 6, 7, 9, 10, 11, 13, 14, 15]
        el = [(4 - r % 4) % 4 + 4 * (1 + r % 3) for r in pl]
    _run_prefill_parity(env, ratio, 256, DT[dts[0]], DT[dts[1]], 1, pl, el, seed=77 + ratio)


@pytest.mark.parametrize("ratio,pl,el", [(4, [3], [1]), (4, [1], [3]), (4, [6], [2]), (128, [100], [28]),
                                         (128, [127], [1])])
def test_prefill_inputs_shorter_than_a_box(env, ratio, pl, el):
    """Ragged inputs of fewer rows than the pools' largest boxes (a handful of
    new tokens whose window is mostly in the state)."""
    for layout in (0, 1):
        _run_prefill_parity(env, ratio, 256, DT["bf16"], DT["f32"], layout, pl, el, seed=5 + ratio)
