"""Seeded random sweep of the prefill and decode paths against the oracle.

Each case draws the ratio, head_dim (128 .. 1024, so every tile and view
shape of the staged pools), the dtype pair, the output layout, the batch and
the prefix / extend mix (prefixes that start mid-group, extends of one token,
long windows), then runs plan + pool + write, or plan + decode, through the C
ABI and checks them with the same bar as the fixed parity cases: plans and
state bit-exact, fp32 outputs within 2e-6 * max|kv|, bf16 within 1 ulp.  The
"wide" cases draw larger batches and lengths, equal extends (the planner's
token-driven path) and the optional boundary-row list and prefetch hints.
"""
import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H
from tests.test_gpu_parity import _run_prefill_parity

pytestmark = pytest.mark.gpu

HEAD_DIMS = [128, 256, 384, 512, 640, 768, 896, 1024]
DTYPES = [(1, 0), (1, 1), (0, 0), (0, 1)]


@pytest.fixture(scope="module")
def env(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_attention_compressplan_gb300 import build as B
    from compressed_kv_attention_compressplan_gb300 import ckv

    B.build()
    ckv.load_library()
    return oracle_mod, ckv, torch.device("cuda")


@pytest.mark.parametrize("case", range(24))
def test_random_prefill(env, case):
    rng = np.random.default_rng(1000 + case)
    ratio = int(rng.choice([4, 128]))
    hd = int(rng.choice(HEAD_DIMS))
    in_dt, out_dt = DTYPES[int(rng.integers(len(DTYPES)))]
    layout = int(rng.integers(2))
    batch = int(rng.integers(1, 12))
    span = 3 * ratio if ratio == 128 else 40
    pl = rng.integers(0, span, batch)
    el = rng.integers(1, span, batch)
    if batch > 2:  # a one-token extend and a request from position 0
        el[0] = 1
        pl[1] = 0
    _run_prefill_parity(env, ratio, hd, in_dt, out_dt, layout, list(pl), list(el), seed=2000 + case,
                        outliers=0.01 if ratio == 128 else 0.0)


@pytest.mark.parametrize("case", range(12))
def test_random_decode(env, case):
    o, ckv, dev = env
    rng = np.random.default_rng(3000 + case)
    ratio = int(rng.choice([4, 128]))
    hd = int(rng.choice(HEAD_DIMS))
    in_dt, out_dt = DTYPES[int(rng.integers(len(DTYPES)))]
    B = int(rng.integers(1, 300))
    sl = rng.integers(1, 4000, B)
    nb = int(rng.integers(0, B + 1))
    sl[:nb] = ratio * rng.integers(1, 30, nb)  # page / group boundary rows
    w = wl.random_decode(ratio, hd, H.torch_dtype(in_dt), H.torch_dtype(out_dt), sl, seed=4000 + case,
                         num_requests_state=B + 5)
    state_d = w.state.to(dev)
    status = ckv.new_status(dev)
    out, pd = ckv.decode_step(ratio, hd, state_d, w.kv_score.to(dev), w.ape.to(dev), w.rid.to(dev),
                              w.seq_lens.to(dev), H.torch_dtype(out_dt), status=status)
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
    if len(bnd):
        kvmax = H.window_kv_absmax(ratio, hd, st0, inp, f["seq_len"][bnd], bnd, np.full(len(bnd), H.window(ratio) - 1),
                                   f["read_page_0"][bnd], f["read_page_1"][bnd])
        H.assert_pool_close(got[bnd], want[bnd], out_dt, kvmax, "random decode boundary rows")
    nb_rows = np.setdiff1d(np.arange(B), bnd)
    assert (got[nb_rows].view(np.uint16 if out_dt else np.uint32) == 0).all()
    assert (H.np_bits(state_d).view(np.uint8) == st.view(np.uint8)).all(), "state after decode"


@pytest.mark.parametrize("case", range(60))
def test_random_prefill_wide(env, case):
    """Wider mixes: batches up to 63, speculative-decoding-like equal extends of
    1 .. 33 tokens over long prefixes, and long extends (up to 20000 tokens in
    all); about half of the cases hand the pool the prefetch hints."""
    rng = np.random.default_rng(50000 + case)
    ratio = int(rng.choice([4, 128]))
    hd = int(rng.choice(HEAD_DIMS))
    in_dt, out_dt = DTYPES[int(rng.integers(len(DTYPES)))]
    layout = int(rng.integers(2))
    batch = int(rng.integers(1, 64))
    kind = int(rng.integers(3))
    if kind == 0:    # equal extends (the planner's token-driven path)
        el = np.full(batch, int(rng.integers(1, 34)))
        pl = rng.integers(0, 3000, batch)
    elif kind == 1:  # long extends
        el = rng.integers(1, 1500, batch)
        pl = rng.integers(0, 1000, batch)
    else:
        span = 3 * ratio if ratio == 128 else 40
        pl = rng.integers(0, span, batch)
        el = rng.integers(1, span, batch)
    while int(el.sum()) > 20000:
        el = np.maximum(1, el // 2)
    _run_prefill_parity(env, ratio, hd, in_dt, out_dt, layout, list(pl), list(el), seed=60000 + case,
                        outliers=0.01 if ratio == 128 else 0.0)


@pytest.mark.parametrize("case", range(40))
def test_random_decode_wide(env, case):
    """Batches up to 3000 rows (C4) / 400 (C128), with or without the
    boundary-row list and with or without the prefetch hints."""
    o, ckv, dev = env
    rng = np.random.default_rng(70000 + case)
    ratio = int(rng.choice([4, 128]))
    hd = int(rng.choice(HEAD_DIMS))
    in_dt, out_dt = DTYPES[int(rng.integers(len(DTYPES)))]
    B = int(rng.integers(1, 3000 if ratio == 4 else 400))
    sl = rng.integers(1, 40000, B)
    nb = int(rng.integers(0, B + 1))
    sl[:nb] = ratio * rng.integers(1, 300, nb)
    rng.shuffle(sl)
    w = wl.random_decode(ratio, hd, H.torch_dtype(in_dt), H.torch_dtype(out_dt), sl, seed=80000 + case,
                         num_requests_state=B + 5)
    state_d = w.state.to(dev)
    status = ckv.new_status(dev)
    order = ckv.new_decode_order(B, dev) if rng.integers(2) else None
    hints = {"rid_hint": w.rid.to(dev), "seq_lens_hint": w.seq_lens.to(dev)} if rng.integers(2) else {}
    pd = ckv.plan_decode(ratio, w.rid.to(dev), w.seq_lens.to(dev), status=status, order=order)
    out = ckv.compress_decode(ratio, hd, state_d, w.kv_score.to(dev), w.ape.to(dev), pd, H.torch_dtype(out_dt),
                              status=status, order=order, **hints)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    st0 = wl.bits(w.state).copy()
    st = st0.copy()
    wpd = o.plan_decode(ratio, w.rid, w.seq_lens)
    assert (pd.cpu().numpy() == wpd).all()
    if order is not None:
        assert (H.decode_order_entries(order) == H.expected_decode_order(wpd, ratio)).all()
    inp = wl.bits(w.kv_score)
    want = o.compress_decode(ratio, hd, in_dt, out_dt, st, inp, wl.bits(w.ape), wpd)
    got = H.np_bits(out)
    f = H.plan_d_fields(wpd)
    bnd = np.nonzero(f["seq_len"] % ratio == 0)[0]
    if len(bnd):
        kvmax = H.window_kv_absmax(ratio, hd, st0, inp, f["seq_len"][bnd], bnd, np.full(len(bnd), H.window(ratio) - 1),
                                   f["read_page_0"][bnd], f["read_page_1"][bnd])
        H.assert_pool_close(got[bnd], want[bnd], out_dt, kvmax, "wide random decode boundary rows")
    nb_rows = np.setdiff1d(np.arange(B), bnd)
    assert (got[nb_rows].view(np.uint16 if out_dt else np.uint32) == 0).all()
    assert (H.np_bits(state_d).view(np.uint8) == st.view(np.uint8)).all(), "state after decode"
