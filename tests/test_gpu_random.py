"""Seeded random sweep of the prefill and decode paths against the oracle.

Each case draws the ratio, head_dim (128 .. 1024, so every tile and view
shape of the staged pools), the dtype pair, the output layout, the batch and
the prefix / extend mix (prefixes that start mid-group, extends of one token,
long windows), then runs plan + pool + write, or plan + decode, through the C
ABI and checks them with the same bar as the fixed parity cases: plans and
state bit-exact, fp32 outputs within 2e-6 * max|kv|, bf16 within 1 ulp.
"""
import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H
from tests.test_gpu_parity import _run_prefill_parity

pytestmark = pytest.mark.gpu

HEAD_DIMS = [128, 256, 384, 512, 640, 768, 1024]
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
