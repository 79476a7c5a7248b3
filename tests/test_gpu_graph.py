"""CUDA-graph capture through the C ABI.

No call reads device data on the host (grid sizes come from host-known
capacities, the kernels read the true record counts on the device), so a whole
step can be captured once and replayed on new inputs of the same shapes: the
fixed-size plan buffers are padded with the invalid record, the shape the
pages' CUDA-graph path asks for.  Each replay is checked against the oracle
with the same bar as the eager calls: plans and state bit-exact, outputs
within 2e-6 * max|kv| (fp32).
"""
import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_attention_compressplan_gb300 import build as B
    from compressed_kv_attention_compressplan_gb300 import ckv

    B.build()
    ckv.load_library()
    return oracle_mod, ckv, torch.device("cuda")


def _compositions(rng, total, parts, count):
    """`count` different ways to split `total` tokens over `parts` requests (each >= 1)."""
    out = []
    for _ in range(count):
        cuts = np.sort(rng.choice(np.arange(1, total), parts - 1, replace=False))
        out.append(np.diff(np.concatenate([[0], cuts, [total]])).astype(np.int64))
    return out


@pytest.mark.parametrize("ratio", [4, 128])
def test_prefill_step_replayed_from_a_graph(env, ratio):
    o, ckv, dev = env
    hd, in_dt, out_dt = 256, 1, 0
    layout = wl.TOKEN if ratio == 4 else wl.COMPACT
    lay = ckv.OUT_TOKEN if ratio == 4 else ckv.OUT_COMPACT
    batch, nq = 12, 900
    rng = np.random.default_rng(50 + ratio)
    mixes = []
    for k, el in enumerate(_compositions(rng, nq, batch, 3)):
        pl = rng.integers(0, 300, batch)
        mixes.append(wl.random_prefill(ratio, hd, torch.bfloat16, torch.float32, layout, pl, el, seed=70 + k,
                                       num_requests_state=batch + 3))
    cap_c = ckv.capacity_compress(ratio, batch, nq)
    cap_w = ckv.capacity_write(ratio, batch, nq)
    w0 = mixes[0]
    rid, sl, el = w0.rid.to(dev), w0.seq_lens.to(dev), w0.extend_lens.to(dev)
    kv, state, ape = w0.kv_score.to(dev), w0.state.to(dev), w0.ape.to(dev)
    plan_c = torch.empty(cap_c, 16, dtype=torch.uint8, device=dev)
    plan_w = torch.empty(cap_w, 8, dtype=torch.uint8, device=dev)
    counts = torch.empty(4, dtype=torch.int32, device=dev)
    status = ckv.new_status(dev)
    out = torch.empty(nq if ratio == 4 else cap_c, hd, dtype=torch.float32, device=dev)

    def step():
        ckv.plan_prefill(ratio, rid, sl, el, nq, cap_c, cap_w, pad_invalid=True, plan_c=plan_c, plan_w=plan_w,
                         counts=counts, status=status)
        ckv.compress_pool_prefill(ratio, hd, state, kv, ape, plan_c, counts, lay, out=out, status=status)
        ckv.compress_write(ratio, hd, state, kv, plan_w, counts, status=status)

    step()  # eager once: first-call set-up (kernel attributes) happens outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for w in (mixes[1], mixes[2], mixes[0]):
        for dst, src in ((rid, w.rid), (sl, w.seq_lens), (el, w.extend_lens), (kv, w.kv_score), (state, w.state),
                         (ape, w.ape)):
            dst.copy_(src)
        status.zero_()
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert int(status[0]) == 0
        st = wl.bits(w.state).copy()
        inp = wl.bits(w.kv_score)
        wc, ww, (nc, nw), _ = o.plan_prefill(ratio, w.rid, w.seq_lens, w.extend_lens, nq, cap_c, cap_w)
        assert counts[:2].tolist() == [nc, nw]
        assert (plan_c.cpu().numpy()[:nc] == wc[:nc]).all() and (plan_c.cpu().numpy()[nc:] == 0xFF).all()
        assert (plan_w.cpu().numpy()[:nw] == ww[:nw]).all() and (plan_w.cpu().numpy()[nw:] == 0xFF).all()
        want = o.compress_pool_prefill(ratio, hd, in_dt, out_dt, st, inp, wl.bits(w.ape), wc[:nc], nc, nq,
                                       0 if ratio == 4 else 1)
        f = H.plan_c_fields(wc[:nc])
        kvmax = H.window_kv_absmax(ratio, hd, st, inp, f["seq_len"], f["ragged_id"], f["buffer_len"],
                                   f["read_page_0"], f["read_page_1"])
        got = H.np_bits(out)
        if ratio == 4:
            rows = f["ragged_id"]
            H.assert_pool_close(got[rows], want[rows], out_dt, kvmax, "graph replay: compress rows")
            others = np.setdiff1d(np.arange(nq), rows)
            assert (got[others].view(np.uint32) == 0).all(), "graph replay: non-compress rows not zero"
        else:
            H.assert_pool_close(got[:nc], want, out_dt, kvmax, "graph replay: compact rows")
        o.compress_write(ratio, hd, in_dt, st, inp, ww[:nw], nw)
        assert (H.np_bits(state).view(np.uint8) == st.view(np.uint8)).all(), "graph replay: state after write"


@pytest.mark.parametrize("ratio", [4, 128])
def test_decode_step_replayed_from_a_graph(env, ratio):
    o, ckv, dev = env
    hd, in_dt, out_dt = 256, 1, 0
    batch = 97
    rng = np.random.default_rng(60 + ratio)
    mixes = []
    for k in range(3):
        sl = rng.integers(1, 3000, batch)
        sl[: 20 + 5 * k] = ratio * rng.integers(1, 20, 20 + 5 * k)  # page-boundary rows
        mixes.append(wl.random_decode(ratio, hd, torch.bfloat16, torch.float32, sl, seed=80 + k,
                                      num_requests_state=128))
    w0 = mixes[0]
    rid, sl_d = w0.rid.to(dev), w0.seq_lens.to(dev)
    kv, state, ape = w0.kv_score.to(dev), w0.state.to(dev), w0.ape.to(dev)
    plan_d = torch.empty(batch, 16, dtype=torch.uint8, device=dev)
    out = torch.empty(batch, hd, dtype=torch.float32, device=dev)
    status = ckv.new_status(dev)

    def step():
        ckv.plan_decode(ratio, rid, sl_d, plan_d, status)
        ckv.compress_decode(ratio, hd, state, kv, ape, plan_d, torch.float32, out=out, status=status)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for w in (mixes[1], mixes[2], mixes[0]):
        for dst, src in ((rid, w.rid), (sl_d, w.seq_lens), (kv, w.kv_score), (state, w.state), (ape, w.ape)):
            dst.copy_(src)
        status.zero_()
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert int(status[0]) == 0
        st0 = wl.bits(w.state).copy()
        st = st0.copy()
        wpd = o.plan_decode(ratio, w.rid, w.seq_lens)
        assert (plan_d.cpu().numpy() == wpd).all()
        inp = wl.bits(w.kv_score)
        want = o.compress_decode(ratio, hd, in_dt, out_dt, st, inp, wl.bits(w.ape), wpd)
        got = H.np_bits(out)
        f = H.plan_d_fields(wpd)
        bnd = np.nonzero(f["seq_len"] % ratio == 0)[0]
        kvmax = H.window_kv_absmax(ratio, hd, st0, inp, f["seq_len"][bnd], bnd, np.full(len(bnd), H.window(ratio) - 1),
                                   f["read_page_0"][bnd], f["read_page_1"][bnd])
        H.assert_pool_close(got[bnd], want[bnd], out_dt, kvmax, "graph replay: decode boundary rows")
        nb = np.setdiff1d(np.arange(batch), bnd)
        assert (got[nb].view(np.uint32) == 0).all()
        assert (H.np_bits(state).view(np.uint8) == st.view(np.uint8)).all(), "graph replay: state after decode"
