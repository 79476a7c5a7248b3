"""Parity at the seven named workloads' full sizes, in the launch configuration the
benchmark times (capacities from ckv_capacity_*, or num_q_tokens-sized plan
buffers padded with the invalid record for the speculative-decoding
workloads; plan -> pool (with the planner's inputs as prefetch hints) ->
write on one stream; plan -> decode).

Plans and state buffers are compared with the oracle byte for byte; decode
outputs in full; prefill outputs of every compress record (the oracle pools
them all), plus every non-compress row of token layouts (which must be +0.0).
"""
import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def env(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_attention_compressplan_gb300 import build as B
    from compressed_kv_attention_compressplan_gb300 import ckv

    B.build()
    ckv.load_library()
    return oracle_mod, ckv, torch.device("cuda")


def code(dt):
    return 1 if dt == torch.bfloat16 else 0


@pytest.mark.parametrize("name", ["c4_prefill_small", "c4_prefill", "c128_prefill", "c4_prefill_mtp",
                                  "c128_prefill_mtp"])
def test_prefill_workload_full_size(env, name):
    """The speculative-decoding workloads (``*_mtp``) run with fixed-shape plan
    buffers of num_q_tokens records whose tails are the invalid record, as a
    captured graph would."""
    o, ckv, dev = env
    w = wl.NAMED[name](0)
    R, hd = w.ratio, w.head_dim
    ci, co = code(w.in_dtype), code(w.out_dtype)
    nq = w.num_q_tokens
    padded = name.endswith("_mtp")
    cap_c = nq if padded else ckv.capacity_compress(R, w.batch, nq)
    cap_w = nq if padded else ckv.capacity_write(R, w.batch, nq)
    state_d = w.state.to(dev)
    kv_d = w.kv_score.to(dev)
    status = ckv.new_status(dev)
    layout = ckv.OUT_TOKEN if w.out_layout == wl.TOKEN else ckv.OUT_COMPACT
    lens = (w.rid.to(dev), w.seq_lens.to(dev), w.extend_lens.to(dev))
    pc, pw, counts = ckv.plan_prefill(R, *lens, nq, cap_c, cap_w, pad_invalid=padded, status=status)
    # with the planner's inputs as prefetch hints, as the benchmark launches it
    out = ckv.compress_prefill(R, hd, state_d, kv_d, w.ape.to(dev), pc, pw, counts, layout, w.out_dtype,
                               status=status, hints=lens)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    wc, ww, (nc, nw), _ = o.plan_prefill(R, w.rid, w.seq_lens, w.extend_lens)
    assert counts[:2].tolist() == [nc, nw]
    assert (pc[:nc].cpu().numpy() == wc).all(), "compress plan"
    assert (pw[:nw].cpu().numpy() == ww).all(), "write plan"
    if padded:
        pcp, pwp, _, _ = o.plan_prefill(R, w.rid, w.seq_lens, w.extend_lens, nq, cap_c, cap_w, pad_invalid=True)
        assert (pc.cpu().numpy() == pcp).all() and (pw.cpu().numpy() == pwp).all(), "padded plans"
    st = wl.bits(w.state).copy()
    inp = wl.bits(w.kv_score)
    ape = wl.bits(w.ape)
    want = o.compress_pool_prefill(R, hd, ci, co, st, inp, ape, np.ascontiguousarray(wc), nc, nq, o.OUT_COMPACT)
    f = H.plan_c_fields(wc)
    kvmax = H.window_kv_absmax(R, hd, st, inp, f["seq_len"], f["ragged_id"], f["buffer_len"], f["read_page_0"],
                               f["read_page_1"])
    got_all = H.np_bits(out)
    rows = f["ragged_id"] if layout == ckv.OUT_TOKEN else np.arange(nc)
    H.assert_pool_close(got_all[rows], want, co, kvmax, f"{name} every record")
    if layout == ckv.OUT_TOKEN:
        others = np.setdiff1d(np.arange(nq), H.plan_c_fields(wc)["ragged_id"])
        zero = got_all[others].view(np.uint16 if co else np.uint32)
        assert (zero == 0).all(), "non-compress rows"
    o.compress_write(R, hd, ci, st, inp, ww, nw)
    assert (H.np_bits(state_d).view(np.uint8) == st.view(np.uint8)).all(), "state after write"


@pytest.mark.parametrize("name", ["c4_decode", "c128_decode"])
@pytest.mark.parametrize("ordered", [True, False])
def test_decode_workload_full_size(env, name, ordered):
    """Every row of the decode workloads, through the boundary-row list with the
    prefetch hints (the benchmark's path) and through the plan scan."""
    o, ckv, dev = env
    w = wl.NAMED[name](0)
    R, hd = w.ratio, w.head_dim
    ci, co = code(w.in_dtype), code(w.out_dtype)
    state_d = w.state.to(dev)
    status = ckv.new_status(dev)
    order = ckv.new_decode_order(w.batch, dev) if ordered else None
    pd = ckv.plan_decode(R, w.rid.to(dev), w.seq_lens.to(dev), status=status, order=order)
    hints = {"rid_hint": w.rid.to(dev), "seq_lens_hint": w.seq_lens.to(dev)} if ordered else {}
    out = ckv.compress_decode(R, hd, state_d, w.kv_score.to(dev), w.ape.to(dev), pd, w.out_dtype, status=status,
                              order=order, **hints)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    wpd = o.plan_decode(R, w.rid, w.seq_lens)
    assert (pd.cpu().numpy() == wpd).all()
    if ordered:
        assert (H.decode_order_entries(order) == H.expected_decode_order(wpd, R)).all()
    st0 = wl.bits(w.state).copy()
    st = st0.copy()
    inp = wl.bits(w.kv_score)
    want = o.compress_decode(R, hd, ci, co, st, inp, wl.bits(w.ape), wpd)
    got = H.np_bits(out)
    f = H.plan_d_fields(wpd)
    bnd = np.nonzero(f["seq_len"] % R == 0)[0]
    kvmax = H.window_kv_absmax(R, hd, st0, inp, f["seq_len"][bnd], bnd, np.full(len(bnd), H.window(R) - 1),
                               f["read_page_0"][bnd], f["read_page_1"][bnd])
    H.assert_pool_close(got[bnd], want[bnd], co, kvmax, f"{name} boundary rows")
    nb = np.setdiff1d(np.arange(w.batch), bnd)
    assert (got[nb].view(np.uint16 if co else np.uint32) == 0).all()
    assert (H.np_bits(state_d).view(np.uint8) == st.view(np.uint8)).all(), "state after decode"


def test_paged_prefill_workload_full_size(env):
    """The C4 prefill workload over SWA-paged state (128-token SWA pages, 8-row
    rings), in the benchmark's launch configuration: paged plans bit-exact,
    every pooled row, every zero row, and the state after the write."""
    o, ckv, dev = env
    w, m = wl.PAGED["c4_prefill_paged"](0)
    R, hd, nq = w.ratio, w.head_dim, w.num_q_tokens
    state_d = w.state.to(dev)
    status = ckv.new_status(dev)
    pc, pw, counts = ckv.plan_prefill_paged(R, w.rid.to(dev), m.req_to_token.to(dev), m.full_to_state.to(dev),
                                            m.swa_page_size, m.ring_size, w.seq_lens.to(dev), w.extend_lens.to(dev),
                                            nq, status=status)
    out = ckv.compress_prefill(R, hd, state_d, w.kv_score.to(dev), w.ape.to(dev), pc, pw, counts, ckv.OUT_TOKEN,
                               w.out_dtype, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    wc, ww, (nc, nw), _ = o.plan_prefill_paged(R, w.rid, m.req_to_token.numpy(), m.full_to_state.numpy(),
                                               m.swa_page_size, m.ring_size, w.seq_lens, w.extend_lens)
    assert counts[:2].tolist() == [nc, nw]
    assert (pc[:nc].cpu().numpy() == wc).all() and (pw[:nw].cpu().numpy() == ww).all(), "paged plans"
    st = wl.bits(w.state).copy()
    inp = wl.bits(w.kv_score)
    want = o.compress_pool_prefill(R, hd, 1, 1, st, inp, wl.bits(w.ape), np.ascontiguousarray(wc), nc, nq,
                                   o.OUT_COMPACT)
    f = H.plan_c_fields(wc)
    kvmax = H.window_kv_absmax(R, hd, st, inp, f["seq_len"], f["ragged_id"], f["buffer_len"], f["read_page_0"],
                               f["read_page_1"])
    got = H.np_bits(out)
    H.assert_pool_close(got[f["ragged_id"]], want, 1, kvmax, "paged, every record")
    others = np.setdiff1d(np.arange(nq), H.plan_c_fields(wc)["ragged_id"])
    assert (got[others] == 0).all(), "non-compress rows"
    o.compress_write(R, hd, 1, st, inp, ww, nw)
    assert (H.np_bits(state_d).view(np.uint8) == st.view(np.uint8)).all(), "state after write"
