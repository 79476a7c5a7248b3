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
@pytest.mark.parametrize("hinted", [False, True])
def test_prefill_step_replayed_from_a_graph(env, ratio, hinted):
    """With ``hinted`` the pool also takes the planner's inputs as prefetch
    hints (their contents change between replays, as the lengths do)."""
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
        ckv.compress_pool_prefill(ratio, hd, state, kv, ape, plan_c, counts, lay, out=out, status=status,
                                  hints=(rid, sl, el) if hinted else None)
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
@pytest.mark.parametrize("ordered", [True, False])
def test_decode_step_replayed_from_a_graph(env, ratio, ordered):
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
    order = ckv.new_decode_order(batch, dev) if ordered else None

    def step():
        ckv.plan_decode(ratio, rid, sl_d, plan_d, status, order=order)
        ckv.compress_decode(ratio, hd, state, kv, ape, plan_d, torch.float32, out=out, status=status, order=order,
                            **({"rid_hint": rid, "seq_lens_hint": sl_d} if ordered else {}))

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
        if ordered:
            assert (H.decode_order_entries(order) == H.expected_decode_order(wpd, ratio)).all()
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


def _replay_matches_eager(step, restore, outputs, mixes, load):
    """Captures `step` once; for every input mix, the graph replay leaves
    `outputs` bit-identical to an eager call of `step` on the same inputs
    (`restore` resets the state, outputs[0]; the other outputs start at zero)."""
    g = torch.cuda.CUDAGraph()
    step()  # eager once: first-call set-up happens outside the capture
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        step()
    for m in mixes:
        load(m)
        restore()
        for t in outputs[1:]:
            t.zero_()
        step()
        torch.cuda.synchronize()
        eager = [t.clone() for t in outputs]
        restore()
        for t in outputs[1:]:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(eager, outputs):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_online_steps_replayed_from_a_graph(env):
    """The online C128 state: plan + fold (two launches) for a prefill, and the
    decode fold, captured once and replayed on new length mixes."""
    o, ckv, dev = env
    hd, batch, nq = 256, 10, 700
    rng = np.random.default_rng(91)
    g = torch.Generator().manual_seed(92)
    slots = batch + 4
    init = torch.randn(slots, 3 * hd, generator=g)
    init[:, hd:2 * hd] = 1.0 + init[:, hd:2 * hd].abs()  # weight sums are >= 1
    init = init.to(dev)
    state = init.clone()
    ape = (torch.randn(128, hd, generator=g) * 0.5).to(torch.bfloat16).to(dev)
    i64 = dict(dtype=torch.int64, device=dev)
    rid, sl, el = torch.zeros(batch, **i64), torch.zeros(batch, **i64), torch.zeros(batch, **i64)
    kv = torch.zeros(nq, 2 * hd, dtype=torch.bfloat16, device=dev)
    cap_u = ckv.capacity_online_units(batch, nq)
    cap_c = ckv.capacity_compress(128, batch, nq)
    units = torch.empty(cap_u, 16, dtype=torch.uint8, device=dev)
    counts = torch.empty(4, dtype=torch.int32, device=dev)
    out = torch.empty(cap_c, hd, dtype=torch.float32, device=dev)
    status = ckv.new_status(dev)
    mixes = []
    for el_m in _compositions(rng, nq, batch, 3):
        pl_m = rng.integers(0, 400, batch)
        mixes.append((torch.from_numpy(rng.permutation(slots)[:batch].astype(np.int64)),
                      torch.from_numpy(pl_m + el_m), torch.from_numpy(el_m),
                      torch.randn(nq, 2 * hd, generator=g).to(torch.bfloat16)))

    def load(m):
        for dst, src in zip((rid, sl, el, kv), m):
            dst.copy_(src)

    def step():
        ckv.plan_online_prefill(rid, sl, el, nq, 0, cap_u, pad_invalid=True, units=units, counts=counts,
                                status=status)
        ckv.compress_online_prefill(hd, state, kv, ape, units, counts, ckv.OUT_COMPACT, out=out, status=status)

    load(mixes[0])
    _replay_matches_eager(step, lambda: state.copy_(init), [state, out], mixes, load)
    assert int(status[0]) == 0

    # decode
    plan_d = torch.empty(batch, 16, dtype=torch.uint8, device=dev)
    kvd = torch.zeros(batch, 2 * hd, dtype=torch.bfloat16, device=dev)
    outd = torch.empty(batch, hd, dtype=torch.float32, device=dev)
    dmixes = []
    for k in range(3):
        sl_m = rng.integers(1, 3000, batch)
        sl_m[: 3 + k] = 128 * rng.integers(1, 20, 3 + k)
        dmixes.append((torch.from_numpy(rng.permutation(slots)[:batch].astype(np.int64)), torch.from_numpy(sl_m),
                       torch.randn(batch, 2 * hd, generator=g).to(torch.bfloat16)))

    def dload(m):
        for dst, src in zip((rid, sl, kvd), m):
            dst.copy_(src)

    def dstep():
        ckv.plan_online_decode(rid, sl, 0, plan_d=plan_d, status=status)
        ckv.compress_online_decode(hd, state, kvd, ape, plan_d, out=outd, status=status)

    dload(dmixes[0])
    _replay_matches_eager(dstep, lambda: state.copy_(init), [state, outd], dmixes, dload)
    assert int(status[0]) == 0


def test_norm_rope_store_replayed_from_a_graph(env):
    """Decode, then RMSNorm + RoPE + store of its rows into a bf16 cache,
    captured once and replayed on new decode batches."""
    o, ckv, dev = env
    ratio, hd, rope, batch = 128, 512, 64, 64
    rng = np.random.default_rng(93)
    mixes = []
    for k in range(3):
        sl_m = rng.integers(1, 3000, batch)
        sl_m[: 10 + k] = 128 * rng.integers(1, 20, 10 + k)
        w = wl.random_decode(ratio, hd, torch.bfloat16, torch.float32, sl_m, seed=94 + k, num_requests_state=80)
        mixes.append((w.rid, w.seq_lens, w.kv_score, w.state,
                      torch.from_numpy(rng.permutation(2 * batch)[:batch].astype(np.int64))))
    w0 = wl.random_decode(ratio, hd, torch.bfloat16, torch.float32, mixes[0][1], seed=94, num_requests_state=80)
    rid, sl, kv = w0.rid.to(dev), w0.seq_lens.to(dev), w0.kv_score.to(dev)
    state0 = w0.state.to(dev)
    state = state0.clone()
    ape = w0.ape.to(dev)
    loc = torch.zeros(batch, dtype=torch.int64, device=dev)
    g = torch.Generator().manual_seed(95)
    weight = (1.0 + 0.1 * torch.randn(hd, generator=g)).to(dev)
    pos = torch.arange(4096, dtype=torch.float64)[:, None]
    inv = 10000.0 ** (-torch.arange(0, rope, 2, dtype=torch.float64) / rope)
    ang = pos * inv[None, :]
    freqs = torch.stack([ang.cos(), ang.sin()], dim=-1).to(torch.float32).contiguous().to(dev)
    cache = torch.zeros(2 * batch, hd, dtype=torch.bfloat16, device=dev)
    plan_d = torch.empty(batch, 16, dtype=torch.uint8, device=dev)
    rows = torch.empty(batch, hd, dtype=torch.float32, device=dev)
    status = ckv.new_status(dev)

    def load(m):
        for dst, src in zip((rid, sl, kv, state0, loc), m):
            dst.copy_(src)

    def step():
        ckv.plan_decode(ratio, rid, sl, plan_d, status)
        ckv.compress_decode(ratio, hd, state, kv, ape, plan_d, torch.float32, out=rows, status=status)
        ckv.norm_rope_store_decode(ratio, rows, plan_d, weight, 1e-6, freqs, loc, cache, status=status)

    _replay_matches_eager(step, lambda: (state.copy_(state0), cache.zero_()), [state, rows, cache], mixes, load)
    assert int(status[0]) == 0
