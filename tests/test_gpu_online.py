"""GPU parity of the online C128 state (ckv_plan_online_prefill / _decode,
ckv_compress_online_prefill / _decode) against the oracle.

Bar: unit and decode plans bit-exact; the running maxima of the state
bit-exact (kept as fp32(m * log2 e), the product of a maximum of identically
rounded scores); emitted rows within
2e-6 * max|kv| of the window (fp32) or 1 ulp / that bound (bf16) against the
whole-history window definition; the same bits on the GPU whether a sequence
comes as one prefill, in chunks or token by token.
"""
import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H

pytestmark = pytest.mark.gpu

L2E = np.float32(1.4426950408889634)  # log2(e) in fp32: the library's m2 = fp32(m * log2(e))


@pytest.fixture(scope="module")
def env(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_attention_compressplan_gb300 import build as B
    from compressed_kv_attention_compressplan_gb300 import ckv

    B.build()
    ckv.load_library()
    return oracle_mod, ckv, torch.device("cuda")


class OnlineGpuBackend:
    def __init__(self, ckv, dev, slot_offset=0):
        self.ckv, self.dev, self.off = ckv, dev, slot_offset
        self.status = ckv.new_status(dev)

    def prefill(self, ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl, el):
        c, d = self.ckv, self.dev
        i64 = dict(dtype=torch.int64, device=d)
        units, counts = c.plan_online_prefill(torch.tensor(rid, **i64), torch.tensor(sl, **i64),
                                              torch.tensor(el, **i64), len(rows), self.off, status=self.status)
        out = c.compress_online_prefill(hd, state, H.to_torch(rows, in_dt).to(d), H.to_torch(ape, in_dt).to(d), units,
                                        counts, c.OUT_TOKEN, H.torch_dtype(out_dt), status=self.status)
        return H.np_bits(out)

    def decode(self, ratio, hd, in_dt, out_dt, state, rows, ape, rid, sl):
        c, d = self.ckv, self.dev
        i64 = dict(dtype=torch.int64, device=d)
        pd = c.plan_online_decode(torch.tensor(rid, **i64), torch.tensor(sl, **i64), self.off, status=self.status)
        out = c.compress_online_decode(hd, state, H.to_torch(rows, in_dt).to(d), H.to_torch(ape, in_dt).to(d), pd,
                                       H.torch_dtype(out_dt), status=self.status)
        return H.np_bits(out)


@pytest.mark.parametrize("case", ["small", "batch1024", "long"])
@pytest.mark.parametrize("pad", [False, True])
def test_online_plans_bit_exact(env, case, pad):
    o, ckv, dev = env
    rng = np.random.default_rng(len(case) + pad)
    if case == "small":
        B, maxl = 6, 600
    elif case == "batch1024":
        B, maxl = 1024, 300
    else:
        B, maxl = 3, 40000
    sl = rng.integers(1, maxl, B)
    el = np.array([int(rng.integers(1, s + 1)) if rng.random() < 0.6 else int(s) for s in sl])
    rid = rng.permutation(B + 5)[:B]
    nq = int(el.sum())
    cap = nq if pad else ckv.capacity_online_units(B, nq)
    i64 = dict(dtype=torch.int64, device=dev)
    status = ckv.new_status(dev)
    units, counts = ckv.plan_online_prefill(torch.tensor(rid, **i64), torch.tensor(sl, **i64),
                                            torch.tensor(el, **i64), nq, 7, cap, pad_invalid=pad, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    want, (nu, nc), _ = o.plan_online_prefill(rid, sl, el, 7, nq, cap, pad_invalid=pad)
    assert counts[:2].tolist() == [nc, nu]
    n = cap if pad else nu
    assert (units[:n].cpu().numpy() == want[:n]).all()
    pd = ckv.plan_online_decode(torch.tensor(rid, **i64), torch.tensor(sl, **i64), 7, status=status)
    assert (pd.cpu().numpy() == o.plan_online_decode(rid, sl, 7)).all()


# head_dim 128 gives the prefill kernel its smallest CTA (one consumer warp);
# 1024 with fp32 input its largest ring (288 threads, 168 KB of stages).
@pytest.mark.parametrize("hd,in_dt,out_dt", [(512, 1, 0), (512, 0, 0), (512, 1, 1), (128, 1, 0), (384, 0, 1),
                                             (1024, 0, 0), (1024, 1, 0)])
def test_online_modes_bitwise_and_window_parity(env, hd, in_dt, out_dt):
    o, ckv, dev = env
    rng = np.random.default_rng(3 + in_dt + 2 * out_dt + hd)
    nreq = 5
    lens = [int(rng.integers(1, 3 * 128 + 80)) for _ in range(nreq)]
    rids = [int(x) for x in rng.permutation(8)[:nreq]]
    tdt = torch.bfloat16 if in_dt else torch.float32
    g = torch.Generator().manual_seed(90 + in_dt)
    hist = [wl.bits(torch.randn(n, 2 * hd, generator=g).to(tdt)).copy() for n in lens]
    ape = wl.bits((torch.randn(128, hd, generator=g) * 0.5).to(tdt)).copy()
    want = [o.compress_history(128, hd, in_dt, out_dt, h, ape) for h in hist]
    backend = OnlineGpuBackend(ckv, dev, slot_offset=1)
    results = {}
    for mode in ["oneshot", "chunked", "decode", "mixed"]:
        if mode == "oneshot":
            sched = [[("prefill", n)] for n in lens]
        elif mode == "chunked":
            sched = [H.split_schedule(n, rng, 150, 0.0) for n in lens]
        elif mode == "decode":
            sched = [[("decode", 1)] * n for n in lens]
        else:
            sched = [H.split_schedule(n, rng, 70, 0.5) for n in lens]
        state = torch.full((9, 3 * hd), float("nan"), device=dev)
        results[mode] = H.run_schedule(backend, 128, hd, in_dt, out_dt, hist, rids, sched, ape, state)
        assert int(backend.status[0]) == 0
    view = np.uint16 if out_dt else np.uint32
    for b in range(nreq):
        ref = results["oneshot"][b]
        for mode in ["chunked", "decode", "mixed"]:
            assert (results[mode][b].view(view) == ref.view(view)).all(), (mode, b)
        emit = [p for p in range(lens[b]) if (p + 1) % 128 == 0]
        zero = np.setdiff1d(np.arange(lens[b]), emit)
        assert (ref[zero].view(view) == 0).all()
        if emit:
            tok = hist[b]
            kvmax = H.window_kv_absmax(128, hd, tok, tok, np.array(emit) + 1, np.array(emit),
                                       np.zeros(len(emit), np.int64), np.zeros(len(emit)), np.zeros(len(emit)))
            H.assert_pool_close(ref[emit], want[b][emit], out_dt, kvmax, f"online b={b}")


@pytest.mark.parametrize("case", range(20))
def test_online_random_schedules(env, case):
    """Seeded random histories and schedules through the online state: head_dim
    128 .. 1024, any dtype pair, 1 .. 8 requests of up to 700 tokens fed as
    chunked prefills, decodes or a mix; every emitted row against the window
    definition and bitwise equal to the one-shot prefill."""
    o, ckv, dev = env
    rng = np.random.default_rng(40000 + case)
    hd = int(rng.choice([128, 256, 384, 512, 640, 768, 896, 1024]))
    in_dt, out_dt = [(1, 0), (1, 1), (0, 0), (0, 1)][int(rng.integers(4))]
    nreq = int(rng.integers(1, 9))
    lens = [int(rng.integers(1, 701)) for _ in range(nreq)]
    rids = [int(x) for x in rng.permutation(nreq + 3)[:nreq]]
    tdt = torch.bfloat16 if in_dt else torch.float32
    g = torch.Generator().manual_seed(500 + case)
    hist = [wl.bits(torch.randn(n, 2 * hd, generator=g).to(tdt)).copy() for n in lens]
    ape = wl.bits((torch.randn(128, hd, generator=g) * 0.5).to(tdt)).copy()
    backend = OnlineGpuBackend(ckv, dev, slot_offset=int(rng.integers(0, 3)))
    chunk = int(rng.choice([20, 70, 150, 400]))
    dec_frac = float(rng.choice([0.0, 0.3, 0.7]))
    results = {}
    for mode, sched in [("oneshot", [[("prefill", n)] for n in lens]),
                        ("random", [H.split_schedule(n, rng, chunk, dec_frac) for n in lens])]:
        state = torch.full((nreq + 6, 3 * hd), float("nan"), device=dev)
        results[mode] = H.run_schedule(backend, 128, hd, in_dt, out_dt, hist, rids, sched, ape, state)
        assert int(backend.status[0]) == 0
    view = np.uint16 if out_dt else np.uint32
    for b in range(nreq):
        ref = results["oneshot"][b]
        assert (results["random"][b].view(view) == ref.view(view)).all(), b
        emit = [p for p in range(lens[b]) if (p + 1) % 128 == 0]
        if emit:
            want = o.compress_history(128, hd, in_dt, out_dt, hist[b], ape)
            tok = hist[b]
            kvmax = H.window_kv_absmax(128, hd, tok, tok, np.array(emit) + 1, np.array(emit),
                                       np.zeros(len(emit), np.int64), np.zeros(len(emit)), np.zeros(len(emit)))
            H.assert_pool_close(ref[emit], want[emit], out_dt, kvmax, f"online random b={b}")


def test_online_state_and_compact_rows(env):
    """One prefill step from a state folded by the oracle: compact rows, the
    state after it (maxima bit-exact, sums to fp32 accuracy) and bad units."""
    o, ckv, dev = env
    hd = 256
    rng = np.random.default_rng(12)
    B = 40
    pl = rng.integers(0, 1000, B)
    el = rng.integers(1, 600, B)
    sl = pl + el
    rid = rng.permutation(B)
    g = torch.Generator().manual_seed(5)
    ape = wl.bits((torch.randn(128, hd, generator=g) * 0.5).to(torch.bfloat16)).copy()
    # the state of each request's current group, folded from synthetic prefix tokens by the oracle
    st64 = np.zeros((B, 3 * hd))
    part = pl % 128
    for b in range(B):
        if part[b]:
            toks = wl.bits(torch.randn(int(part[b]), 2 * hd, generator=g).to(torch.bfloat16)).copy()
            u, _, _ = o.plan_online_prefill([rid[b]], [int(pl[b])], [int(part[b])])
            o.online_prefill(hd, 1, 0, st64, toks, ape, u)
    st32 = st64.astype(np.float32)
    st64 = st32.astype(np.float64)  # both sides start from the same fp32 values
    # the library keeps m2 = fp32(m * log2(e)) in place of the maximum m
    gpu_init = st32.copy()
    gpu_init[:, :hd] = st32[:, :hd] * L2E
    nq = int(el.sum())
    inp = wl.bits(torch.randn(nq, 2 * hd, generator=g).to(torch.bfloat16)).copy()
    units, (nu, nc), _ = o.plan_online_prefill(rid, sl, el)
    want = o.online_prefill(hd, 1, 0, st64, inp, ape, units, o.OUT_COMPACT, nc)
    state = torch.from_numpy(gpu_init).to(dev)
    status = ckv.new_status(dev)
    counts = torch.tensor([nc, nu, 0, 0], dtype=torch.int32, device=dev)
    out = ckv.compress_online_prefill(hd, state, H.to_torch(inp, 1).to(dev), H.to_torch(ape, 1).to(dev),
                                      torch.from_numpy(units).to(dev), counts, ckv.OUT_COMPACT, torch.float32,
                                      out_rows=nc, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    got = out.cpu().numpy()
    scale = np.abs(H.bf16_to_f32(inp[:, :hd])).max()
    assert np.abs(got - want).max() <= 4e-6 * scale
    gs = state.cpu().numpy().reshape(B, 3, hd)
    ws = st64.reshape(B, 3, hd)
    assert (gs[:, 0] == ws[:, 0].astype(np.float32) * L2E).all(), "running maxima"
    np.testing.assert_allclose(gs[:, 1], ws[:, 1], rtol=2e-5, atol=0)  # sums of positive weights
    # weighted sums may cancel: bound them by the weight sum times max|kv|
    assert (np.abs(gs[:, 2] - ws[:, 2]) <= 2e-5 * ws[:, 1] * scale).all()
    # a unit naming a slot past the state is skipped and flagged
    bad = units.copy()
    bad.view(np.int32).reshape(-1, 4)[0, 2] = B + 100
    status.zero_()
    ckv.compress_online_prefill(hd, state, H.to_torch(inp, 1).to(dev), H.to_torch(ape, 1).to(dev),
                                torch.from_numpy(bad).to(dev), counts, ckv.OUT_COMPACT, torch.float32, out_rows=nc,
                                status=status)
    torch.cuda.synchronize()
    assert int(status[0]) & ckv.STATUS_BAD_INDEX


def _fold_prefix(o, ckv, dev, x, hd):
    """Each side folds the requests' earlier tokens of their current group into its own state."""
    batch = x.rid.numel()
    st64 = np.zeros((batch, 3 * hd))
    st = torch.zeros(batch, 3 * hd, dtype=torch.float32, device=dev)
    has = (x.prefix_lens > 0).numpy()
    end = (x.seq_lens - (x.extend_lens if x.extend_lens is not None else 1)).numpy()
    n = int(x.prefix_lens.sum())
    rows = wl.bits(x.prefix_rows)
    ape = wl.bits(x.ape)
    units, _, _ = o.plan_online_prefill(x.rid.numpy()[has], end[has], x.prefix_lens.numpy()[has])
    o.online_prefill(hd, 1, 0, st64, rows, ape, units)
    i64 = dict(dtype=torch.int64, device=dev)
    gu, gc = ckv.plan_online_prefill(torch.tensor(x.rid.numpy()[has], **i64), torch.tensor(end[has], **i64),
                                     torch.tensor(x.prefix_lens.numpy()[has], **i64), n)
    ckv.compress_online_prefill(hd, st, x.prefix_rows.to(dev), x.ape.to(dev), gu, gc, ckv.OUT_TOKEN)
    return st64, st


@pytest.mark.slow
def test_full_size_online_prefill(env):
    """The C128 prefill workload through the online state, in the benchmark's
    launch configuration; every emitted row checked against the oracle folding
    the same units."""
    o, ckv, dev = env
    x = wl.c128_online_prefill(0)
    hd = x.head_dim
    st64, st = _fold_prefix(o, ckv, dev, x, hd)
    nq = int(x.extend_lens.sum())
    i64 = dict(dtype=torch.int64, device=dev)
    status = ckv.new_status(dev)
    units, counts = ckv.plan_online_prefill(x.rid.to(dev), x.seq_lens.to(dev), x.extend_lens.to(dev), nq,
                                            status=status)
    cap_c = ckv.capacity_compress(128, x.rid.numel(), nq)
    out = ckv.compress_online_prefill(hd, st, x.kv_score.to(dev), x.ape.to(dev), units, counts, ckv.OUT_COMPACT,
                                      out_rows=cap_c, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    wu, (nu, nc), _ = o.plan_online_prefill(x.rid, x.seq_lens, x.extend_lens)
    assert counts[:2].tolist() == [nc, nu] and (units[:nu].cpu().numpy() == wu).all()
    w = wu.view(np.uint32).reshape(-1, 4)
    pick = np.nonzero((w[:, 3] >> 24) & 2)[0]  # every emitting unit
    want = o.online_prefill(hd, 1, 0, st64, wl.bits(x.kv_score), wl.bits(x.ape), np.ascontiguousarray(wu),
                            o.OUT_COMPACT, nc)
    rows = (w[pick, 3] & 0xFFFFFF).astype(np.int64)
    got = out[: nc].cpu().numpy()[rows]
    kv_in = H.bf16_to_f32(wl.bits(x.kv_score)[:, :hd])
    # per channel, the largest |kv| of the group's tokens (earlier tokens from the prefix rows)
    pre_off = np.concatenate([[0], np.cumsum(x.prefix_lens.numpy())])
    kv_pre = H.bf16_to_f32(wl.bits(x.prefix_rows)[:, :hd])
    starts = np.concatenate([[0], np.cumsum(x.extend_lens.numpy())])
    kvmax = np.zeros((len(pick), hd), np.float32)
    for i, k in enumerate(pick):
        r0, cnt = w[k, 1] & 0xFFFFFF, w[k, 1] >> 24
        m = np.abs(kv_in[r0:r0 + cnt]).max(0)
        if (w[k, 3] >> 24) & 1:
            b = np.searchsorted(starts, r0, side="right") - 1
            m = np.maximum(m, np.abs(kv_pre[pre_off[b]:pre_off[b + 1]]).max(0))
        kvmax[i] = m
    H.assert_pool_close(got, want[rows], 0, kvmax, "online prefill, every emitted row")


@pytest.mark.slow
def test_full_size_online_decode(env):
    o, ckv, dev = env
    x = wl.c128_online_decode(0)
    hd = x.head_dim
    st64, st = _fold_prefix(o, ckv, dev, x, hd)
    status = ckv.new_status(dev)
    pd = ckv.plan_online_decode(x.rid.to(dev), x.seq_lens.to(dev), status=status)
    out = ckv.compress_online_decode(hd, st, x.kv_score.to(dev), x.ape.to(dev), pd, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    wpd = o.plan_online_decode(x.rid, x.seq_lens)
    assert (pd.cpu().numpy() == wpd).all()
    want = o.online_decode(hd, 1, 0, st64, wl.bits(x.kv_score), wl.bits(x.ape), wpd)
    got = out.cpu().numpy()
    bnd = np.nonzero((x.seq_lens.numpy() % 128) == 0)[0]
    assert (got[np.setdiff1d(np.arange(len(got)), bnd)].view(np.uint32) == 0).all()
    pre_off = np.concatenate([[0], np.cumsum(x.prefix_lens.numpy())])
    kv_pre = H.bf16_to_f32(wl.bits(x.prefix_rows)[:, :hd])
    kv_in = H.bf16_to_f32(wl.bits(x.kv_score)[:, :hd])
    kvmax = np.stack([np.maximum(np.abs(kv_in[b]), np.abs(kv_pre[pre_off[b]:pre_off[b + 1]]).max(0)) for b in bnd])
    H.assert_pool_close(got[bnd], want[bnd], 0, kvmax, "online decode boundary rows")


def test_online_empty_inputs(env):
    """Batch 0 and capacity 0: zero counts, nothing launched that touches the state."""
    o, ckv, dev = env
    i64 = dict(dtype=torch.int64, device=dev)
    e = torch.zeros(0, **i64)
    status = ckv.new_status(dev)
    units, counts = ckv.plan_online_prefill(e, e, e, 0, capacity_u=4, pad_invalid=True, status=status)
    torch.cuda.synchronize()
    assert counts[:2].tolist() == [0, 0] and int(status[0]) == 0
    assert (units.cpu().numpy() == 0xFF).all()
    state = torch.full((2, 3 * 128), 7.0, device=dev)
    kv = torch.zeros(1, 256, dtype=torch.bfloat16, device=dev)
    ape = torch.zeros(128, 128, dtype=torch.bfloat16, device=dev)
    ckv.compress_online_prefill(128, state, kv, ape, units, counts, ckv.OUT_COMPACT, out_rows=1, status=status)
    pd = ckv.plan_online_decode(e, e, status=status)
    assert pd.shape[0] == 0
    torch.cuda.synchronize()
    assert (state == 7.0).all() and int(status[0]) == 0
