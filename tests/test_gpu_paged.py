"""GPU parity of the SWA-paged planners (ckv_plan_prefill_paged /
ckv_plan_decode_paged) against the oracle, and of whole schedules that run
through paged plans over a randomly allocated SWA pool.

Bar: plans bit-exact; pooled rows of a paged schedule bitwise equal to the
same rows of a legacy one-shot prefill on the GPU (the same windows), and
within the parity bar of the oracle's whole-history definition.
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


def _pool_for(rng, B, sl, S, prefix_hits=True):
    """A pool with every request mapped up to its seq_len; some requests reuse
    another's first pages (prefix-cache hits)."""
    num_reqs = B + 3
    stride = max(sl) + 5
    pages = sum(s // S + 2 for s in sl) + 8
    pool = H.SwaPagedPool(num_reqs, stride, S, pages, rng)
    rids = [int(x) for x in rng.permutation(num_reqs)[:B]]
    for b in range(B):
        if prefix_hits and b > 0 and rng.random() < 0.3:
            a = int(rng.integers(0, b))
            n = (min(sl[a], sl[b]) // S) * S
            if n > 0:
                pool.share(rids[b], rids[a], n)
        pool.ensure(rids[b], sl[b])
    return pool, rids


CASES = {
    "small": dict(B=5, max_sl=200, S=16, ring=8),
    "many": dict(B=300, max_sl=90, S=32, ring=16),
    "long": dict(B=3, max_sl=6000, S=256, ring=64),
}


@pytest.mark.parametrize("ratio", [4, 128])
@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("pad", [False, True])
def test_paged_prefill_plans_bit_exact(env, ratio, case, pad):
    o, ckv, dev = env
    c = CASES[case]
    rng = np.random.default_rng(len(case) * 7 + ratio + pad)
    B, S = c["B"], c["S"]
    ring = c["ring"] if ratio == 4 else 128
    sl = [int(rng.integers(1, c["max_sl"] + 1)) for _ in range(B)]
    el = [int(rng.integers(1, s + 1)) if rng.random() < 0.7 else s for s in sl]
    pool, rids = _pool_for(rng, B, sl, S)
    nq = int(sum(el))
    r2t = torch.from_numpy(pool.r2t).to(dev) if ratio == 4 else None
    f2s = torch.from_numpy(pool.f2s).to(dev) if ratio == 4 else None
    i64 = dict(dtype=torch.int64, device=dev)
    cap_c = nq if pad else ckv.capacity_compress(ratio, B, nq)
    cap_w = nq if pad else ckv.capacity_write_paged(ratio, B, nq, S)
    status = ckv.new_status(dev)
    pc, pw, counts = ckv.plan_prefill_paged(ratio, torch.tensor(rids, **i64), r2t, f2s, S, ring,
                                            torch.tensor(sl, **i64), torch.tensor(el, **i64), nq, cap_c, cap_w,
                                            pad_invalid=pad, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    wc, ww, (nc, nw), _ = o.plan_prefill_paged(ratio, rids, pool.r2t if ratio == 4 else None,
                                               pool.f2s if ratio == 4 else None, S, ring, sl, el, nq, cap_c, cap_w,
                                               pad_invalid=pad)
    assert counts[:2].tolist() == [nc, nw]
    assert nw <= cap_w and nc <= cap_c
    n_c, n_w = (cap_c, cap_w) if pad else (nc, nw)
    assert (pc[:n_c].cpu().numpy() == wc[:n_c]).all(), "compress plan"
    assert (pw[:n_w].cpu().numpy() == ww[:n_w]).all(), "write plan"


@pytest.mark.parametrize("ratio", [4, 128])
def test_paged_decode_plan_bit_exact(env, ratio):
    o, ckv, dev = env
    rng = np.random.default_rng(11 + ratio)
    B, S = 700, 64
    ring = 16 if ratio == 4 else 128
    sl = [int(rng.integers(1, 400)) for _ in range(B)]
    pool, rids = _pool_for(rng, B, sl, S)
    i64 = dict(dtype=torch.int64, device=dev)
    status = ckv.new_status(dev)
    maps = (torch.from_numpy(pool.r2t).to(dev), torch.from_numpy(pool.f2s).to(dev)) if ratio == 4 else (None, None)
    pd = ckv.plan_decode_paged(ratio, torch.tensor(rids, **i64), *maps, S, ring, torch.tensor(sl, **i64),
                               status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    omaps = (pool.r2t, pool.f2s) if ratio == 4 else (None, None)
    want = o.plan_decode_paged(ratio, rids, *omaps, S, ring, sl)
    assert (pd.cpu().numpy() == want).all()
    order = ckv.new_decode_order(B, dev)
    pd = ckv.plan_decode_paged(ratio, torch.tensor(rids, **i64), *maps, S, ring, torch.tensor(sl, **i64),
                               status=status, order=order)
    assert (pd.cpu().numpy() == want).all()
    assert (H.decode_order_entries(order) == H.expected_decode_order(want, ratio)).all()


def test_paged_bad_mapping_is_flagged(env):
    o, ckv, dev = env
    i64 = dict(dtype=torch.int64, device=dev)
    r2t = torch.arange(40, dtype=torch.int32, device=dev)[None, :].contiguous()
    f2s = torch.arange(40, dtype=torch.int64, device=dev)
    f2s[37] = -1  # a written position
    status = ckv.new_status(dev)
    ckv.plan_prefill_paged(4, torch.tensor([0], **i64), r2t, f2s, 16, 8, torch.tensor([40], **i64),
                           torch.tensor([40], **i64), 40, status=status)
    ckv.plan_decode_paged(4, torch.tensor([0], **i64), r2t, f2s, 16, 8, torch.tensor([38], **i64), status=status)
    torch.cuda.synchronize()
    assert int(status[0]) & ckv.STATUS_BAD_INDEX
    status.zero_()
    r2t[0, 3] = 1 << 20  # out of the full pool; the first window reads position 3
    ckv.plan_prefill_paged(4, torch.tensor([0], **i64), r2t, torch.arange(40, **i64), 16, 8,
                           torch.tensor([40], **i64), torch.tensor([34], **i64), 34, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) & ckv.STATUS_BAD_INDEX
    with pytest.raises(ckv.CkvError):  # C128 state needs a 128-row ring
        ckv.plan_decode_paged(128, torch.tensor([0], **i64), None, None, 256, 256, torch.tensor([38], **i64),
                              status=status)


def test_paged_schedule_matches_one_shot(env):
    """Chunked prefills, decode steps and prefix-cache hits through paged plans
    give, on the GPU, bitwise the rows of a legacy one-shot prefill of the same
    histories, and the oracle's whole-history rows within the parity bar."""
    o, ckv, dev = env
    ratio, hd, S, ring = 4, 512, 16, 8
    rng = np.random.default_rng(21)
    width = wl.width_of(ratio, hd)
    g = torch.Generator().manual_seed(21)
    ape = wl.bits((torch.randn(8, hd, generator=g) * 0.1).to(torch.bfloat16)).copy()
    lens = [int(rng.integers(40, 120)) for _ in range(5)]
    hist = [wl.bits(torch.randn(n, width, generator=g).to(torch.bfloat16)).copy() for n in lens]
    pool = H.SwaPagedPool(num_reqs=10, stride=200, swa_page_size=S, num_swa_pages=80, rng=rng)
    state = wl.sentinel((80 * ring, width), torch.bfloat16).to(dev)
    paged = H.PagedGpuBackend(pool, ring, dev)
    rids = [4, 0, 7, 2, 9]
    sched = [H.split_schedule(n, rng, 11, 0.35) for n in lens]
    got = H.run_schedule(paged, ratio, hd, 1, 0, hist, rids, sched, ape, state)
    assert int(paged.status[0]) == 0
    shared = [S * (lens[0] // S), S * 2]
    new_rids = [1, 3]
    for a, n, r in zip([0, 1], shared, new_rids):
        pool.share(r, rids[a], n)
    tails = [23, 37]
    hist2 = [np.concatenate([hist[a][:n], wl.bits(torch.randn(t, width, generator=g).to(torch.bfloat16))])
             for a, n, t in zip([0, 1], shared, tails)]
    sched2 = [H.split_schedule(t, rng, 9, 0.4) for t in tails]
    got2 = H.run_schedule(paged, ratio, hd, 1, 0, hist2, new_rids, sched2, ape, state, start=shared)
    assert int(paged.status[0]) == 0
    # the same histories in one legacy prefill each
    legacy = H.GpuBackend(dev)
    all_hist = hist + hist2
    lstate = wl.sentinel((8 * 8, width), torch.bfloat16).to(dev)
    ref = H.run_schedule(legacy, ratio, hd, 1, 0, all_hist, list(range(7)), [[("prefill", len(h))] for h in all_hist],
                         ape, lstate)
    outs = got + [x for x in got2]
    starts = [0] * 5 + shared
    for b, h in enumerate(all_hist):
        n0 = starts[b]
        assert (outs[b][n0:].view(np.uint32) == ref[b][n0:].view(np.uint32)).all(), b
        want = o.compress_history(ratio, hd, 1, 0, h, ape)
        emit = [p for p in range(n0, len(h)) if (p + 1) % ratio == 0]
        seq = np.array(emit) + 1
        kvmax = H.window_kv_absmax(ratio, hd, h, h, seq, np.array(emit), np.zeros(len(emit), np.int64),
                                   np.zeros(len(emit)), np.zeros(len(emit)))
        H.assert_pool_close(outs[b][emit], want[emit], 0, kvmax, f"history b={b}")


@pytest.mark.parametrize("case", range(30))
def test_paged_plans_random(env, case):
    """Seeded random SWA-paged steps: page size 16 .. 256, ring 8 .. 64 rows, up to 200 requests with
    prefix-cache hits, equal or mixed extends, padded or not; prefill and decode plans bit-exact."""
    o, ckv, dev = env
    rng = np.random.default_rng(90000 + case)
    ratio = int(rng.choice([4, 128]))
    S = int(rng.choice([16, 32, 64, 128, 256]))
    ring = int(rng.choice([r for r in (8, 16, 32, 64) if S % r == 0])) if ratio == 4 else 128
    B = int(rng.integers(1, 201))
    max_sl = int(rng.choice([40, 300, 3000]))
    sl = [int(rng.integers(1, max_sl + 1)) for _ in range(B)]
    if rng.random() < 0.3:  # equal extends
        e = int(rng.integers(1, 9))
        sl = [max(s, e) for s in sl]
        el = [e] * B
    else:
        el = [int(rng.integers(1, s + 1)) if rng.random() < 0.7 else s for s in sl]
    pad = bool(rng.integers(2))
    pool, rids = _pool_for(rng, B, sl, S, prefix_hits=bool(rng.integers(2)))
    nq = int(sum(el))
    i64 = dict(dtype=torch.int64, device=dev)
    maps = (torch.from_numpy(pool.r2t).to(dev), torch.from_numpy(pool.f2s).to(dev)) if ratio == 4 else (None, None)
    omaps = (pool.r2t, pool.f2s) if ratio == 4 else (None, None)
    cap_c = nq if pad else ckv.capacity_compress(ratio, B, nq)
    cap_w = nq if pad else ckv.capacity_write_paged(ratio, B, nq, S)
    status = ckv.new_status(dev)
    pc, pw, counts = ckv.plan_prefill_paged(ratio, torch.tensor(rids, **i64), *maps, S, ring, torch.tensor(sl, **i64),
                                            torch.tensor(el, **i64), nq, cap_c, cap_w, pad_invalid=pad,
                                            status=status)
    pd = ckv.plan_decode_paged(ratio, torch.tensor(rids, **i64), *maps, S, ring, torch.tensor(sl, **i64),
                               status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    wc, ww, (nc, nw), _ = o.plan_prefill_paged(ratio, rids, *omaps, S, ring, sl, el, nq, cap_c, cap_w,
                                               pad_invalid=pad)
    assert counts[:2].tolist() == [nc, nw]
    n_c, n_w = (cap_c, cap_w) if pad else (nc, nw)
    assert (pc[:n_c].cpu().numpy() == wc[:n_c]).all(), "compress plan"
    assert (pw[:n_w].cpu().numpy() == ww[:n_w]).all(), "write plan"
    assert (pd.cpu().numpy() == o.plan_decode_paged(ratio, rids, *omaps, S, ring, sl)).all(), "decode plan"
