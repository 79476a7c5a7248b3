"""Bounded waits that expire leave the context usable.

The pooling kernels that stage their inputs through the TMA engine (C4 and
C128 prefill pools, the persistent C128 decode, the online prefill) wait on
mbarriers for their copies with a time limit.  Here the limit is set to 1 ns
(ckv_set_wait_limit_ns), so that those waits expire while copies are still in
flight -- a wait that expires on its own, with no fault and nothing left
hanging.  Each launch must then report CKV_STATUS_TIMEOUT and finish (every
CTA waits for the copies it issued before it exits), and the context must stay
usable: the same launch with the default limit afterwards gives results
bit-identical to one made before the expired run.
"""
import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TIMEOUT = 16  # CKV_STATUS_TIMEOUT


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_attention_compressplan_gb300 import build as B
    from compressed_kv_attention_compressplan_gb300 import ckv

    B.build()
    ckv.load_library()
    ckv.set_wait_limit_ns(0)
    yield ckv, torch.device("cuda")
    ckv.set_wait_limit_ns(0)


def _split(rng, total, parts):
    cuts = np.sort(rng.choice(np.arange(1, total), parts - 1, replace=False))
    return np.diff(np.concatenate([[0], cuts, [total]])).astype(np.int64)


def _expire_then_recover(ckv, run):
    """run() -> (tensors to compare, status tensor); it resets whatever it mutates."""
    before, status = run()
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    before = [t.clone() for t in before]
    ckv.set_wait_limit_ns(1)
    try:
        _, status = run()
        torch.cuda.synchronize()  # the launch finished: no CTA was left waiting
        expired = int(status[0])
    finally:
        ckv.set_wait_limit_ns(0)
    assert expired & TIMEOUT, f"status {expired:#x}: no wait expired at a 1 ns limit"
    after, status = run()
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    for x, y in zip(before, after):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), "results differ after the expired run"


@pytest.mark.parametrize("ratio", [4, 128])
def test_prefill_pool_wait_expiry(env, ratio):
    ckv, dev = env
    hd, batch = 512, 16
    nq = 16384 if ratio == 4 else 65536
    rng = np.random.default_rng(7 + ratio)
    el = _split(rng, nq, batch)
    pl = rng.integers(0, 1000, batch)
    layout = wl.TOKEN if ratio == 4 else wl.COMPACT
    lay = ckv.OUT_TOKEN if ratio == 4 else ckv.OUT_COMPACT
    w = wl.random_prefill(ratio, hd, torch.bfloat16, torch.float32, layout, pl, el, seed=11 + ratio,
                          num_requests_state=batch + 2)
    rid, sl, ext = w.rid.to(dev), w.seq_lens.to(dev), w.extend_lens.to(dev)
    kv, state, ape = w.kv_score.to(dev), w.state.to(dev), w.ape.to(dev)
    plan_c, _, counts = ckv.plan_prefill(ratio, rid, sl, ext, nq)
    status = ckv.new_status(dev)
    out = torch.empty(nq if ratio == 4 else plan_c.shape[0], hd, dtype=torch.float32, device=dev)

    def run():
        status.zero_()
        out.fill_(float("nan"))
        ckv.compress_pool_prefill(ratio, hd, state, kv, ape, plan_c, counts, lay, out=out, status=status)
        return [out], status

    _expire_then_recover(ckv, run)


@pytest.mark.parametrize("ordered", [True, False])
def test_c128_decode_wait_expiry(env, ordered):
    ckv, dev = env
    hd, batch = 512, 512
    rng = np.random.default_rng(21)
    sl = rng.integers(1, 32768, batch)
    sl[rng.permutation(batch)[: batch // 4]] = 128 * rng.integers(1, 256, batch // 4)  # page boundaries
    w = wl.random_decode(128, hd, torch.bfloat16, torch.float32, sl, seed=22, num_requests_state=batch + 5)
    init = w.state.to(dev)
    state = init.clone()
    kv, ape, rid, seq = w.kv_score.to(dev), w.ape.to(dev), w.rid.to(dev), w.seq_lens.to(dev)
    status = ckv.new_status(dev)

    def run():
        status.zero_()
        state.copy_(init)
        if ordered:
            out, _ = ckv.decode_step(128, hd, state, kv, ape, rid, seq, torch.float32, status=status)
        else:
            pd = ckv.plan_decode(128, rid, seq, status=status)
            out = ckv.compress_decode(128, hd, state, kv, ape, pd, torch.float32, status=status)
        return [out, state], status

    _expire_then_recover(ckv, run)


def test_online_prefill_wait_expiry(env):
    ckv, dev = env
    hd, batch, nq = 512, 16, 16384
    rng = np.random.default_rng(31)
    g = torch.Generator().manual_seed(32)
    slots = batch + 3
    init = torch.randn(slots, 3 * hd, generator=g)
    init[:, hd:2 * hd] = 1.0 + init[:, hd:2 * hd].abs()  # weight sums are >= 1
    init = init.to(dev)
    state = init.clone()
    ape = (torch.randn(128, hd, generator=g) * 0.5).to(torch.bfloat16).to(dev)
    el = _split(rng, nq, batch)
    pl = rng.integers(0, 400, batch)
    rid = torch.from_numpy(rng.permutation(slots)[:batch].astype(np.int64)).to(dev)
    sl, ext = torch.from_numpy(pl + el).to(dev), torch.from_numpy(el).to(dev)
    kv = torch.randn(nq, 2 * hd, generator=g).to(torch.bfloat16).to(dev)
    units, counts = ckv.plan_online_prefill(rid, sl, ext, nq)
    status = ckv.new_status(dev)
    out = torch.empty(ckv.capacity_compress(128, batch, nq), hd, dtype=torch.float32, device=dev)

    def run():
        status.zero_()
        state.copy_(init)
        out.fill_(float("nan"))
        ckv.compress_online_prefill(hd, state, kv, ape, units, counts, ckv.OUT_COMPACT, out=out, status=status)
        return [out, state], status

    _expire_then_recover(ckv, run)
