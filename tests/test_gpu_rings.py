"""Mid-size cases in which every persistent CTA of the staged pools streams at
least ten tiles through its shared-memory ring, so every stage is reused, every
mbarrier phase flips several times, and the producers' records fetched a group
(a unit) ahead are used; every record is compared with the oracle.

Ring shapes (bf16 input): the C4 prefill pool stages 256 / (hd / 8) records per
stage in a 3-stage ring over min(groups, SMs) CTAs; the C128 prefill pool gives
each CTA one 128-channel slice and every (SMs / slices)-th record of it; the
online prefill streams each unit's tokens 7 per stage through a 2-stage ring,
persistent over units.
"""
import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H
from tests.test_gpu_online import _fold_prefix
from tests.test_gpu_parity import _run_prefill_parity

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


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _lengths(rng, batch, lo, hi, max_prefix):
    pl = rng.integers(0, max_prefix + 1, batch)
    el = rng.integers(lo, hi + 1, batch)
    return pl, el


@pytest.mark.parametrize("hd", [128, 512])
def test_c4_prefill_pool_laps_its_ring(env, hd):
    rng = np.random.default_rng(40 + hd)
    recs = 256 // (hd // 8)                       # records per stage (bf16)
    batch = 24 if hd == 512 else 48
    lo, hi = (900, 1300) if hd == 512 else (1900, 2300)
    pl, el = _lengths(rng, batch, lo, hi, 4096)
    o = env[0]
    _, _, (nc, _), _ = o.plan_prefill(4, np.arange(batch), pl + el, el)
    groups = -(-nc // recs)
    assert groups / min(groups, _sms()) >= 10, "each CTA must stream >= 10 stages"
    _run_prefill_parity(env, 4, hd, 1, 1, 0, list(pl), list(el), seed=hd)


@pytest.mark.parametrize("hd", [128, 512])
def test_c128_prefill_pool_laps_its_ring(env, hd):
    rng = np.random.default_rng(50 + hd)
    batch = 24 if hd == 512 else 64
    lo, hi = (2000, 2600) if hd == 512 else (3000, 3400)
    pl, el = _lengths(rng, batch, lo, hi, 4096)   # most windows start in the state
    o = env[0]
    _, _, (nc, _), _ = o.plan_prefill(128, np.arange(batch), pl + el, el)
    per_slice = min(_sms() // (hd // 128), nc)
    assert nc / per_slice >= 10, "each CTA must stream >= 10 tiles"
    _run_prefill_parity(env, 128, hd, 1, 0, 1, list(pl), list(el), seed=hd, outliers=0.01)


@pytest.mark.parametrize("hd", [128, 512])
def test_online_prefill_laps_its_ring(env, hd):
    """Every emitted row of ~3.5k units (several units per CTA, each of up to
    19 stages) against the oracle folding the same units."""
    o, ckv, dev = env
    rng = np.random.default_rng(60 + hd)
    batch = 1024
    pl = rng.integers(0, 4096, batch)
    el = rng.integers(150, 450, batch)
    rid = torch.from_numpy(rng.permutation(batch)).to(torch.int64)
    sl, elt = torch.from_numpy(pl + el).to(torch.int64), torch.from_numpy(el).to(torch.int64)
    x = wl.c128_online_prefill(hd, head_dim=hd, lengths=(rid, sl, elt))
    st64, st = _fold_prefix(o, ckv, dev, x, hd)
    nq = int(el.sum())
    status = ckv.new_status(dev)
    units, counts = ckv.plan_online_prefill(x.rid.to(dev), x.seq_lens.to(dev), x.extend_lens.to(dev), nq,
                                            status=status)
    cap_c = ckv.capacity_compress(128, batch, nq)
    out = ckv.compress_online_prefill(hd, st, x.kv_score.to(dev), x.ape.to(dev), units, counts, ckv.OUT_COMPACT,
                                      out_rows=cap_c, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    wu, (nu, nc), _ = o.plan_online_prefill(x.rid, x.seq_lens, x.extend_lens)
    assert counts[:2].tolist() == [nc, nu] and (units[:nu].cpu().numpy() == wu).all()
    assert nu >= 3 * 5 * _sms(), "several units per CTA (up to 5 CTAs per SM)"
    want = o.online_prefill(hd, 1, 0, st64, wl.bits(x.kv_score), wl.bits(x.ape), wu, o.OUT_COMPACT, nc)
    w = wu.view(np.uint32).reshape(-1, 4)
    emitting = np.nonzero((w[:, 3] >> 24) & 2)[0]
    rows = (w[emitting, 3] & 0xFFFFFF).astype(np.int64)
    got = out[:nc].cpu().numpy()[rows]
    kv_in = H.bf16_to_f32(wl.bits(x.kv_score)[:, :hd])
    pre_off = np.concatenate([[0], np.cumsum(x.prefix_lens.numpy())])
    kv_pre = H.bf16_to_f32(wl.bits(x.prefix_rows)[:, :hd])
    starts = np.concatenate([[0], np.cumsum(x.extend_lens.numpy())])
    kvmax = np.zeros((len(emitting), hd), np.float32)
    for i, k in enumerate(emitting):
        r0, cnt = w[k, 1] & 0xFFFFFF, w[k, 1] >> 24
        m = np.abs(kv_in[r0:r0 + cnt]).max(0)
        if (w[k, 3] >> 24) & 1:
            b = np.searchsorted(starts, r0, side="right") - 1
            m = np.maximum(m, np.abs(kv_pre[pre_off[b]:pre_off[b + 1]]).max(0))
        kvmax[i] = m
    H.assert_pool_close(got, want[rows], 0, kvmax, "online prefill, every emitted row")
