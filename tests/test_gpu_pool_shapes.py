"""The prefill pools' launch shapes, each against the oracle on every record,
for every head_dim class and dtype pair.

C4 prefill pool:

The host picks the shape from what it knows before launch: the plan's
capacity and the token count.
  * staged, large geometry: more than eight full stages per SM
    (capacity > 8 * SMs * records per stage);
  * staged, small geometry (two CTAs per SM, half-size stages): the rest,
    unless the direct kernel takes the step;
  * direct (one thread per record and 16-byte chunk, one resident wave,
    4 blocks of 128 threads per SM at its register count): steps whose
    records, bounded by min(capacity, num_q_tokens / 4 + 768), fit 1.6
    waves.
The cases are sized from those rules with margin: "small" at ~2.5 waves of
the direct kernel, "direct2" at ~1.3 waves (some threads take a second
record), "large" just past the small geometry's limit.  The small cases of
test_gpu_parity.py all take the direct kernel.

C128 prefill pool: one persistent CTA per (SM, channel slice) takes records
first, first + stride, ... (stride = SMs / slices, or the capacity when that
is smaller) through its TMA ring.  "ring" gives every CTA at least two
records, "mixed" about half of the CTAs one and half two (the speculative-
decoding verify step's shape, where the producer's record requested with the
count and the consumers' record requested before the tile wait are the whole
chain); the small cases of test_gpu_parity.py give every CTA at most one.
"""
import numpy as np
import pytest
import torch

from tests.test_gpu_parity import DT, _run_prefill_parity

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

BATCH = 16


@pytest.fixture(scope="module")
def env(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_attention_compressplan_gb300 import build as B
    from compressed_kv_attention_compressplan_gb300 import ckv

    B.build()
    ckv.load_library()
    return oracle_mod, ckv, torch.device("cuda")


def _records_for(regime, hd, in_dt, sms):
    chunks = hd // (8 if in_dt == "bf16" else 4)   # 16-byte chunks of a record
    per_stage = 256 // chunks if chunks < 256 else 1
    wave = 4 * sms * 128                             # direct kernel threads resident at once
    if regime == "large":
        return 8 * sms * per_stage + 64
    if per_stage < 2:
        return None                                  # no small geometry at this width
    recs = int((2.5 if regime == "small" else 1.3) * wave / chunks)
    assert recs + BATCH <= 8 * sms * per_stage
    return recs


@pytest.mark.parametrize("regime", ["direct2", "small", "large"])
@pytest.mark.parametrize("hd", [128, 384, 512, 640, 1024])
@pytest.mark.parametrize("dts", [("bf16", "f32"), ("bf16", "bf16"), ("f32", "f32"), ("f32", "bf16")])
def test_c4_prefill_pool_shapes(env, regime, hd, dts):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    recs = _records_for(regime, hd, dts[0], sms)
    if recs is None:
        pytest.skip("one record fills a stage: only the large geometry exists at this width")
    nq = 4 * recs
    rng = np.random.default_rng(hd * 7 + len(regime) + 3 * DT[dts[0]] + DT[dts[1]])
    cuts = np.sort(rng.choice(np.arange(1, nq), BATCH - 1, replace=False))
    el = np.diff(np.concatenate([[0], cuts, [nq]]))
    pl = rng.integers(0, 1000, BATCH)
    layout = (hd // 128 + len(regime) + DT[dts[1]]) % 2
    _run_prefill_parity(env, 4, hd, DT[dts[0]], DT[dts[1]], layout, list(pl), list(el), seed=hd + len(regime))


@pytest.mark.parametrize("regime", ["ring", "mixed"])
@pytest.mark.parametrize("hd", [128, 384, 512, 1024])
@pytest.mark.parametrize("dts", [("bf16", "f32"), ("bf16", "bf16"), ("f32", "f32"), ("f32", "bf16")])
def test_c128_prefill_pool_shapes(env, regime, hd, dts):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    slices = hd // (128 if dts[0] == "bf16" else 64)
    stride = sms // slices
    want = 3 * stride if regime == "ring" else stride + stride // 2
    rng = np.random.default_rng(hd * 5 + len(regime) + 3 * DT[dts[0]] + DT[dts[1]])
    pl = rng.integers(1, 4096, BATCH)                     # most first windows start in the state
    per = -(-want // BATCH)
    el = 128 * per - pl % 128 + rng.integers(0, 128, BATCH)
    o = env[0]
    _, _, (nc, _), _ = o.plan_prefill(128, np.arange(BATCH), pl + el, el)
    assert nc >= (2 * stride if regime == "ring" else stride + 1), nc
    if regime == "mixed":
        assert nc < 2 * stride, nc
    layout = (hd // 128 + len(regime) + DT[dts[1]]) % 2
    _run_prefill_parity(env, 128, hd, DT[dts[0]], DT[dts[1]], layout, list(pl), list(el), seed=hd + len(regime),
                        outliers=0.01)
