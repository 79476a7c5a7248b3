"""The test helpers that the GPU parity tests lean on, checked on the CPU: the
vectorised per-channel window max|kv| (the tolerance reference of every pooled
row) equals its one-entry-at-a-time statement on oracle plans of both ratios,
both dtypes, windows that start in the state and C4 first groups."""
import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H


@pytest.mark.parametrize("ratio", [4, 128])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_window_kv_absmax_matches_loop(oracle_mod, ratio, dt):
    o = oracle_mod
    rng = np.random.default_rng(ratio)
    pl = list(rng.integers(0, 3 * ratio, 7)) + [0, ratio - 1]
    el = list(rng.integers(1, 3 * ratio + 9, 7)) + [ratio, 2]
    w = wl.random_prefill(ratio, 128, dt, torch.float32, wl.COMPACT, pl, el, seed=ratio, num_requests_state=12)
    wc, _, (nc, _), _ = o.plan_prefill(ratio, w.rid, w.seq_lens, w.extend_lens)
    f = H.plan_c_fields(wc)
    assert (f["buffer_len"] > 0).any() and nc > 10
    if ratio == 4:
        assert (f["seq_len"] == 4).any()
    args = (ratio, 128, wl.bits(w.state), wl.bits(w.kv_score), f["seq_len"], f["ragged_id"], f["buffer_len"],
            f["read_page_0"], f["read_page_1"])
    want = H.window_kv_absmax_loop(*args)
    for chunk in (1, 5, 64):
        assert np.array_equal(H.window_kv_absmax(*args, chunk=chunk), want)
