"""The benchmark's byte accounting against the oracle's plans.

bench.py derives each launch's algorithmic bytes -- the numerator of every
roofline fraction it reports -- from closed forms of the per-request loops:
per compress record its buffer_len and masked entries, the compress and write
record counts, and for a decode the rows on a group or page boundary.  Here
those closed forms are checked against the records the oracle emits for the
same lengths: seeded length mixes with the edge cases (a first C4 group, a
prefix on a boundary, one-token extends) and the benchmark workloads' own
lengths.  Only lengths are drawn; no kernel runs.
"""
import numpy as np
import pytest

import bench
from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H


def _check_prefill(o, ratio, sl, el):
    sl = np.asarray(sl, np.int64)
    el = np.asarray(el, np.int64)
    bl, first, nc, nw = bench.prefill_events(ratio, sl, el)
    rid = np.arange(len(sl), dtype=np.int64)
    pc, _, (onc, onw), _ = o.plan_prefill(ratio, rid, sl, el)
    assert (nc, nw) == (onc, onw), "record counts"
    f = H.plan_c_fields(pc[:onc])
    assert (np.asarray(bl) == f["buffer_len"]).all(), "buffer_len per record"
    # the C4 window of the first group (seq_len 4) has no previous group: 4 masked entries
    assert (np.asarray(first) == np.where((ratio == 4) & (f["seq_len"] == 4), 4, 0)).all(), "masked entries"
    return nc


@pytest.mark.parametrize("ratio", [4, 128])
def test_prefill_events_match_oracle_plans(oracle_mod, ratio):
    rng = np.random.default_rng(ratio)
    span = 3 * ratio if ratio == 128 else 40
    total = 0
    for case in range(40):
        batch = int(rng.integers(1, 30))
        pl = rng.integers(0, span, batch)
        el = rng.integers(1, span, batch)
        if batch >= 4:
            pl[0], el[0] = 0, 4              # exactly the first group (C4: masked window)
            pl[1] = ratio * int(rng.integers(0, 3))  # a prefix that ends on a boundary
            el[2] = 1                         # a one-token extend
            pl[3] = 0
        total += _check_prefill(oracle_mod, ratio, pl + el, el)
    assert total > 0


@pytest.mark.parametrize("name", ["c4_prefill", "c128_prefill", "c4_prefill_mtp", "c128_prefill_mtp"])
def test_prefill_events_on_benchmark_lengths(oracle_mod, name):
    if name == "c4_prefill":
        _, sl, el = wl.c4_prefill_lengths(0)
        ratio = 4
    elif name == "c128_prefill":
        _, sl, el = wl.c128_prefill_lengths(0)
        ratio = 128
    else:  # the verify step: 1024 requests extend by 4 from a prefix U[0, 65536]
        import torch

        ratio = 4 if name.startswith("c4") else 128
        el = torch.full((1024,), 4, dtype=torch.int64)
        pl = torch.randint(0, 65537, (1024,), generator=torch.Generator().manual_seed(3), dtype=torch.int64)
        sl = pl + el
    nc = _check_prefill(oracle_mod, ratio, sl.numpy(), el.numpy())
    assert nc > 0


@pytest.mark.parametrize("ratio", [4, 128])
def test_decode_bytes_from_oracle_plans(oracle_mod, ratio):
    """bench's decode bytes against a per-row sum over the oracle's decode plan:
    every row reads its token row and record and writes the row into the state
    and one output row; a boundary row also reads its window's other entries
    (W - 1, minus the 4 masked ones of a first C4 group); ape is read once."""
    import torch

    hd = 128
    rng = np.random.default_rng(10 + ratio)
    sl = rng.integers(1, 4000, 300)
    sl[:40] = ratio * rng.integers(1, 20, 40)
    sl[40] = 4  # C4: the first group
    w = wl.random_decode(ratio, hd, torch.bfloat16, torch.float32, sl, seed=5, num_requests_state=300)
    got = bench.algorithmic_bytes(w)
    f = H.plan_d_fields(oracle_mod.plan_decode(ratio, w.rid.numpy(), w.seq_lens.numpy()))
    W = 8 if ratio == 4 else 128
    row = (4 if ratio == 4 else 2) * hd * 2     # bf16 kv_score row
    entry = 2 * hd * 2                          # kv + score of one window entry
    want = 0
    for s in f["seq_len"]:
        want += 2 * row + hd * 4 + 16
        if s % ratio == 0:
            want += (W - 1 - (4 if ratio == 4 and s == 4 else 0)) * entry
    want += W * hd * 2
    assert got["decode"] == want
    assert got["rows"] == int((f["seq_len"] % ratio == 0).sum())


def test_clock_sampler_summary():
    """The clocks summary of the JSON line (median SM clock, max clock, throttle
    reasons seen), parsed from nvidia-smi's CSV rows; the scratch file is removed."""
    import os

    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.path = os.path.join(bench.tempfile.gettempdir(), f"ckv_clocks_test_{os.getpid()}.csv")
    with open(c.path, "w") as f:
        f.write("2070, 2070, 900.1, Not Active, Not Active, Not Active, Active\n"
                "1995, 2070, 1000.0, Not Active, Not Active, Not Active, Not Active\n"
                "2070, 2070, 1010.5, Not Active, Active, Not Active, Not Active\n"
                "[N/A], 2070, 0, Not Active, Not Active, Not Active, Not Active\n")

    class Proc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    c.f = open(os.devnull, "w")
    c.proc = Proc()
    got = c.stop()
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["hw_thermal_slowdown", "sw_power_cap"],
                   "samples": 3}
    assert not os.path.exists(c.path)
