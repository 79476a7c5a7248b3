"""Pins of the oracle's SWA-paged planners (c_plan.cuh plan_compress_prefill /
plan_compress_decode with their kernel_1 / decode-kernel translation).

Two independent anchors:
  * an identity SWA mapping whose pages never end inside the sequences must
    give back the legacy plans (themselves pinned by brute force and by the
    worked examples), except that compress records that read no state keep
    (-1, batch index) as kernel_1 leaves them;
  * chunked prefills, decode steps and prefix-cache hits at SWA page
    boundaries, all through paged plans over a randomly allocated SWA pool,
    must give exactly the rows of the stateless whole-history definition.  A
    missing page-end write, a wrong ring offset or a wrong read page makes a
    window read a NaN sentinel or another page's row.
"""
import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H


def _identity_maps(num_reqs, S):
    """r2t[rid][p] = a permuted full slot f with f2s[f] = rid * S + p, p < S:
    with S a multiple of 8 and an 8-row ring, position p of request rid lands on
    row rid * 8 + p % 8, the legacy two pages of the request."""
    rng = np.random.default_rng(5)
    perm = rng.permutation(num_reqs * S)
    r2t = perm.reshape(num_reqs, S).astype(np.int32)
    f2s = np.full(num_reqs * S, -1, np.int64)
    f2s[perm] = np.arange(num_reqs * S)
    return r2t, f2s


@pytest.mark.parametrize("ratio", [4, 128])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_identity_mapping_gives_legacy_plans(oracle_mod, ratio, seed):
    o = oracle_mod
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 7))
    num_reqs = 9
    rids = [int(x) for x in rng.permutation(num_reqs)[:B]]
    sl = [int(rng.integers(1, 3 * ratio + 40)) for _ in range(B)]
    el = [int(rng.integers(1, s + 1)) for s in sl]
    if ratio == 4:
        ring = 8
        S = ((max(sl) + 4) // ring + 1) * ring  # no SWA page ends inside the sequences
        r2t, f2s = _identity_maps(num_reqs, S)
    else:
        ring, S, r2t, f2s = 128, 128, None, None
    lc, lw, (nc, nw), _ = o.plan_prefill(ratio, rids, sl, el)
    pc, pw, (mc, mw), _ = o.plan_prefill_paged(ratio, rids, r2t, f2s, S, ring, sl, el)
    assert (mc, mw) == (nc, nw)
    assert (pw == lw).all(), "write records"
    fl, fp = H.plan_c_fields(lc), H.plan_c_fields(pc)
    for k in ("seq_len", "ragged_id", "buffer_len"):
        assert (fl[k] == fp[k]).all(), k
    reads = fl["buffer_len"] > 0
    assert (fp["read_page_0"][reads] == fl["read_page_0"][reads]).all()
    assert (fp["read_page_1"][reads] == fl["read_page_1"][reads]).all()
    # records without state reads: (-1, index of the request in the batch)
    starts = np.concatenate([[0], np.cumsum(el)])
    batch_of = np.searchsorted(starts, fp["ragged_id"], side="right") - 1
    assert (fp["read_page_0"][~reads] == -1).all()
    assert (fp["read_page_1"][~reads] == batch_of[~reads]).all()
    # decode plans: identical
    dsl = [int(rng.integers(1, S + 1)) for _ in range(B)]
    assert (o.plan_decode_paged(ratio, rids, r2t, f2s, S, ring, dsl) == o.plan_decode(ratio, rids, dsl)).all()


def test_page_end_positions_are_written_before_first_write(oracle_mod):
    """A worked case: SWA pages of 16 tokens, one 40-token prefill.  Legacy
    writes 36..39; the paged plan also writes the page ends 12..15 and 28..31,
    in position order, at rows (page * ring + offset)."""
    o = oracle_mod
    S, ring, L = 16, 8, 40
    r2t = np.arange(L, dtype=np.int32)[None, :]
    pages = [5, 2, 7]  # SWA page of positions 0..15, 16..31, 32..39
    f2s = np.array([pages[p // S] * S + p % S for p in range(L)], np.int64)
    _, pw, (_, nw), _ = o.plan_prefill_paged(4, [0], r2t, f2s, S, ring, [L], [L])
    f = H.plan_w_fields(pw)
    want_pos = [12, 13, 14, 15, 28, 29, 30, 31, 36, 37, 38, 39]
    assert nw == len(want_pos)
    assert f["ragged_id"].tolist() == want_pos
    assert f["write_loc"].tolist() == [pages[p // S] * ring + p % ring for p in want_pos]


@pytest.mark.parametrize("seed", [0, 1])
def test_paged_schedules_equal_history(oracle_mod, seed):
    o = oracle_mod
    ratio, hd = 4, 128
    S, ring = 16, 8
    rng = np.random.default_rng(300 + seed)
    in_dt, out_dt = (0, 0) if seed == 0 else (1, 1)
    tdt = torch.bfloat16 if in_dt else torch.float32
    width = wl.width_of(ratio, hd)
    g = torch.Generator().manual_seed(60 + seed)
    ape = wl.bits((torch.randn(H.window(ratio), hd, generator=g) * 0.1).to(tdt)).copy()
    # requests 0..3 from scratch; 4 and 5 reuse the first pages of 0 and 1
    lens = [int(rng.integers(35, 90)) for _ in range(4)]
    hist = [wl.bits(torch.randn(n, width, generator=g).to(tdt)).copy() for n in lens]
    num_pages = 64
    pool = H.SwaPagedPool(num_reqs=8, stride=160, swa_page_size=S, num_swa_pages=num_pages, rng=rng)
    state = wl.bits(wl.sentinel((num_pages * ring, width), tdt)).copy()
    backend = H.PagedOracleBackend(o, pool, ring)
    rids = [3, 0, 6, 1]
    sched = [H.split_schedule(n, rng, 13, 0.3) for n in lens]
    got = H.run_schedule(backend, ratio, hd, in_dt, out_dt, hist, rids, sched, ape, state)
    for b in range(4):
        want = o.compress_history(ratio, hd, in_dt, out_dt, hist[b], ape)
        assert (got[b].view(np.uint8) == want.view(np.uint8)).all(), ("from scratch", b)
    # prefix-cache hits at page boundaries: the first window after the shared
    # pages reads the owner's page-end rows
    shared = [S * (lens[0] // S), S * min(2, lens[1] // S)]
    new_rids = [2, 5]
    for (a, n), r in zip(zip([0, 1], shared), new_rids):
        pool.share(r, rids[a], n)
    tails = [int(rng.integers(5, 40)) for _ in range(2)]
    hist2 = [np.concatenate([hist[a][:n], wl.bits(torch.randn(t, width, generator=g).to(tdt))])
             for a, n, t in zip([0, 1], shared, tails)]
    sched2 = [H.split_schedule(t, rng, 9, 0.4) for t in tails]
    got2 = H.run_schedule(backend, ratio, hd, in_dt, out_dt, hist2, new_rids, sched2, ape, state, start=shared)
    for k in range(2):
        want = o.compress_history(ratio, hd, in_dt, out_dt, hist2[k], ape)
        n = shared[k]
        assert (got2[k][n:].view(np.uint8) == want[n:].view(np.uint8)).all(), ("prefix hit", k)


def test_paged_bad_mapping_is_an_error(oracle_mod):
    o = oracle_mod
    r2t = np.arange(12, dtype=np.int32)[None, :]
    f2s = np.arange(12, dtype=np.int64)
    f2s[7] = -1  # position 7 is neither written nor read through the map: no error
    o.plan_prefill_paged(4, [0], r2t, f2s, 16, 8, [12], [12])
    f2s[9] = -1  # position 9 is written
    with pytest.raises(o.OracleError):
        o.plan_prefill_paged(4, [0], r2t, f2s, 16, 8, [12], [12])
    with pytest.raises(o.OracleError):  # seq_len beyond the map's stride
        o.plan_decode_paged(4, [0], r2t, f2s, 16, 8, [13])
    with pytest.raises(o.OracleError):  # C128 state needs a 128-row ring
        o.plan_prefill_paged(128, [0], None, None, 256, 256, [12], [12])
