"""GPU parity of ckv_norm_rope_store_prefill / _decode against the oracle.

Bar: fp32 cache rows within E = (head_dim + 8) * 2^-24 * max|y| of the
oracle's double result per row (the fp32 sum of squares over head_dim terms
dominates the error); bf16 cache rows within 1 ulp, except where a value is so
much smaller than its row (cancellation in a rotated pair) that E alone exceeds
a bf16 ulp of it -- there E applies to the bf16 values; cache rows no record
names are left untouched, byte for byte.
"""
import numpy as np
import pytest
import torch

from compressed_kv_attention_compressplan_gb300 import workloads as wl
from tests import helpers as H
from tests.test_oracle_norm_rope import textbook_freqs

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


def _sentinel_cache(rows, hd, code):
    if code == 1:
        return np.full((rows, hd), 0x7FC1, np.uint16)
    return np.full((rows, hd), np.nan, np.float32)


def assert_bf16_close(got: np.ndarray, want: np.ndarray, hd: int, what: str):
    d = H.ulp_distance(got, want)
    g, w = H.bf16_to_f32(got).astype(np.float64), H.bf16_to_f32(want).astype(np.float64)
    e_row = (hd + 8) * 2.0 ** -24 * np.abs(w).max(axis=1, keepdims=True)
    bad = (d > 1) & (np.abs(g - w) > e_row)
    assert not bad.any(), f"{what}: {bad.sum()} bf16 values off by > 1 ulp and > E; max ulp {d.max()}"


def _compare(got: np.ndarray, want: np.ndarray, code: int, rows, hd, what):
    if code == 1:
        assert_bf16_close(got[rows], want[rows], hd, what)
    else:
        g, w = got[rows].astype(np.float64), want[rows].astype(np.float64)
        bound = (hd + 8) * 2.0 ** -24 * np.abs(w).max(axis=1, keepdims=True)
        assert (np.abs(g - w) <= bound).all(), f"{what}: {np.abs(g - w).max()}"
    others = np.setdiff1d(np.arange(got.shape[0]), rows)
    assert (got[others].view(np.uint8) == want[others].view(np.uint8)).all(), f"{what}: untouched rows"


def _rows(rng, n, hd, code):
    x = torch.from_numpy((rng.standard_normal((n, hd)) * rng.uniform(0.1, 20, (n, 1))).astype(np.float32))
    return wl.bits(x.to(torch.bfloat16 if code else torch.float32)).copy()


@pytest.mark.parametrize("ratio", [4, 128])
@pytest.mark.parametrize("in_code,cache_code", [(0, 1), (0, 0), (1, 1)])
@pytest.mark.parametrize("hd,rope", [(512, 64), (128, 64), (1024, 0)])
def test_decode_parity(env, ratio, in_code, cache_code, hd, rope):
    o, ckv, dev = env
    rng = np.random.default_rng(ratio + 10 * in_code + cache_code + hd)
    B = 300
    sl = rng.integers(1, 4000, B)
    on = rng.random(B) < 0.4
    sl[on] = ratio * rng.integers(1, 4000 // ratio, int(on.sum()))
    plan = o.plan_decode(ratio, np.arange(B), sl)
    plan[rng.random(B) < 0.05] = 0xFF  # a few padding records
    rows = _rows(rng, B, hd, in_code)
    w = (1 + 0.2 * rng.standard_normal(hd)).astype(np.float32)
    freqs = textbook_freqs(4096, rope) if rope else np.zeros((1, 0, 2), np.float32)
    cache_rows = B + 50
    loc = rng.permutation(cache_rows)[:B]
    want = _sentinel_cache(cache_rows, hd, cache_code)
    o.norm_rope_store(ratio, 1, hd, rope, in_code, rows, 1, plan, w, 1e-6, freqs, loc, cache_code, want)
    cache = H.to_torch(_sentinel_cache(cache_rows, hd, cache_code), cache_code).to(dev)
    status = ckv.new_status(dev)
    ckv.norm_rope_store_decode(ratio, H.to_torch(rows, in_code).to(dev), torch.from_numpy(plan).to(dev),
                               torch.from_numpy(w).to(dev), 1e-6, torch.from_numpy(freqs).to(dev),
                               torch.from_numpy(loc.astype(np.int64)).to(dev), cache, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    valid = H.plan_d_fields(plan)["seq_len"] != 0xFFFFFFFF
    _compare(H.np_bits(cache), want, cache_code, loc[valid], hd, "decode")


@pytest.mark.parametrize("ratio,layout", [(4, 0), (128, 1), (4, 1)])
def test_prefill_parity(env, ratio, layout):
    o, ckv, dev = env
    rng = np.random.default_rng(7 + ratio + layout)
    hd, rope = 512, 64
    B = 40
    pl = rng.integers(0, 3000, B)
    el = rng.integers(1, 700, B)
    sl = pl + el
    nq = int(el.sum())
    pc, _, (nc, _), _ = o.plan_prefill(ratio, np.arange(B), sl, el)
    nrows = nq if layout == 0 else nc
    rows = _rows(rng, nrows, hd, 0)
    w = (1 + 0.2 * rng.standard_normal(hd)).astype(np.float32)
    freqs = textbook_freqs(int(sl.max()) + 1, rope)
    cache_rows = nq + 7
    out_loc = rng.permutation(cache_rows)[:nq].astype(np.int64)
    want = _sentinel_cache(cache_rows, hd, 1)
    o.norm_rope_store(ratio, 0, hd, rope, 0, rows, layout, pc[:nc], w, 1e-5, freqs, out_loc, 1, want)
    cap = nc + 5  # device count below the capacity: the tail is not read
    pcd = torch.full((cap, 16), 0xFF, dtype=torch.uint8, device=dev)
    pcd[:nc] = torch.from_numpy(pc[:nc]).to(dev)
    counts = torch.tensor([nc, 0, 0, 0], dtype=torch.int32, device=dev)
    cache = H.to_torch(_sentinel_cache(cache_rows, hd, 1), 1).to(dev)
    status = ckv.new_status(dev)
    ckv.norm_rope_store_prefill(ratio, H.to_torch(rows, 0).to(dev), pcd, counts, torch.from_numpy(w).to(dev), 1e-5,
                                torch.from_numpy(freqs).to(dev), torch.from_numpy(out_loc).to(dev), cache,
                                in_layout=layout, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    stored = out_loc[H.plan_c_fields(pc[:nc])["ragged_id"]]
    _compare(H.np_bits(cache), want, 1, stored, hd, "prefill")


@pytest.mark.parametrize("case", range(20))
def test_random_norm_rope(env, case):
    """Seeded random cases of both entry points: head_dim 128 .. 1024 (every
    kChunks instance), rope_dim any multiple of 4 up to head_dim, row and cache
    dtypes, ratio, layout; against the oracle with the same bar."""
    o, ckv, dev = env
    rng = np.random.default_rng(60000 + case)
    ratio = int(rng.choice([4, 128]))
    hd = 128 * int(rng.integers(1, 9))
    rope = 4 * int(rng.integers(0, hd // 4 + 1))
    in_code, cache_code = int(rng.integers(2)), int(rng.integers(2))
    eps = float(rng.choice([1e-6, 1e-5, 1e-3]))
    w = (1 + 0.2 * rng.standard_normal(hd)).astype(np.float32)
    if rng.integers(2):  # decode
        B = int(rng.integers(1, 400))
        sl = rng.integers(1, 3000, B)
        on = rng.random(B) < 0.5
        sl[on] = ratio * rng.integers(1, max(2, 3000 // ratio), int(on.sum()))
        plan = o.plan_decode(ratio, np.arange(B), sl)
        rows = _rows(rng, B, hd, in_code)
        freqs = textbook_freqs(3000 + ratio, rope) if rope else np.zeros((1, 0, 2), np.float32)
        cache_rows = B + 20
        loc = rng.permutation(cache_rows)[:B].astype(np.int64)
        want = _sentinel_cache(cache_rows, hd, cache_code)
        o.norm_rope_store(ratio, 1, hd, rope, in_code, rows, 1, plan, w, eps, freqs, loc, cache_code, want)
        cache = H.to_torch(_sentinel_cache(cache_rows, hd, cache_code), cache_code).to(dev)
        status = ckv.new_status(dev)
        ckv.norm_rope_store_decode(ratio, H.to_torch(rows, in_code).to(dev), torch.from_numpy(plan).to(dev),
                                   torch.from_numpy(w).to(dev), eps, torch.from_numpy(freqs).to(dev),
                                   torch.from_numpy(loc).to(dev), cache, status=status)
        stored = loc
    else:  # prefill
        layout = int(rng.integers(2))
        B = int(rng.integers(1, 30))
        pl = rng.integers(0, 2000, B)
        el = rng.integers(1, 600, B)
        sl = pl + el
        nq = int(el.sum())
        pc, _, (nc, _), _ = o.plan_prefill(ratio, np.arange(B), sl, el)
        rows = _rows(rng, nq if layout == 0 else max(nc, 1), hd, in_code)
        freqs = textbook_freqs(int(sl.max()) + 1, rope) if rope else np.zeros((1, 0, 2), np.float32)
        cache_rows = nq + 5
        loc = rng.permutation(cache_rows)[:nq].astype(np.int64)
        want = _sentinel_cache(cache_rows, hd, cache_code)
        o.norm_rope_store(ratio, 0, hd, rope, in_code, rows, layout, pc[:nc], w, eps, freqs, loc, cache_code, want)
        cache = H.to_torch(_sentinel_cache(cache_rows, hd, cache_code), cache_code).to(dev)
        status = ckv.new_status(dev)
        pcd = torch.from_numpy(np.ascontiguousarray(pc[:max(nc, 1)])).to(dev)
        counts = torch.tensor([nc, 0, 0, 0], dtype=torch.int32, device=dev)
        ckv.norm_rope_store_prefill(ratio, H.to_torch(rows, in_code).to(dev), pcd, counts,
                                    torch.from_numpy(w).to(dev), eps, torch.from_numpy(freqs).to(dev),
                                    torch.from_numpy(loc).to(dev), cache, in_layout=layout, status=status)
        stored = loc[H.plan_c_fields(pc[:nc])["ragged_id"]]
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    _compare(H.np_bits(cache), want, cache_code, stored, hd, f"random case {case}")


def test_errors_and_bad_records(env):
    o, ckv, dev = env
    hd = 512
    rows = torch.ones(2, hd, device=dev)
    w = torch.ones(hd, device=dev)
    freqs = torch.from_numpy(textbook_freqs(16, 64)).to(dev)
    cache = torch.zeros(4, hd, dtype=torch.bfloat16, device=dev)
    plan = torch.from_numpy(o.plan_decode(4, np.arange(2), np.array([8, 400]))).to(dev)
    loc = torch.tensor([1, 2], dtype=torch.int64, device=dev)
    with pytest.raises(ckv.CkvError):
        ckv.norm_rope_store_decode(4, rows, plan, w, 0.0, freqs, loc, cache)
    with pytest.raises(ckv.CkvError):
        ckv.norm_rope_store_decode(4, rows, plan, w, 1e-6, freqs[:, :15].contiguous(), loc, cache)  # rope_dim 30
    status = ckv.new_status(dev)
    ckv.norm_rope_store_decode(4, rows, plan, w, 1e-6, freqs, loc, cache, status=status)  # position 396 > table
    torch.cuda.synchronize()
    assert int(status[0]) & ckv.STATUS_BAD_INDEX
    assert (cache[2] == 0).all() and (cache[1] != 0).any()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["norm_rope_c128_prefill", "norm_rope_c128_decode"])
def test_full_size_inputs(env, name):
    """The benchmark's norm + RoPE + store inputs (the C128 workloads' record
    counts and positions; fp32 rows into a bf16 cache), every stored row checked,
    with the plan built on the GPU as the benchmark builds it."""
    o, ckv, dev = env
    x = wl.NORM_ROPE[name](0)
    hd, R = x.head_dim, x.ratio
    status = ckv.new_status(dev)
    rows_d = x.rows.to(dev)
    cache = torch.full((x.cache_rows, hd), float("nan"), dtype=torch.bfloat16, device=dev)
    if x.extend_lens is not None:
        nq = int(x.extend_lens.sum())
        pc, _, counts = ckv.plan_prefill(R, x.rid.to(dev), x.seq_lens.to(dev), x.extend_lens.to(dev), nq,
                                         status=status)
        ckv.norm_rope_store_prefill(R, rows_d, pc, counts, x.weight.to(dev), x.eps, x.freqs.to(dev),
                                    x.out_loc.to(dev), cache, in_layout=ckv.OUT_COMPACT, status=status)
        torch.cuda.synchronize()
        wc, _, (nc, _), _ = o.plan_prefill(R, x.rid, x.seq_lens, x.extend_lens)
        assert int(counts[0]) == nc and (pc[:nc].cpu().numpy() == wc).all()
        plan, mode, stored = wc, 0, x.out_loc.numpy()[H.plan_c_fields(wc)["ragged_id"]]
    else:
        pd = ckv.plan_decode(R, x.rid.to(dev), x.seq_lens.to(dev), status=status)
        ckv.norm_rope_store_decode(R, rows_d, pd, x.weight.to(dev), x.eps, x.freqs.to(dev), x.out_loc.to(dev),
                                   cache, status=status)
        torch.cuda.synchronize()
        plan, mode, stored = o.plan_decode(R, x.rid, x.seq_lens), 1, x.out_loc.numpy()
    assert int(status[0]) == 0
    want = np.full((x.cache_rows, hd), 0x7FC0, np.uint16)  # torch's bf16 NaN
    o.norm_rope_store(R, mode, hd, x.rope_dim, 0, wl.bits(x.rows), 1, plan, wl.bits(x.weight), x.eps,
                      wl.bits(x.freqs), x.out_loc.numpy(), 1, want)
    got = H.np_bits(cache)
    assert_bf16_close(got[stored], want[stored], hd, name)
    untouched = np.ones(x.cache_rows, bool)
    untouched[stored] = False
    assert (got[untouched] == want[untouched]).all()


def test_no_records(env):
    o, ckv, dev = env
    hd = 256
    cache = torch.full((3, hd), 5.0, device=dev)
    rows = torch.ones(4, hd, device=dev)
    plan_c = torch.full((4, 16), 0xFF, dtype=torch.uint8, device=dev)  # all invalid
    counts = torch.tensor([0, 0, 0, 0], dtype=torch.int32, device=dev)
    status = ckv.new_status(dev)
    freqs = torch.from_numpy(textbook_freqs(8, 64)).to(dev)
    w = torch.ones(hd, device=dev)
    loc = torch.zeros(4, dtype=torch.int64, device=dev)
    ckv.norm_rope_store_prefill(4, rows, plan_c, counts, w, 1e-6, freqs, loc, cache, status=status)
    ckv.norm_rope_store_prefill(4, rows, plan_c, None, w, 1e-6, freqs, loc, cache, status=status)
    torch.cuda.synchronize()
    assert (cache == 5.0).all() and int(status[0]) == 0


@pytest.mark.parametrize("hd,rope", [(512, 64), (128, 64), (384, 32), (1024, 0)])
@pytest.mark.parametrize("in_code,cache_code", [(1, 1), (1, 0), (0, 1)])
@pytest.mark.parametrize("hinted", [False, True])
def test_fused_c4_decode_norm_rope_store(env, hd, rope, in_code, cache_code, hinted):
    """ckv_compress_decode_norm_rope_store against the same step in two
    launches (decode with fp32 rows, then norm + RoPE + store on them): the
    state bytes equal, every stored cache row within the norm step's bar (the
    RMS's fp32 sum runs in another order), rows of invalid records untouched;
    and the two-launch rows against the oracle."""
    o, ckv, dev = env
    rng = np.random.default_rng(hd + rope + 10 * in_code + cache_code + (5 if hinted else 0))
    B = 257
    sl = rng.integers(1, 3000, B)
    on = rng.random(B) < 0.4
    sl[on] = 4 * rng.integers(1, 750, int(on.sum()))
    sl[:3] = [4, 8, 3]  # the first group (masked previous group), the second, none
    w = wl.random_decode(4, hd, H.torch_dtype(in_code), torch.float32, sl, seed=hd + 3, num_requests_state=B + 7)
    plan = o.plan_decode(4, w.rid, w.seq_lens)
    plan[rng.random(B) < 0.04] = 0xFF  # a few padding records
    weight = (1 + 0.2 * rng.standard_normal(hd)).astype(np.float32)
    freqs = textbook_freqs(4096, rope) if rope else np.zeros((1, 0, 2), np.float32)
    cache_rows = B + 40
    loc = rng.permutation(cache_rows)[:B].astype(np.int64)
    pd = torch.from_numpy(plan).to(dev)
    args = dict(norm_weight=torch.from_numpy(weight).to(dev), eps=1e-6, freqs=torch.from_numpy(freqs).to(dev),
                out_loc=torch.from_numpy(loc).to(dev))
    kv, ape = w.kv_score.to(dev), w.ape.to(dev)
    # two launches
    st2 = w.state.to(dev)
    cache2 = H.to_torch(_sentinel_cache(cache_rows, hd, cache_code), cache_code).to(dev)
    status = ckv.new_status(dev)
    rows = ckv.compress_decode(4, hd, st2, kv, ape, pd, torch.float32, status=status)
    ckv.norm_rope_store_decode(4, rows, pd, args["norm_weight"], args["eps"], args["freqs"], args["out_loc"], cache2,
                               status=status)
    # one launch
    st1 = w.state.to(dev)
    cache1 = H.to_torch(_sentinel_cache(cache_rows, hd, cache_code), cache_code).to(dev)
    hints = {"rid_hint": w.rid.to(dev), "seq_lens_hint": w.seq_lens.to(dev)} if hinted else {}
    ckv.compress_decode_norm_rope_store(hd, st1, kv, ape, pd, kv_cache=cache1, status=status, **args, **hints)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    assert (H.np_bits(st1).view(np.uint8) == H.np_bits(st2).view(np.uint8)).all(), "state"
    valid = H.plan_d_fields(plan)["seq_len"] != 0xFFFFFFFF
    _compare(H.np_bits(cache1), H.np_bits(cache2), cache_code, loc[valid], hd, "fused against two launches")
    # the two-launch rows against the oracle (decode with fp32 rows, then norm + RoPE + store)
    st = wl.bits(w.state).copy()
    pooled = o.compress_decode(4, hd, in_code, 0, st, wl.bits(w.kv_score), wl.bits(w.ape), plan)
    want = _sentinel_cache(cache_rows, hd, cache_code)
    o.norm_rope_store(4, 1, hd, rope, 0, H.np_bits(rows).copy(), 1, plan, weight, 1e-6, freqs, loc, cache_code, want)
    _compare(H.np_bits(cache2), want, cache_code, loc[valid], hd, "two launches against the oracle")
    f = H.plan_d_fields(plan)
    bnd = np.nonzero(valid & (f["seq_len"] % 4 == 0))[0]
    kvmax = H.window_kv_absmax(4, hd, wl.bits(w.state), wl.bits(w.kv_score), f["seq_len"][bnd], bnd,
                               np.full(len(bnd), 7), f["read_page_0"][bnd], f["read_page_1"][bnd])
    H.assert_pool_close(H.np_bits(rows)[bnd], pooled[bnd], 0, kvmax, "decode rows")


def test_fused_c4_decode_norm_rope_store_bad_records(env):
    """A location outside the cache or a position outside the table is flagged
    and stores nothing; a record that writes outside the state is flagged and
    stores the normalised zero row; the other rows are stored."""
    o, ckv, dev = env
    hd, B = 256, 40
    w = wl.random_decode(4, hd, torch.bfloat16, torch.float32, 4 * np.arange(1, B + 1), seed=8, num_requests_state=B)
    plan = o.plan_decode(4, w.rid, w.seq_lens)
    plan.view(np.int32).reshape(B, 4)[7, 1] = 2 ** 30  # row 7 writes outside the state
    pd = torch.from_numpy(plan).to(dev)
    loc = torch.arange(B, dtype=torch.int64, device=dev)
    loc[5] = 10 ** 6
    cache = torch.full((B, hd), float("nan"), device=dev)
    status = ckv.new_status(dev)
    freqs = torch.from_numpy(textbook_freqs(100, 64)).to(dev)  # rows with seq_len - 4 >= 100 fall outside
    ckv.compress_decode_norm_rope_store(hd, w.state.to(dev), w.kv_score.to(dev), w.ape.to(dev), pd,
                                        torch.ones(hd, device=dev), 1e-6, freqs, loc, cache, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) & ckv.STATUS_BAD_INDEX
    stored = torch.isfinite(cache).all(dim=1).cpu().numpy()
    want = np.array([b != 5 and 4 * (b + 1) - 4 < 100 for b in range(B)])
    assert (stored == want).all()
    assert (cache[7] == 0).all()  # no state written, the normalised zero row stored
