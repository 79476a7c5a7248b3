"""Pins of the oracle's norm + RoPE + store step (compressor_v2.py
compress_norm_rope_store: RMSNorm, RoPE at position seq_len - ratio, store at
out_loc).

Anchors outside the oracle: a constant row normalises to the weight; float64
torch (rms_norm and complex multiplication) on random rows; the rotation keeps
every pair's length and depends only on relative positions; a worked case in
which only position seq_len - ratio rotates by a quarter turn; zero rows for
non-boundary decode rows and nothing stored for invalid records.
"""
import numpy as np
import pytest
import torch

from tests import helpers as H

HD, ROPE = 512, 64


def textbook_freqs(max_pos: int, rope_dim: int, base: float = 10000.0) -> np.ndarray:
    """cos / sin of pos * base^(-2i/rope_dim), rounded to fp32: [max_pos, rope_dim/2, 2]."""
    inv = base ** (-np.arange(0, rope_dim, 2, dtype=np.float64) / rope_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)


def identity_freqs(max_pos: int, rope_dim: int) -> np.ndarray:
    f = np.zeros((max_pos, rope_dim // 2, 2), np.float32)
    f[..., 0] = 1.0
    return f


def decode_plan(seq_lens) -> np.ndarray:
    """DecodePlan records carrying only seq_len (the step reads nothing else)."""
    p = np.zeros((len(seq_lens), 4), np.uint32)
    p[:, 0] = seq_lens
    return p.view(np.uint8).reshape(-1, 16)


def compress_plan(seq_lens, ragged) -> np.ndarray:
    p = np.zeros((len(seq_lens), 4), np.uint32)
    p[:, 0] = seq_lens
    p[:, 1] = ragged
    return p.view(np.uint8).reshape(-1, 16)


def run(o, rows, plan, weight, eps, freqs, out_loc, ratio=4, mode=1, layout=1, cache_rows=16, cache_dt=0,
        in_dt=0, hd=HD, rope=ROPE):
    cache = np.full((cache_rows, hd), np.nan, np.float32) if cache_dt == 0 else \
        np.full((cache_rows, hd), 0x7FC0, np.uint16)
    o.norm_rope_store(ratio, mode, hd, rope, in_dt, rows, layout, plan, weight, eps, freqs, out_loc, cache_dt, cache)
    return cache


def test_constant_row_normalises_to_the_weight(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(0)
    w = rng.standard_normal(HD).astype(np.float32)
    rows = np.full((1, HD), 2.0, np.float32)
    cache = run(o, rows, decode_plan([8]), w, 1e-30, identity_freqs(8, ROPE), [3])
    assert (cache[3] == w).all()


def test_eps_sits_inside_the_root(oracle_mod):
    """A constant row c with eps comparable to c^2: every channel becomes
    c * w / sqrt(c^2 + eps) (the RMSNorm definition), which for c = 1e-3 and
    eps = 1e-6 is w / sqrt(2), far from w / (1 + 1e-3) (eps outside the root)
    and from w (eps dropped)."""
    o = oracle_mod
    rng = np.random.default_rng(3)
    w = (1 + 0.1 * rng.standard_normal(HD)).astype(np.float32)
    rows = np.full((1, HD), 1e-3, np.float32)
    cache = run(o, rows, decode_plan([8]), w, 1e-6, identity_freqs(8, ROPE), [5])
    c = np.float64(np.float32(1e-3))
    want = c * w.astype(np.float64) / np.sqrt(c * c + np.float64(np.float32(1e-6)))
    assert np.abs(cache[5].astype(np.float64) - want).max() <= 4 * np.finfo(np.float32).eps * np.abs(want).max()


@pytest.mark.parametrize("mode", [0, 1])
def test_matches_float64_torch(oracle_mod, mode):
    o = oracle_mod
    rng = np.random.default_rng(1 + mode)
    n, R = 6, 128
    rows = rng.standard_normal((n, HD)).astype(np.float32) * 3
    w = (1 + 0.1 * rng.standard_normal(HD)).astype(np.float32)
    eps = 1e-6
    freqs = textbook_freqs(2048, ROPE)
    sl = (rng.integers(1, 15, n) * R).astype(np.int64)
    loc = rng.permutation(16)[:n]
    if mode == 1:
        plan, out_loc, order = decode_plan(sl), loc, np.arange(n)
    else:
        ragged = np.arange(n) * 3 + 1
        plan = compress_plan(sl, ragged)
        out_loc = np.zeros(3 * n + 1, np.int64)
        out_loc[ragged] = loc
        order = np.arange(n)
    cache = run(o, rows, plan, w, eps, freqs, out_loc, ratio=R, mode=mode)
    x = torch.from_numpy(rows.astype(np.float64))
    y = torch.nn.functional.rms_norm(x, (HD,), torch.from_numpy(w.astype(np.float64)), eps)
    f = torch.from_numpy(freqs.astype(np.float64))[torch.from_numpy(sl - R)]
    rot = torch.view_as_complex(f.contiguous())
    pe = torch.view_as_complex(y[:, HD - ROPE:].reshape(n, ROPE // 2, 2).contiguous()) * rot
    want = torch.cat([y[:, :HD - ROPE], torch.view_as_real(pe).reshape(n, ROPE)], dim=1).numpy()
    got = cache[loc[order]].astype(np.float64)
    assert np.abs(got - want).max() <= 2 * np.finfo(np.float32).eps * np.abs(want).max()


def test_rotation_keeps_pair_lengths_and_relative_positions(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(3)
    w = np.ones(HD, np.float32)
    q = rng.standard_normal((1, HD)).astype(np.float32)
    k = rng.standard_normal((1, HD)).astype(np.float32)
    R = 4
    freqs = textbook_freqs(4096, ROPE)
    plain = run(o, np.concatenate([q, k]), decode_plan([R, R]), w, 1e-6, identity_freqs(4096, ROPE), [0, 1])
    pairs = lambda r: r[HD - ROPE:].astype(np.float64).reshape(-1, 2)

    def rope_dot(m, n):
        c = run(o, np.concatenate([q, k]), decode_plan([m + R, n + R]), w, 1e-6, freqs, [0, 1])
        lq, lk = np.linalg.norm(pairs(c[0]), axis=1), np.linalg.norm(pairs(c[1]), axis=1)
        np.testing.assert_allclose(lq, np.linalg.norm(pairs(plain[0]), axis=1), rtol=1e-6)
        np.testing.assert_allclose(lk, np.linalg.norm(pairs(plain[1]), axis=1), rtol=1e-6)
        assert (c[0][:HD - ROPE] == plain[0][:HD - ROPE]).all()
        return float(pairs(c[0]).ravel() @ pairs(c[1]).ravel())

    scale = float(np.abs(pairs(plain[0])).sum() * np.abs(pairs(plain[1])).max())
    for m, n, s in [(8, 4, 100), (1000, 16, 4), (12, 12, 2000)]:  # boundary rows only
        assert abs(rope_dot(m, n) - rope_dot(m + s, n + s)) <= 1e-5 * scale


def test_position_is_seq_len_minus_ratio(oracle_mod):
    """Only position seq_len - ratio turns by a quarter: (a, b) -> (-b, a) on the
    last rope_dim channels; the first HD - rope_dim channels are the norm alone."""
    o = oracle_mod
    rng = np.random.default_rng(4)
    w = np.ones(HD, np.float32)
    rows = rng.standard_normal((1, HD)).astype(np.float32)
    for ratio, sl in [(4, 8), (128, 256)]:
        freqs = identity_freqs(300, ROPE)
        freqs[sl - ratio] = [0.0, 1.0]
        ref = run(o, rows, decode_plan([sl]), w, 1e-6, identity_freqs(300, ROPE), [0], ratio=ratio)[0]
        got = run(o, rows, decode_plan([sl]), w, 1e-6, freqs, [0], ratio=ratio)[0]
        a, b = ref[HD - ROPE::2], ref[HD - ROPE + 1::2]
        assert (got[HD - ROPE::2] == -b).all() and (got[HD - ROPE + 1::2] == a).all()
        assert (got[:HD - ROPE] == ref[:HD - ROPE]).all()
        # prefill, compact layout: the same record through a CompressPlan
        out_loc = np.zeros(10, np.int64)
        out_loc[7] = 2
        gp = run(o, rows, compress_plan([sl], [7]), w, 1e-6, freqs, out_loc, ratio=ratio, mode=0)[2]
        assert (gp == got).all()


def test_decode_zero_rows_and_invalid_records(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(5)
    rows = rng.standard_normal((3, HD)).astype(np.float32)
    plan = decode_plan([9, 12, 0])
    plan[2] = 0xFF  # invalid record
    cache = run(o, rows, plan, np.ones(HD, np.float32), 1e-6, textbook_freqs(64, ROPE), [4, 5, 6])
    assert (cache[4] == 0).all()  # seq_len 9: not a boundary -> a zero row (signs from the rotation)
    assert np.isfinite(cache[5]).all() and np.abs(cache[5]).max() > 0
    assert np.isnan(cache[6]).all()  # untouched


def test_bf16_cache_is_the_rounded_fp32_result(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(6)
    rows = (rng.standard_normal((2, HD)) * 5).astype(np.float32)
    w = rng.standard_normal(HD).astype(np.float32)
    args = (rows, decode_plan([8, 12]), w, 1e-6, textbook_freqs(64, ROPE), [0, 1])
    c32 = run(o, *args)
    c16 = run(o, *args, cache_dt=1)
    # the oracle rounds its double result once; rounding the fp32 result (RNE, written out) lands on the same
    # bf16 value or, at a near-tie, on its neighbour
    b = c32.view(np.uint32).astype(np.uint64)
    rne = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    d = H.ulp_distance(c16, rne)
    assert d.max() <= 1 and (d == 0).mean() > 0.99


def test_bad_locations_are_errors(oracle_mod):
    o = oracle_mod
    rows = np.ones((1, HD), np.float32)
    with pytest.raises(o.OracleError):
        run(o, rows, decode_plan([8]), np.ones(HD, np.float32), 1e-6, identity_freqs(8, ROPE), [16])
    with pytest.raises(o.OracleError):  # position beyond the table
        run(o, rows, decode_plan([400]), np.ones(HD, np.float32), 1e-6, identity_freqs(8, ROPE), [1])
    with pytest.raises(o.OracleError):  # eps must be positive (a zero row would give 0 / 0)
        run(o, rows, decode_plan([8]), np.ones(HD, np.float32), 0.0, identity_freqs(8, ROPE), [1])
