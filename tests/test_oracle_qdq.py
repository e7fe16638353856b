"""Pins for the oracle's fp32 fake QDQ (E4M3 and INT8), independent of the oracle's own code.

What the pages fix ("[1/4] GDN state/W QAT foundation", "What does this PR do?"
and "Usage": dynamic E4M3; "[2/4] GDN/KDA decode QAT with INT8 recurrent
state", "What does this PR do?": INT8 codes in [-127, 127], zero point zero,
nearest-even rounding; "Testing": rounded reciprocal multiplication), checked
against the E4M3 format definition, torch's float8_e4m3fn conversion, brute
force search, and invariants.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _table():
    codes = np.arange(256, dtype=np.uint8)
    return codes, oracle.e4m3_decode(codes)


def test_e4m3_decode_known_values():
    # values from the E4M3FN bit layout: exponent bias 7, 3 mantissa bits
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x39: 1.125, 0x40: 2.0, 0x77: 240.0, 0x78: 256.0, 0x7E: 448.0, 0xB8: -1.0,
             0xFE: -448.0}
    for c, val in known.items():
        assert oracle.e4m3_decode(np.array([c], np.uint8))[0] == np.float32(val), hex(c)
    assert math.isnan(oracle.e4m3_decode(np.array([0x7F], np.uint8))[0])
    assert math.isnan(oracle.e4m3_decode(np.array([0xFF], np.uint8))[0])
    neg0 = oracle.e4m3_decode(np.array([0x80], np.uint8))[0]
    assert neg0 == 0 and math.copysign(1.0, neg0) < 0


def test_e4m3_decode_matches_torch_float8():
    codes, vals = _table()
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(vals))
    assert np.array_equal(ref[~nan].view(np.uint32), vals[~nan].view(np.uint32))


def test_e4m3_all_codes_round_trip_and_monotone():
    codes, vals = _table()
    ok = ~np.isnan(vals)
    assert np.array_equal(oracle.e4m3_encode(vals[ok]), codes[ok])
    pos = vals[:0x7F]
    assert np.all(np.diff(pos) > 0)
    assert ok.sum() == 254


def _brute_nearest(u):
    """Nearest E4M3 code by search over the sorted grid; ties to the even code; saturate."""
    codes, vals = _table()
    grid = vals[:0x7F].astype(np.float64)        # 0 .. 448, increasing
    gcode = codes[:0x7F]
    a = np.abs(u.astype(np.float64))
    hi = np.clip(np.searchsorted(grid, a, side="left"), 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    dlo = np.abs(a - grid[lo])
    dhi = np.abs(grid[hi] - a)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (gcode[hi] % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(a >= 448.0, len(grid) - 1, idx)
    c = gcode[idx]
    return np.where(np.signbit(u), c | 0x80, c).astype(np.uint8)


def test_e4m3_encode_brute_force_random():
    rng = np.random.default_rng(1)
    n = 2_000_000
    mags = np.exp2(rng.uniform(-14, 9.5, n)).astype(np.float32)
    u = (mags * np.where(rng.random(n) < 0.5, -1, 1)).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(u), _brute_nearest(u))


def test_e4m3_encode_exact_ties_go_to_even():
    codes, vals = _table()
    grid = vals[:0x7F].astype(np.float64)
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)   # exact in fp32
    got = oracle.e4m3_encode(mids)
    assert np.all(got % 2 == 0)
    assert np.array_equal(got, _brute_nearest(mids))
    # saturation: beyond 448 (including the 464 midpoint and inf) stays +-448
    big = np.array([448.0, 460.0, 464.0, 470.0, 1e6, np.inf, -500.0], np.float32)
    assert list(oracle.e4m3_encode(big)) == [0x7E] * 6 + [0xFE]


def test_e4m3_encode_in_range_matches_torch_float8():
    rng = np.random.default_rng(2)
    u = (rng.standard_normal(500_000) * 60).astype(np.float32)
    u = u[np.abs(u) <= 448]
    ref = torch.from_numpy(u).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(u), ref)


def test_int8_encode_nearest_even_and_clamp():
    rng = np.random.default_rng(3)
    u = (rng.standard_normal(200_000) * 80).astype(np.float32)
    ties = np.arange(-130, 130).astype(np.float32) + np.float32(0.5)
    u = np.concatenate([u, ties, np.array([127.4, 127.5, 200, -127.6, -1e9], np.float32)])
    c = oracle.int8_encode(u).astype(np.float64)
    uc = np.clip(u.astype(np.float64), -127, 127)
    assert np.all(np.abs(c - uc) <= 0.5)
    tie = np.abs(np.abs(uc - np.trunc(uc)) - 0.5) == 0
    assert np.all(c[tie] % 2 == 0)
    assert c.min() >= -127 and c.max() <= 127


@pytest.mark.parametrize("mode,M", [("e4m3", 448.0), ("int8", 127.0)])
def test_group_amax_maps_to_max_code_and_scale(mode, M):
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((7, 33, 128)) * np.exp(rng.uniform(-20, 20, (7, 1, 1)))).astype(np.float32)
    y, sc, cd = oracle.qdq_groups(x, 64, mode, with_codes=True)
    for b in range(7):
        for j in range(2):
            blk = x[b, :, j * 64:(j + 1) * 64]
            a = np.abs(blk).max()
            assert sc[b, j] == np.float32(a) / np.float32(M)
            i = np.unravel_index(np.abs(blk).argmax(), blk.shape)
            code = cd[b, :, j * 64:(j + 1) * 64][i]
            val = oracle.e4m3_decode(np.array([code], np.uint8))[0] if mode == "e4m3" \
                else float(np.int8(code))
            assert abs(val) == M and np.sign(val) == np.sign(blk[i])


@pytest.mark.parametrize("mode", ["e4m3", "int8"])
def test_qdq_idempotent_and_codes_representable(mode):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((50, 64, 64)) * rng.uniform(0.01, 100, (50, 1, 1))).astype(np.float32)
    y, sc, cd = oracle.qdq_groups(x, 64, mode, with_codes=True)
    y2, sc2, cd2 = oracle.qdq_groups(y, 64, mode, with_codes=True)
    assert np.array_equal(cd, cd2)
    same = (sc == sc2)[:, 0]
    assert same.mean() > 0.5
    assert np.array_equal(y[same].view(np.uint32), y2[same].view(np.uint32))
    rel = np.abs(y2[~same] - y[~same]) / np.maximum(np.abs(y[~same]), 1e-30)
    assert np.all(rel <= 2.0 ** -23 * 1.01)
    if mode == "e4m3":
        vals = oracle.e4m3_decode(cd)
        assert not np.isnan(vals).any() and np.abs(vals).max() <= 448
        # dequantized values are the decoded codes times the scale
        assert np.allclose(y, vals * sc[:, None, :], rtol=0, atol=0)
    else:
        ci = cd.view(np.int8)
        assert ci.min() >= -127 and ci.max() <= 127


@pytest.mark.parametrize("mode", ["e4m3", "int8"])
def test_qdq_relative_error_bound(mode):
    # Round-to-nearest on the grid bounds the error by half a step: for E4M3,
    # 2^-4 relative in the normal range; for INT8 half the scale.
    rng = np.random.default_rng(6)
    x = rng.standard_normal((20, 16, 64)).astype(np.float32)
    y, sc = oracle.qdq_groups(x, 64, mode)
    s = sc[:, None, :]
    err = np.abs(y.astype(np.float64) - x)
    if mode == "int8":
        assert np.all(err <= 0.5 * s * (1 + 1e-5) + 1e-12)
    else:
        normal = np.abs(x) >= s * 2.0 ** -6
        assert np.all(err[normal] <= np.abs(x[normal]) * 2.0 ** -4 * (1 + 1e-5))
        sb = np.broadcast_to(s, x.shape)
        assert np.all(err[~normal] <= sb[~normal] * 2.0 ** -10 * (1 + 1e-5))


def test_qdq_zero_group_and_signed_zero():
    x = np.zeros((1, 4, 64), np.float32)
    x[0, 1, 3] = -0.0
    y, sc, cd = oracle.qdq_groups(x, 64, "e4m3", with_codes=True)
    assert sc[0, 0] == 0 and np.array_equal(y.view(np.uint32), x.view(np.uint32))
    assert cd[0, 1, 3] == 0x80
    # negative values that round to zero keep the sign in E4M3
    x = np.array([[[448.0, -1e-9, 1e-9, 0.0]]], np.float32)
    y, sc, cd = oracle.qdq_groups(x, 4, "e4m3", with_codes=True)
    assert list(cd[0, 0]) == [0x7E, 0x80, 0x00, 0x00]


@pytest.mark.parametrize("mode,M", [("e4m3", 448.0), ("int8", 127.0)])
def test_qdq_tiny_amax_threshold(mode, M):
    """Where fl(1/s) stops being finite.  a = M 2^-127 gives s = 2^-127 exactly
    and r = 2^127, finite: the group quantizes normally and its largest element
    is reproduced exactly (code M, M * 2^-127 = a).  a = M 2^-129 gives
    s = 2^-129 and 1/s = 2^129, beyond binary32: the group has no usable scale
    and every value becomes a zero of its sign (E4M3) or +0 (INT8), with scale 0
    -- in particular no NaN from 0 * inf at the zero elements."""
    lo = np.float32(M * 2.0 ** -127)
    x = np.array([[[lo, -lo / 4, 0.0, -0.0]]], np.float32)
    y, sc, cd = oracle.qdq_groups(x, 4, mode, with_codes=True)
    assert sc[0, 0] == np.float32(2.0 ** -127)
    assert y[0, 0, 0] == lo and np.isfinite(y).all()
    assert y[0, 0, 1] < 0
    for a in (np.float32(M * 2.0 ** -129), np.float32(1e-40), np.float32(2.0 ** -149)):
        x = np.array([[[a, -a / 2, 0.0, -0.0]]], np.float32)
        y, sc, cd = oracle.qdq_groups(x, 4, mode, with_codes=True)
        assert sc[0, 0] == 0.0
        assert not y.any() and np.isfinite(y).all()
        if mode == "e4m3":
            assert list(cd[0, 0]) == [0x00, 0x80, 0x00, 0x80]
            assert list(np.signbit(y[0, 0])) == [False, True, False, True]
        else:
            assert not cd.any()


@pytest.mark.parametrize("mode", ["e4m3", "int8"])
def test_qdq_odd_symmetry_and_monotone_within_a_group(mode):
    """Both grids and their rounding are symmetric about zero and order
    preserving: within a group (one scale) Q(-x) = -Q(x), and x <= y implies
    Q(x) <= Q(y).  A rounding that leans one way, or a wrong sign or exponent
    path, breaks one of the two."""
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((6, 8, 64)) * np.exp(rng.uniform(-6, 6, (6, 1, 1)))).astype(np.float32)
    y, sc = oracle.qdq_groups(x, 64, mode)
    yn, scn = oracle.qdq_groups(-x, 64, mode)
    assert np.array_equal(sc, scn)
    assert np.array_equal(np.abs(yn), np.abs(y)) and np.all((yn == -y) | ((yn == 0) & (y == 0)))
    for b in range(x.shape[0]):
        order = np.argsort(x[b].ravel(), kind="stable")
        assert np.all(np.diff(y[b].ravel()[order].astype(np.float64)) >= 0)


@pytest.mark.parametrize("mode", ["e4m3", "int8"])
def test_qdq_scale_invariance_by_powers_of_two(mode):
    """Scaling a group by 2^k (inside the normal range of s) scales its scale
    and every dequantized value by exactly 2^k: the codes depend on x / amax
    only, and powers of two pass through fl(a / M), fl(1 / s) and the products
    without rounding."""
    rng = np.random.default_rng(9)
    x = rng.standard_normal((4, 16, 32)).astype(np.float32)
    y, sc, cd = oracle.qdq_groups(x, 32, mode, with_codes=True)
    for k in (-20, -3, 5, 17):
        xs = (x * np.float32(2.0 ** k)).astype(np.float32)
        ys, scs, cds = oracle.qdq_groups(xs, 32, mode, with_codes=True)
        assert np.array_equal(cds, cd)
        assert np.array_equal(scs, (sc * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(ys, (y * np.float32(2.0 ** k)).astype(np.float32))


@pytest.mark.gpu
def test_reciprocal_reading_matches_torch_cuda_scalar_division():
    """The pages' 'rounded reciprocal multiplication as Torch scalar division':
    torch on CUDA divides by a host scalar through its rounded reciprocal; the
    oracle's codes equal codes of torch-CUDA's x / s."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((64, 64, 64)) * 3).astype(np.float32)
    y, sc, cd = oracle.qdq_groups(x, 64, "e4m3", with_codes=True)
    xt = torch.from_numpy(x).cuda()
    n_diff_true_div = 0
    for b in range(64):
        s = float(sc[b, 0])
        u = (xt[b] / s).cpu().numpy()
        assert np.array_equal(oracle.e4m3_encode(u), cd[b])
        n_diff_true_div += int((x[b] / np.float32(s) != u).sum())
    assert n_diff_true_div > 0   # the two readings do differ on these inputs
