"""Pins of the oracle's NVFP4 quantiser (CPU only).

What fixes the expected values:
* the rounding rule at its tie points and saturation bounds (golden fixture,
  worked by hand from round-to-nearest-even on the OCP e2m1 / e4m3 grids);
* fixed points: every representable value rounds to itself;
* brute force: every code is the nearest grid value (checked against all
  codes, independently of the oracle's search order);
* an exhaustive check over all finite bf16 and fp16 inputs that rounding the
  quotients x / dec and amax / 6 to fp32 first never changes the decision
  (so the oracle's double-precision quotients and a kernel's fp32 or exact
  comparisons agree);
* round trips: blocks built from e2m1 values times an e4m3 scale, with the
  block maximum at 6 x scale, quantise back to exactly those bytes.
"""
import json
from pathlib import Path

import numpy as np
import pytest

GOLDEN = Path(__file__).resolve().parent / "golden"

E2M1_TIES = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])   # midpoints of the e2m1 magnitude grid


@pytest.fixture(scope="module")
def o(oracle_mod):
    return oracle_mod


@pytest.fixture(scope="module")
def e4m3_grid(o):
    return np.array([o.e4m3fn_value(c) for c in range(0x7F)])     # codes 0..126, increasing


def test_golden_tie_points(o):
    g = json.loads((GOLDEN / "quantize_rounding.json").read_text())
    for t in g["e2m1_ties"] + g["e2m1_saturation"]:
        assert o.e2m1_round(t["q"]) == t["code"], t
    for t in g["e4m3_ties"] + g["e4m3_saturation"]:
        assert o.e4m3fn_round(t["s"]) == t["code"], t
        assert o.e4m3fn_value(t["code"]) == t.get("value", o.e4m3fn_value(t["code"]))


def test_e4m3_round_fixed_points_and_midpoints(o, e4m3_grid):
    for c, v in enumerate(e4m3_grid):
        assert o.e4m3fn_round(v) == c
    for c in range(0x7E):
        lo, hi = e4m3_grid[c], e4m3_grid[c + 1]
        mid = (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert o.e4m3fn_round(mid) == even, (c, mid)
        assert o.e4m3fn_round(np.nextafter(mid, 0)) == c
        assert o.e4m3fn_round(np.nextafter(mid, np.inf)) == c + 1


def test_e2m1_round_is_nearest_by_brute_force(o):
    grid = np.array([o.e2m1_value(c) for c in range(16)])
    rng = np.random.default_rng(3)
    qs = np.concatenate([rng.normal(0, 3, 4000), E2M1_TIES, -E2M1_TIES, [0.0, -0.0, 6.0, -6.0, 9.0]])
    for q in qs:
        c = o.e2m1_round(q)
        assert (c >> 3) == (1 if np.signbit(q) else 0), q
        d_all = np.abs(np.abs(grid[:8]) - min(abs(q), 6.0))
        assert abs(abs(grid[c]) - min(abs(q), 6.0)) == d_all.min(), (q, c)
        if np.sum(d_all == d_all.min()) == 2:           # a tie: the even code
            assert c % 2 == 0, (q, c)


def _bf16_values():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    return v[np.isfinite(v)]


def _f16_values():
    v = np.arange(1 << 16, dtype=np.uint16).view(np.float16).astype(np.float32)
    return v[np.isfinite(v)]


@pytest.mark.parametrize("values", [_bf16_values, _f16_values], ids=["bf16", "fp16"])
def test_fp32_quotients_decide_like_exact_ones(values, e4m3_grid):
    """For every finite input x and every non-zero e4m3 scale, x / dec rounded
    to fp32 sits on the same side of every e2m1 rounding boundary as the
    exact quotient (and on it exactly when the exact one is); likewise amax/6
    against every e4m3 rounding boundary."""
    x = np.abs(values())
    x64 = x.astype(np.float64)
    bounds = np.concatenate([E2M1_TIES, [6.0]])
    for dec in e4m3_grid[1:]:
        with np.errstate(over="ignore"):                # huge x over a small scale: inf, still above 6
            q32 = (x / np.float32(dec)).astype(np.float64)
        q64 = x64 / dec
        for t in bounds:
            assert np.array_equal(np.sign(q32 - t), np.sign(q64 - t)), (dec, t)
    mids = np.concatenate([(e4m3_grid[:-1] + e4m3_grid[1:]) / 2, [448.0]])
    s32 = (x / np.float32(6.0)).astype(np.float64)
    s64 = x64 / 6.0
    for t in mids:
        assert np.array_equal(np.sign(s32 - t), np.sign(s64 - t)), t


def test_round_trip_of_representable_blocks(o, e4m3_grid):
    rng = np.random.default_rng(11)
    rows, k = 37, 96
    grid = np.array([o.e2m1_value(c) for c in range(16)])
    codes = rng.integers(0, 16, (rows, k)).astype(np.uint8)
    codes[codes == 8] = 0                               # -0 and +0 are the same value; keep +0
    sfc = rng.integers(1, 0x7F, (rows, k // 16)).astype(np.uint8)
    # the largest magnitude of each block is 6 (code 7 or 15), so amax / 6 = dec exactly
    for r in range(rows):
        for b in range(k // 16):
            codes[r, 16 * b + rng.integers(0, 16)] = 7 if rng.random() < 0.5 else 15
    x = grid[codes] * np.repeat(e4m3_grid[sfc], 16, axis=1)
    got_codes, got_sf = o.quantize(x.astype(np.float32))
    np.testing.assert_array_equal(got_sf, sfc)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    np.testing.assert_array_equal(got_codes, packed)


def test_quantize_picks_nearest_values_and_zero_blocks(o):
    rng = np.random.default_rng(12)
    rows, k = 9, 160
    x = rng.normal(0, 1, (rows, k)).astype(np.float32)
    x[2, 16:32] = 0.0                                   # zero block: scale 0, codes +0
    x[3, 32:48] = -1e-6                                 # amax/6 below half the smallest scale: +0 codes
    x[4, 0:16] *= 1e5                                   # saturating scale (448)
    codes, sf = o.quantize(x)
    assert np.all(sf[2, 1] == 0) and np.all(codes[2, 8:16] == 0)
    assert sf[3, 2] == 0 and np.all(codes[3, 16:24] == 0)
    assert sf[4, 0] == 0x7E
    grid = np.array([o.e2m1_value(c) for c in range(8)])
    for r in range(rows):
        for b in range(k // 16):
            blk = x[r, 16 * b: 16 * b + 16].astype(np.float64)
            dec = o.e4m3fn_value(int(sf[r, b]))
            amax = np.abs(blk).max()
            # the scale is the e4m3 value nearest amax / 6 (or 448)
            assert abs(dec - min(amax / 6, 448.0)) <= min(abs(o.e4m3fn_value(c) - min(amax / 6, 448.0))
                                                          for c in range(0x7F))
            for j in range(16):
                byte = int(codes[r, 8 * b + j // 2])
                c = (byte >> (4 * (j % 2))) & 0xF
                if dec == 0:
                    assert c == 0
                    continue
                q = blk[j] / dec
                assert (c >> 3) == (1 if np.signbit(q) else 0)
                err = abs(grid[c & 7] - min(abs(q), 6.0))
                assert err == np.abs(grid - min(abs(q), 6.0)).min(), (r, b, j, q, c)
