"""Pins for the CPU oracle: each check ties it to something other than itself.

* decode tables: the OCP e2m1 value list (golden fixture) and torch's float8
  e4m3fn decoder;
* fp16 rounding: numpy's float64 -> float16 conversion;
* the grouped sum: exact integer arithmetic (every term is an integer multiple
  of 2^-20), rounded by an integer round-to-nearest-even written here;
* brute force: dequantise to dense fp64 and multiply with numpy;
* closed forms / invariants: unit scales reduce to an integer matmul; doubling
  one scale block changes exactly that block's contribution;
* zero-size and k = 0 groups;
* the reordered scale layout: evaluated from the CuTe shape/stride/order printed
  on the submission 385043 page (golden fixture) with a layout evaluator written
  here.
"""
import json
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_grouped_gb300 import workloads

GOLDEN = Path(__file__).resolve().parent / "golden"


# ---------------------------------------------------------------- independent helpers

def e2m1_table():
    d = json.loads((GOLDEN / "e2m1_values.json").read_text())
    return np.array(d["values"], dtype=np.float64)


def e4m3_table_torch():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dequant(codes, sf, k):
    """Dense fp64 [rows, k] from packed codes and row-major scales (test-side)."""
    rows = codes.shape[0]
    lo = codes & 0xF
    hi = codes >> 4
    idx = np.empty((rows, k), dtype=np.int64)
    idx[:, 0::2] = lo
    idx[:, 1::2] = hi
    vals = e2m1_table()[idx]
    scale = e4m3_table_torch()[sf.astype(np.int64)]
    return vals * np.repeat(scale, 16, axis=1)


def int_operand(codes, sf, k):
    """Integer representation: 2*e2m1 * 512*e4m3 = value * 2^10 (exact ints)."""
    two_a = (2 * e2m1_table()).astype(np.int64)
    s512 = e4m3_table_torch() * 512.0
    assert np.all(np.isnan(s512) | (s512 == np.round(s512)))
    s512 = np.nan_to_num(s512).astype(np.int64)
    rows = codes.shape[0]
    idx = np.empty((rows, k), dtype=np.int64)
    idx[:, 0::2] = codes & 0xF
    idx[:, 1::2] = codes >> 4
    return two_a[idx] * np.repeat(s512[sf.astype(np.int64)], 16, axis=1)


def exact_fp16_bits(num: int, den_log2: int) -> int:
    """Round num / 2^den_log2 to binary16, nearest-even, with integer arithmetic only."""
    if num == 0:
        return 0
    sign = 0x8000 if num < 0 else 0
    a = abs(num)
    e = a.bit_length() - 1 - den_log2           # value in [2^e, 2^(e+1))
    binade = max(e, -14)
    if binade > 15:
        return sign | 0x7C00
    shift = den_log2 + binade - 10               # quantum = 2^(binade-10)
    if shift > 0:
        r, rem = divmod(a, 1 << shift)
        half = 1 << (shift - 1)
        if rem > half or (rem == half and (r & 1)):
            r += 1
    else:
        r = a << (-shift)
    if r >= 2048:
        r >>= 1
        binade += 1
    if r < 1024:
        return sign | r
    if binade + 15 >= 31:
        return sign | 0x7C00
    return sign | ((binade + 15) << 10) | (r - 1024)


def bits16(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def quantized(rng, rows, k, scale=1.0):
    x = torch.from_numpy((rng.standard_normal((rows, k)) * scale).astype(np.float32))
    return workloads.quantize_nvfp4(x)


# ---------------------------------------------------------------- decode tables

def test_e2m1_all_codes_match_ocp_table(oracle_mod):
    table = e2m1_table()
    for code in range(16):
        v = oracle_mod.e2m1_value(code)
        assert v == table[code], code
        assert np.signbit(v) == np.signbit(table[code]), code  # code 8 is -0


def test_e4m3fn_all_codes_match_torch(oracle_mod):
    ref = e4m3_table_torch()
    for code in range(256):
        v = oracle_mod.e4m3fn_value(code)
        if np.isnan(ref[code]):
            assert np.isnan(v), code
        else:
            assert v == ref[code], (code, v, ref[code])
            assert np.signbit(v) == np.signbit(ref[code]), code
    assert np.isnan(oracle_mod.e4m3fn_value(0x7F)) and np.isnan(oracle_mod.e4m3fn_value(0xFF))
    assert oracle_mod.e4m3fn_value(0x7E) == 448.0
    assert oracle_mod.e4m3fn_value(0x01) == 2.0 ** -9
    assert oracle_mod.e4m3fn_value(0x38) == 1.0


# ---------------------------------------------------------------- fp16 rounding

def test_fp16_rounding_matches_numpy(oracle_mod):
    rng = np.random.default_rng(7)
    xs = [0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e300, -1e300, float("inf"),
          -float("inf"), 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -26, 2.0 ** -14,
          2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0, 1e-300]
    # random values over the whole fp16 range and beyond, plus exact ties
    mags = np.ldexp(rng.random(20000) + 0.5, rng.integers(-30, 18, 20000))
    xs += list(mags * rng.choice([-1.0, 1.0], 20000))
    ties = (rng.integers(0, 4096, 4000) * 2 + 1).astype(np.float64)
    xs += list(np.ldexp(ties, rng.integers(-36, 4, 4000)))   # odd multiples of half quanta
    for x in xs:
        got = oracle_mod.fp16_bits(x)
        want = int(np.array(x, dtype=np.float64).astype(np.float16).view(np.uint16))
        assert got == want, (x, hex(got), hex(want))
    assert oracle_mod.fp16_bits(float("nan")) & 0x7C00 == 0x7C00 and oracle_mod.fp16_bits(float("nan")) & 0x3FF


def test_exact_fp16_helper_matches_numpy():
    """The test's own integer rounding agrees with numpy where fp64 is exact."""
    rng = np.random.default_rng(3)
    for _ in range(5000):
        num = int(rng.integers(-(1 << 50), 1 << 50))
        den = int(rng.integers(0, 60))
        want = int(np.array(Fraction(num, 1 << den).__float__(), dtype=np.float64)
                   .astype(np.float16).view(np.uint16))
        assert exact_fp16_bits(num, den) == want, (num, den)


# ---------------------------------------------------------------- the grouped sum

SHAPES = [(1, 1, 32), (2, 3, 64), (3, 2, 256), (17, 5, 288), (5, 17, 96), (128, 1, 64),
          (129, 3, 32), (1, 129, 256), (3, 128, 288)]


@pytest.mark.parametrize("m,n,k", SHAPES)
def test_bruteforce_dequant_matmul(oracle_mod, m, n, k):
    rng = np.random.default_rng(m * 1000 + n * 10 + k)
    a, sfa = quantized(rng, m, k)
    b, sfb = quantized(rng, n, k)
    (c,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [a], [b], [sfa], [sfb])
    ref = dequant(a, sfa, k) @ dequant(b, sfb, k).T
    np.testing.assert_array_equal(c.view(np.uint16), bits16(ref))


@pytest.mark.parametrize("m,n,k", [(4, 5, 64), (7, 3, 288), (16, 16, 1024)])
def test_exact_integer_sum(oracle_mod, m, n, k):
    """Moderate scales (2^-4..2^4): the fp64 sum is exact, so the oracle must
    equal the exactly rounded integer result bit for bit."""
    rng = np.random.default_rng(11 + k)
    codes = [c for c in range(0x7F) if 3 <= (c >> 3) <= 11]
    a, sfa = workloads.random_codes(rng, m, k, sf_codes=codes)
    b, sfb = workloads.random_codes(rng, n, k, sf_codes=codes)
    N = int_operand(a, sfa, k) @ int_operand(b, sfb, k).T
    (c,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [a], [b], [sfa], [sfb])
    want = np.array([[exact_fp16_bits(int(N[i, j]), 20) for j in range(n)] for i in range(m)],
                    dtype=np.uint16)
    got = c.view(np.uint16).copy()
    got[got == 0x8000] = 0  # an exact zero sum is +0
    np.testing.assert_array_equal(got, want)


def test_extreme_scales_within_fp64_bound(oracle_mod):
    """All finite positive e4m3 codes (incl. subnormals): the fp64 sums stay
    within the forward error bound k * 2^-53 * sum|terms| of the exact sum, and
    C is the round-to-nearest-even fp16 of that fp64 sum."""
    m, n, k = 9, 7, 512
    rng = np.random.default_rng(5)
    a, sfa = workloads.random_codes(rng, m, k)
    b, sfb = workloads.random_codes(rng, n, k)
    ia, ib = int_operand(a, sfa, k), int_operand(b, sfb, k)
    N = ia @ ib.T
    S = np.abs(ia) @ np.abs(ib).T
    (c64,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [a], [b], [sfa], [sfb], want_f64=True)
    (c16,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [a], [b], [sfa], [sfb])
    for i in range(m):
        for j in range(n):
            err = abs(Fraction(float(c64[i, j])) - Fraction(int(N[i, j]), 1 << 20))
            bound = Fraction(k * int(S[i, j]), 1 << 20) * Fraction(1, 1 << 53)
            assert err <= bound, (i, j)
    np.testing.assert_array_equal(c16.view(np.uint16), bits16(c64))


def test_unit_scales_reduce_to_integer_matmul(oracle_mod):
    """All scales 1.0 (0x38): 2*e2m1 is an integer in [-12, 12], so
    C = (IA @ IB^T) / 4 with an int64 matmul."""
    m, n, k = 33, 19, 160
    rng = np.random.default_rng(9)
    a = rng.integers(0, 256, (m, k // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    sfa = np.full((m, k // 16), 0x38, dtype=np.uint8)
    sfb = np.full((n, k // 16), 0x38, dtype=np.uint8)
    two = np.array([0, 1, 2, 3, 4, 6, 8, 12], dtype=np.int64)
    two = np.concatenate([two, -two])

    def ints(c):
        idx = np.empty((c.shape[0], k), dtype=np.int64)
        idx[:, 0::2], idx[:, 1::2] = c & 0xF, c >> 4
        return two[idx]

    ref = (ints(a) @ ints(b).T).astype(np.float64) / 4.0
    (c,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [a], [b], [sfa], [sfb])
    np.testing.assert_array_equal(c.view(np.uint16), bits16(ref))


def test_scale_block_of_a_single_element(oracle_mod):
    """One non-zero A element at k=17 (high nibble of byte 8) is scaled by SFA
    block 1 and meets SFB block 1 only: C[0, j] = a * sfa[1] * b[17] * sfb[j, 1]."""
    m, n, k = 1, 2, 32
    a = np.zeros((m, k // 2), dtype=np.uint8)
    a[0, 8] = 0x30  # code 3 (1.5) in the high nibble, +0 in the low nibble
    sfa = np.array([[0x38, 0x40]], dtype=np.uint8)                  # 1.0, 2.0
    b = np.full((n, k // 2), 0x44, dtype=np.uint8)                  # 2.0 everywhere
    sfb = np.array([[0x38, 0x30], [0x38, 0x48]], dtype=np.uint8)    # block 1: 0.5 and 4.0
    (c,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [a], [b], [sfa], [sfb])
    assert c[0, 0] == np.float16(1.5 * 2.0 * 2.0 * 0.5)
    assert c[0, 1] == np.float16(1.5 * 2.0 * 2.0 * 4.0)


def test_nibble_swap_invariance(oracle_mod):
    """Elements 2p and 2p+1 share a byte and a 16-wide scale block, so swapping
    the nibbles of every byte of both A and B permutes the terms of each sum
    and leaves C unchanged: the nibble order is a convention between producer
    and consumer, not something C can reveal."""
    m, n, k = 9, 11, 96
    rng = np.random.default_rng(12)
    a, sfa = quantized(rng, m, k)
    b, sfb = quantized(rng, n, k)
    swap = lambda x: ((x & 0xF) << 4) | (x >> 4)
    (c,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [a], [b], [sfa], [sfb])
    (cs,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [swap(a)], [swap(b)], [sfa], [sfb])
    np.testing.assert_array_equal(c.view(np.uint16), cs.view(np.uint16))
    (ca,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [swap(a)], [b], [sfa], [sfb])
    assert not np.array_equal(c.view(np.uint16), ca.view(np.uint16))


@pytest.mark.parametrize("which", ["sfa", "sfb"])
def test_scale_doubling_invariant(oracle_mod, which):
    m, n, k = 12, 10, 256
    rng = np.random.default_rng(21)
    a, sfa = quantized(rng, m, k)
    b, sfb = quantized(rng, n, k)
    row, blk = 5, 7
    (base,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [a], [b], [sfa], [sfb], want_f64=True)
    sfa2, sfb2 = sfa.copy(), sfb.copy()
    target = sfa2 if which == "sfa" else sfb2
    code = int(target[row, blk])
    assert 1 <= (code >> 3) <= 13
    target[row, blk] = code + 8          # exponent field + 1: the scale doubles
    (dbl,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [a], [b], [sfa2], [sfb2], want_f64=True)
    # the block's own partial sum, from a k = 16 problem on that slice
    sl = slice(blk * 8, blk * 8 + 8)
    if which == "sfa":
        (part,) = oracle_mod.grouped_gemm([(1, n, 16, 1)], [a[row:row + 1, sl]], [b[:, sl]],
                                          [sfa[row:row + 1, blk:blk + 1]], [sfb[:, blk:blk + 1]],
                                          want_f64=True)
        np.testing.assert_array_equal(dbl[row] - base[row], part[0])
        others = np.arange(m) != row
        np.testing.assert_array_equal(dbl[others], base[others])
    else:
        (part,) = oracle_mod.grouped_gemm([(m, 1, 16, 1)], [a[:, sl]], [b[row:row + 1, sl]],
                                          [sfa[:, blk:blk + 1]], [sfb[row:row + 1, blk:blk + 1]],
                                          want_f64=True)
        np.testing.assert_array_equal(dbl[:, row] - base[:, row], part[:, 0])
        others = np.arange(n) != row
        np.testing.assert_array_equal(dbl[:, others], base[:, others])


def test_zero_size_groups_untouched_and_k0_zero(oracle_mod):
    rng = np.random.default_rng(2)
    sizes = [(0, 64, 64, 1), (3, 0, 64, 1), (4, 32, 0, 1), (5, 32, 64, 1)]
    A, B, SFA, SFB, out = [], [], [], [], []
    for m, n, k, _ in sizes:
        a, sa = quantized(rng, m, k) if m and k else (np.zeros((m, k // 2), np.uint8), np.zeros((m, k // 16), np.uint8))
        b, sb = quantized(rng, n, k) if n and k else (np.zeros((n, k // 2), np.uint8), np.zeros((n, k // 16), np.uint8))
        A.append(a); B.append(b); SFA.append(sa); SFB.append(sb)
        out.append(np.full((m, n), np.uint16(0x7E00)).view(np.float16))
    res = oracle_mod.grouped_gemm(sizes, A, B, SFA, SFB, out=out)
    assert res[0].size == 0 and res[1].size == 0
    np.testing.assert_array_equal(res[2].view(np.uint16), np.zeros((4, 32), np.uint16))
    assert not np.isnan(res[3].astype(np.float32)).any()


def test_sampled_matches_full(oracle_mod):
    m, n, k = 40, 24, 320
    rng = np.random.default_rng(4)
    a, sfa = quantized(rng, m, k)
    b, sfb = quantized(rng, n, k)
    (c,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [a], [b], [sfa], [sfb])
    rows = rng.integers(0, m, 200)
    cols = rng.integers(0, n, 200)
    s = oracle_mod.gemm_sampled(m, n, k, a, b, sfa, sfb, rows, cols)
    np.testing.assert_array_equal(s.view(np.uint16), c[rows, cols].view(np.uint16))


def test_single_thread_equals_all_threads(oracle_mod):
    m, n, k = 20, 30, 256
    rng = np.random.default_rng(8)
    a, sfa = quantized(rng, m, k)
    b, sfb = quantized(rng, n, k)
    (c1,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [a], [b], [sfa], [sfb], threads=1)
    (cn,) = oracle_mod.grouped_gemm([(m, n, k, 1)], [a], [b], [sfa], [sfb], threads=0)
    np.testing.assert_array_equal(c1.view(np.uint16), cn.view(np.uint16))


# ---------------------------------------------------------------- reordered scale layout

def _flatten(shape, stride):
    if isinstance(shape, (list, tuple)):
        out = []
        for s, d in zip(shape, stride):
            out += _flatten(s, d)
        return out
    return [(shape, stride)]


def _mode_offset(shape, stride, idx):
    """Offset of a 1-D index into a (possibly nested) CuTe mode: colexicographic."""
    off = 0
    for s, d in _flatten(shape, stride):
        off += (idx % s) * d
        idx //= s
    return off


def cute_tile_to_shape_offset(atom_shape, atom_stride, order, full_shape, coord):
    """Offset of coord in tile_to_shape(atom, full_shape, order): the atom is
    repeated over ceil(full/atom) per mode; the repeats are laid out compactly
    with the mode of the smallest order value fastest; each repeat spans the
    atom's cosize."""
    atom_sizes = [int(np.prod([s for s, _ in _flatten(sh, sh)])) for sh in atom_shape]
    cosize = 1 + sum((s - 1) * d for s, d in _flatten(atom_shape, atom_stride))
    reps = [-(-f // a) for f, a in zip(full_shape, atom_sizes)]
    rep_stride = [0] * len(reps)
    acc = cosize
    for mode in sorted(range(len(reps)), key=lambda i: order[i]):
        rep_stride[mode] = acc
        acc *= reps[mode]
    off = 0
    for mode, c in enumerate(coord):
        a = atom_sizes[mode]
        off += _mode_offset(atom_shape[mode], atom_stride[mode], c % a)
        off += (c // a) * rep_stride[mode]
    return off


@pytest.mark.parametrize("rows,k", [(1, 32), (128, 64), (129, 96), (300, 256), (256, 7168 // 8)])
def test_atom_offsets_match_page_layout(oracle_mod, rows, k):
    spec = json.loads((GOLDEN / "scale_atom_layout.json").read_text())
    atom_shape = [tuple(x) for x in spec["atom_shape"]] + [1]
    atom_stride = [tuple(x) for x in spec["atom_stride"]] + [0]
    order = spec["tile_order"]
    for r in range(rows):
        for kk in range(0, k, 16):
            want = cute_tile_to_shape_offset(atom_shape, atom_stride, order, (rows, k, 1), (r, kk, 0))
            assert oracle_mod.scale_atom_offset(r, kk // 16, k) == want, (r, kk)
            # every element of the 16-wide block shares the scale (stride 0)
            assert cute_tile_to_shape_offset(atom_shape, atom_stride, order, (rows, k, 1), (r, kk + 15, 0)) == want


@pytest.mark.parametrize("rows,k", [(1, 32), (128, 64), (129, 96), (300, 256), (513, 2048)])
def test_pack_is_bijective_with_zero_padding(oracle_mod, rows, k):
    rng = np.random.default_rng(rows + k)
    sf = rng.integers(1, 256, (rows, k // 16), dtype=np.uint8)  # non-zero so padding is visible
    packed = oracle_mod.pack_scales(sf, k)
    assert packed.size == (-(-rows // 128) * 128) * (-(-k // 64) * 4)
    seen = np.zeros(packed.size, dtype=bool)
    for r in range(rows):
        for kb in range(k // 16):
            off = oracle_mod.scale_atom_offset(r, kb, k)
            assert not seen[off]
            seen[off] = True
            assert packed[off] == sf[r, kb]
    assert np.all(packed[~seen] == 0)
    assert seen.sum() == rows * (k // 16)
