"""CPU oracle for the NVFP4 block-scaled grouped GEMM (ctypes shim over nvfp4_oracle.c).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The product library neither imports nor links it, and it shares no code
with the GPU path.

What it computes is stated in ``nvfp4_oracle.c``: per group,
``C[i,j] = fp16_rne(sum_k e2m1(A[i,k]) e4m3(SFA[i,k/16]) e2m1(B[j,k]) e4m3(SFB[j,k/16]))``
accumulated in fp64 ("nvfp4 group gemm" submission 499344, kernel main loop at
the block-scaled gemm call; submission 506336, kernel configuration parameters
and the epilogue's single conversion to the C type).

Every function here is pinned by ``tests/test_oracle_pins.py`` against things
other than itself: torch's float8 decoder, numpy's float16 rounding, exact
integer arithmetic, brute force, closed forms and the scale-atom layout algebra
as printed on the submission 385043 page.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "nvfp4_oracle.c"
_SO = _HERE / "_build" / "libnvfp4_oracle.so"
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> Path:
    """Compile nvfp4_oracle.c with gcc (OpenMP, -O2, no fast-math)."""
    if not force and _SO.exists() and _SO.stat().st_mtime >= _SRC.stat().st_mtime:
        return _SO
    _SO.parent.mkdir(parents=True, exist_ok=True)
    tmp = _SO.with_suffix(f".so.tmp{os.getpid()}")
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-o", str(tmp), str(_SRC), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(str(build()))
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.nvfp4_oracle_e2m1_value.restype = ctypes.c_double
        lib.nvfp4_oracle_e2m1_value.argtypes = [ctypes.c_uint32]
        lib.nvfp4_oracle_e4m3fn_value.restype = ctypes.c_double
        lib.nvfp4_oracle_e4m3fn_value.argtypes = [ctypes.c_uint32]
        lib.nvfp4_oracle_fp16_bits.restype = ctypes.c_uint16
        lib.nvfp4_oracle_fp16_bits.argtypes = [ctypes.c_double]
        lib.nvfp4_oracle_max_threads.restype = ctypes.c_int
        lib.nvfp4_oracle_grouped_gemm.restype = None
        lib.nvfp4_oracle_grouped_gemm.argtypes = [
            ctypes.c_int, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.nvfp4_oracle_gemm_sampled.restype = None
        lib.nvfp4_oracle_gemm_sampled.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.nvfp4_oracle_scale_atom_bytes.restype = ctypes.c_size_t
        lib.nvfp4_oracle_scale_atom_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
        lib.nvfp4_oracle_scale_atom_offset.restype = ctypes.c_size_t
        lib.nvfp4_oracle_scale_atom_offset.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.nvfp4_oracle_pack_scales.restype = None
        lib.nvfp4_oracle_pack_scales.argtypes = [u8p, ctypes.c_int, ctypes.c_int, u8p]
        lib.nvfp4_oracle_e4m3fn_round.restype = ctypes.c_uint32
        lib.nvfp4_oracle_e4m3fn_round.argtypes = [ctypes.c_double]
        lib.nvfp4_oracle_e2m1_round.restype = ctypes.c_uint32
        lib.nvfp4_oracle_e2m1_round.argtypes = [ctypes.c_double]
        lib.nvfp4_oracle_quantize.restype = None
        lib.nvfp4_oracle_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint8, a.dtype
    return a


def max_threads() -> int:
    return int(_load().nvfp4_oracle_max_threads())


def e2m1_value(code: int) -> float:
    return float(_load().nvfp4_oracle_e2m1_value(int(code)))


def e4m3fn_value(code: int) -> float:
    return float(_load().nvfp4_oracle_e4m3fn_value(int(code)))


def fp16_bits(x: float) -> int:
    return int(_load().nvfp4_oracle_fp16_bits(float(x)))


def grouped_gemm(problem_sizes, A, B, SFA, SFB, *, threads: int = 0, out=None,
                 want_f64: bool = False):
    """Full C for every group.

    problem_sizes: sequence of (m, n, k, l). A[g]: uint8 [m, k/2]; B[g]: uint8
    [n, k/2]; SFA[g]: uint8 [m, k/16]; SFB[g]: uint8 [n, k/16] (row-major
    e4m3fn codes). Returns a list of float16 [m, n] arrays (``out`` may supply
    pre-filled arrays; groups with m == 0 or n == 0 are left as given). With
    ``want_f64`` the fp64 sums before rounding are returned instead.
    """
    lib = _load()
    G = len(problem_sizes)
    sizes = np.ascontiguousarray(np.asarray(problem_sizes, dtype=np.int32).reshape(G, 4))
    keep = []

    def ptrs(arrs):
        vals = []
        for a in arrs:
            if a is None:
                vals.append(0)
            else:
                keep.append(a)
                vals.append(_ptr(a))
        return np.asarray(vals, dtype=np.uint64)

    a_l = [_u8(a) for a in A]
    b_l = [_u8(b) for b in B]
    sa_l = [_u8(s) for s in SFA]
    sb_l = [_u8(s) for s in SFB]
    outs = []
    for g in range(G):
        m, n = int(sizes[g, 0]), int(sizes[g, 1])
        if out is not None:
            o = out[g]
            assert o.flags.c_contiguous
        elif want_f64:
            o = np.zeros((max(m, 0), max(n, 0)), dtype=np.float64)
        else:
            o = np.zeros((max(m, 0), max(n, 0)), dtype=np.float16)
        outs.append(o)
    pa, pb, psa, psb = ptrs(a_l), ptrs(b_l), ptrs(sa_l), ptrs(sb_l)
    pc = ptrs(outs)
    keep.extend([pa, pb, psa, psb, pc])
    if want_f64:
        lib.nvfp4_oracle_grouped_gemm(G, _ptr(sizes), _ptr(pa), _ptr(pb), _ptr(psa), _ptr(psb),
                                      None, _ptr(pc), int(threads))
    else:
        lib.nvfp4_oracle_grouped_gemm(G, _ptr(sizes), _ptr(pa), _ptr(pb), _ptr(psa), _ptr(psb),
                                      _ptr(pc), None, int(threads))
    return outs


def gemm_sampled(m, n, k, A, B, SFA, SFB, rows, cols, *, threads: int = 0) -> np.ndarray:
    """C[rows[s], cols[s]] of one group as float16, one output at a time."""
    lib = _load()
    A, B, SFA, SFB = _u8(A), _u8(B), _u8(SFA), _u8(SFB)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    cols = np.ascontiguousarray(cols, dtype=np.int32)
    assert rows.shape == cols.shape
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < m and cols.min() >= 0 and cols.max() < n)
    out = np.zeros(rows.shape, dtype=np.uint16)
    lib.nvfp4_oracle_gemm_sampled(int(m), int(n), int(k), _ptr(A), _ptr(B), _ptr(SFA), _ptr(SFB),
                                  int(rows.size), _ptr(rows), _ptr(cols), _ptr(out), int(threads))
    return out.view(np.float16)


def scale_atom_bytes(rows: int, k: int) -> int:
    return int(_load().nvfp4_oracle_scale_atom_bytes(int(rows), int(k)))


def scale_atom_offset(r: int, kb: int, k: int) -> int:
    return int(_load().nvfp4_oracle_scale_atom_offset(int(r), int(kb), int(k)))


def pack_scales(sf_rowmajor: np.ndarray, k: int) -> np.ndarray:
    """Row-major [rows, k/16] e4m3 codes -> the reordered atom layout (flat uint8)."""
    sf = _u8(sf_rowmajor)
    rows = sf.shape[0]
    assert sf.shape == (rows, k // 16), (sf.shape, k)
    out = np.empty(scale_atom_bytes(rows, k), dtype=np.uint8)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    _load().nvfp4_oracle_pack_scales(sf.ctypes.data_as(u8p), int(rows), int(k),
                                     out.ctypes.data_as(u8p))
    return out


def e4m3fn_round(s: float) -> int:
    """e4m3fn code nearest to s >= 0, ties to the even code, 448 for s >= 448."""
    return int(_load().nvfp4_oracle_e4m3fn_round(float(s)))


def e2m1_round(q: float) -> int:
    """e2m1 code nearest to q, ties to the even code, |q| saturating at 6, sign kept."""
    return int(_load().nvfp4_oracle_e2m1_round(float(q)))


def quantize(x: np.ndarray):
    """NVFP4 quantisation of a real matrix [rows, k] (k % 16 == 0; the values
    are taken as float32): returns (codes uint8 [rows, k/2], row-major scales
    uint8 [rows, k/16])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, k = x.shape
    assert k % 16 == 0
    codes = np.zeros((rows, k // 2), np.uint8)
    sf = np.zeros((rows, k // 16), np.uint8)
    if rows and k:
        _load().nvfp4_oracle_quantize(x.ctypes.data, rows, k, _ptr(codes), _ptr(sf))
    return codes, sf
