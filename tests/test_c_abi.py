"""CPU checks of the C ABI: the library builds, loads without a GPU, exports
every function include/nvfp4_grouped.h declares, and rejects bad arguments on
the host before touching CUDA. No call here reaches a kernel."""
import ctypes
import re
from pathlib import Path

import pytest

import nvfp4_block_scaled_grouped_gb300 as nv
from nvfp4_block_scaled_grouped_gb300 import build

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def L():
    build.build_library()
    return nv.lib()


def _declared_functions():
    text = "\n".join(p.read_text() for p in (ROOT / "include").glob("*.h"))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(nvfp4_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("nvfp4_grouped_gemm", "nvfp4_pack_scales", "nvfp4_scale_bytes", "nvfp4_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_scale_bytes_matches_oracle(L, oracle_mod):
    for rows in (0, 1, 127, 128, 129, 1000, 4096):
        for k in (0, 16, 32, 64, 96, 2048, 7168):
            want = oracle_mod.scale_atom_bytes(rows, k) if rows > 0 and k > 0 else 0
            assert nv.scale_bytes(rows, k) == want, (rows, k)


def _call(sizes, ptr=0x10000, **over):
    G = len(sizes)
    fields = {name: [over.get(name, {}).get(g, ptr) for g in range(G)] for name in ("A", "B", "SFA", "SFB", "C")}
    return nv.grouped_gemm(sizes, fields["A"], fields["B"], fields["SFA"], fields["SFB"], fields["C"],
                           stream=0, check=False)


def test_argument_errors_are_reported_on_the_host(L):
    assert _call([]) == 0                                                  # no groups: no-op
    assert _call([(0, 64, 64, 1), (5, 0, 64, 1)]) == 0                     # only empty groups: no-op
    assert L.nvfp4_grouped_gemm(-1, None, None, None, None, None, None, None) == -1
    assert L.nvfp4_grouped_gemm(1, None, None, None, None, None, None, None) == -1
    assert _call([(4, 64, 64, 1)] * (nv.MAX_GROUPS + 1)) == -1             # too many groups
    assert _call([(-1, 64, 64, 1)]) == -1                                  # negative size
    assert _call([(4, 64, 64, 65536)]) == -2                               # l above 65535
    assert _call([(40000, 64, 64, 60000)]) == -2                           # l * m above 2^31 - 1
    assert _call([(4, 64, 64, -1)]) == -1                                  # negative l
    assert _call([(4, 64, 64, 0), (0, 64, 64, 3)]) == 0                    # l == 0 or m == 0: empty, no-op
    assert _call([(4, 64, 48, 1)]) == -2                                   # k % 32
    assert _call([(4, 48, 64, 1)]) == -2                                   # n % 32
    assert _call([(4, 64, 64, 1)], C={0: 0}) == -1                         # null C
    assert _call([(4, 64, 64, 1)], A={0: 0}) == -1                         # null A
    assert _call([(4, 64, 64, 1)], SFB={0: 0x10008}) == -3                 # misaligned
    assert _call([(4, 64, 64, 1)], C={0: 0x10002}) == -3
    # k == 0: A/B/scales may be null, C still required
    assert _call([(4, 64, 0, 1)], C={0: 0}) == -1


def test_device_table_host_argument_errors(L):
    """nvfp4_grouped_gemm_device checks what the host can see (count range,
    null or misaligned arrays) before it touches the GPU; the group rules are
    checked by the kernel."""
    vp = ctypes.c_void_p
    arrays = [vp(0x10000 + 0x100 * i) for i in range(5)]
    f = L.nvfp4_grouped_gemm_device
    assert f(0, None, None, None, None, None, None, None) == 0                 # no groups: no-op
    assert f(-1, vp(0x20000), *arrays, None) == -1
    assert f(nv.MAX_GROUPS + 1, vp(0x20000), *arrays, None) == -1
    assert f(2, None, *arrays, None) == -1                                     # null sizes
    assert f(2, vp(0x20000), None, *arrays[1:], None) == -1                    # null pointer array
    assert f(2, vp(0x20008), *arrays, None) == -3                              # sizes not 16-byte aligned
    assert f(2, vp(0x20000), vp(0x10004), *arrays[1:], None) == -3             # pointer array not 8-byte aligned


def test_batched_call_host_argument_errors(L):
    f = L.nvfp4_grouped_gemm_batched
    counts = (ctypes.c_int * 3)(2, -1, 1)
    assert f(0, None, None, None, None, None, None, None, None) == 0       # no problems: no-op
    assert f(-1, None, None, None, None, None, None, None, None) == -1
    assert f(2, None, None, None, None, None, None, None, None) == -1      # null counts
    assert f(3, counts, None, None, None, None, None, None, None) == -1    # negative count
    big = (ctypes.c_int * 2)(300, 213)
    assert f(2, big, None, None, None, None, None, None, None) == -1       # 513 groups
    zero = (ctypes.c_int * 2)(0, 0)
    assert f(2, zero, None, None, None, None, None, None, None) == 0       # only empty problems


def test_quantize_pack_host_argument_errors(L):
    vp = ctypes.c_void_p
    f = L.nvfp4_quantize_pack
    x, c, s = vp(0x10000), vp(0x20000), vp(0x30000)
    assert f(x, 0, 0, 64, c, s, None) == 0                 # no rows: no-op
    assert f(x, 1, 4, 0, c, s, None) == 0                  # k == 0: no-op
    assert f(x, 0, -1, 64, c, s, None) == -1
    assert f(x, 7, 4, 64, c, s, None) == -1                # unknown input type
    assert f(x, 0, 4, 40, c, s, None) == -2                # k % 16
    assert f(None, 0, 4, 64, c, s, None) == -1
    assert f(vp(0x10008), 1, 4, 64, c, s, None) == -3      # misaligned


def test_pack_scales_argument_errors(L):
    vp = ctypes.c_void_p
    assert L.nvfp4_pack_scales(vp(0x10000), -1, 64, vp(0x20000), None) == -1
    assert L.nvfp4_pack_scales(vp(0x10000), 4, 40, vp(0x20000), None) == -2
    assert L.nvfp4_pack_scales(vp(0x10000), 4, 64, vp(0x20008), None) == -3
    assert L.nvfp4_pack_scales(None, 4, 64, vp(0x20000), None) == -1
    assert L.nvfp4_pack_scales(None, 0, 64, None, None) == 0              # nothing to do


def test_status_strings_and_tile_option(L):
    for code, name in nv.STATUS.items():
        assert L.nvfp4_status_string(code).decode() == name
    assert L.nvfp4_status_string(7).decode() == "NVFP4_ERR_UNKNOWN"
    assert L.nvfp4_set_tile_n(64) == -1
    assert L.nvfp4_set_tile_n(256) == 0
    assert L.nvfp4_set_tile_n(0) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    """The product path has no fallback: a missing library is an error."""
    monkeypatch.setattr(nv, "_lib", None)
    monkeypatch.setattr(nv, "_LIB_PATH", tmp_path / "missing.so")
    with pytest.raises(RuntimeError, match="missing"):
        nv.lib()


def test_pack_scales_batched_argument_errors(L):
    """Every entry is checked on the host before anything is enqueued."""
    vp = ctypes.c_void_p
    f = L.nvfp4_pack_scales_batched
    arr = lambda *v: (vp * len(v))(*[vp(x) if x else None for x in v])
    ints = lambda *v: (ctypes.c_int * len(v))(*v)
    assert f(0, None, None, None, None, None) == 0                                       # nothing to pack
    assert f(-1, None, None, None, None, None) == -1
    assert f(1025, None, None, None, None, None) == -1                                   # above NVFP4_PACK_MAX_BATCH
    assert f(1, None, ints(4), ints(64), arr(0x20000), None) == -1                       # null array
    src, dst = arr(0x10000, 0x11000), arr(0x20000, 0x21000)
    assert f(2, arr(0x10000, 0x11000), ints(4, -1), ints(64, 64), dst, None) == -1       # negative rows
    assert f(2, src, ints(4, 4), ints(64, 40), dst, None) == -2                          # k % 16
    assert f(2, src, ints(4, 4), ints(64, 64), arr(0x20000, 0x21008), None) == -3        # misaligned output
    assert f(2, arr(0x10000, 0), ints(4, 4), ints(64, 64), dst, None) == -1              # null pointer
    assert f(2, arr(0, 0), ints(0, 4), ints(64, 0), arr(0, 0), None) == 0                # only empty entries
