"""NVFP4 block-scaled grouped GEMM for GB300 (sm_103a): Python binding.

A thin ctypes layer over the C ABI in ``include/nvfp4_grouped.h``
(``_lib/libnvfp4_grouped.so``): argument marshalling only, every step of the
computation runs in the library's CUDA kernels. There is no fallback: if the
library is missing or fails to load, every call raises.

The functions mirror the C entry points:

* :func:`grouped_gemm` -- ``nvfp4_grouped_gemm`` (raw device pointers);
* :func:`grouped_gemm_tensors` -- the same call taking torch CUDA tensors;
* :func:`grouped_gemm_batched` -- ``nvfp4_grouped_gemm_batched`` (several
  grouped problems, one launch);
* :func:`grouped_gemm_device` / :class:`DeviceGroupTable` --
  ``nvfp4_grouped_gemm_device`` (group table in device memory);
* :func:`pack_scales` / :func:`scale_bytes` -- the scale-layout packer;
* :func:`quantize_pack` / :func:`quantize_pack_tensor` -- ``nvfp4_quantize_pack``
  (bf16 / fp16 activations to e2m1 codes and atom-layout scales);
* :func:`device_status`, :func:`set_tile_n`.
"""
from __future__ import annotations

import ctypes
import threading
from pathlib import Path

__all__ = [
    "Nvfp4Error", "lib", "library_path", "grouped_gemm", "grouped_gemm_tensors", "grouped_gemm_batched",
    "grouped_gemm_device",
    "DeviceGroupTable", "quantize_pack", "quantize_pack_tensor", "DTYPE_BF16", "DTYPE_F16", "pack_scales",
    "pack_scales_tensor", "pack_scales_batched", "pack_scales_tensors", "scale_bytes", "device_status",
    "set_tile_n", "MAX_GROUPS", "PACK_MAX_BATCH", "STATUS",
]

_PKG = Path(__file__).resolve().parent
_LIB_PATH = _PKG / "_lib" / "libnvfp4_grouped.so"
MAX_GROUPS = 512
PACK_MAX_BATCH = 1024
STATUS = {0: "NVFP4_OK", -1: "NVFP4_ERR_INVALID_ARG", -2: "NVFP4_ERR_UNSUPPORTED",
          -3: "NVFP4_ERR_MISALIGNED", -4: "NVFP4_ERR_CUDA", -5: "NVFP4_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class ProblemSize(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int32), ("n", ctypes.c_int32), ("k", ctypes.c_int32), ("l", ctypes.c_int32)]


def library_path() -> Path:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load the CUDA library (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not _LIB_PATH.exists():
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(str(_LIB_PATH))
        vp, vpp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
        L.nvfp4_grouped_gemm.restype = ctypes.c_int
        L.nvfp4_grouped_gemm.argtypes = [ctypes.c_int, ctypes.POINTER(ProblemSize), vpp, vpp, vpp, vpp, vpp, vp]
        L.nvfp4_grouped_gemm_batched.restype = ctypes.c_int
        L.nvfp4_grouped_gemm_batched.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ProblemSize),
                                                 vpp, vpp, vpp, vpp, vpp, vp]
        L.nvfp4_grouped_gemm_device.restype = ctypes.c_int
        L.nvfp4_grouped_gemm_device.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp, vp, vp]
        L.nvfp4_quantize_pack.restype = ctypes.c_int
        L.nvfp4_quantize_pack.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp]
        L.nvfp4_scale_bytes.restype = ctypes.c_size_t
        L.nvfp4_scale_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
        L.nvfp4_pack_scales.restype = ctypes.c_int
        L.nvfp4_pack_scales.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, vp]
        L.nvfp4_pack_scales_batched.restype = ctypes.c_int
        L.nvfp4_pack_scales_batched.argtypes = [ctypes.c_int, vpp, ctypes.POINTER(ctypes.c_int),
                                                ctypes.POINTER(ctypes.c_int), vpp, vp]
        L.nvfp4_device_status.restype = ctypes.c_int
        L.nvfp4_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
        L.nvfp4_status_string.restype = ctypes.c_char_p
        L.nvfp4_status_string.argtypes = [ctypes.c_int]
        L.nvfp4_last_error_message.restype = ctypes.c_char_p
        L.nvfp4_last_error_message.argtypes = []
        L.nvfp4_set_tile_n.restype = ctypes.c_int
        L.nvfp4_set_tile_n.argtypes = [ctypes.c_int]
        _lib = L
        return L


def _check(status: int) -> None:
    if status != 0:
        raise Nvfp4Error(status, lib().nvfp4_last_error_message().decode(errors="replace"))


def _stream_handle(stream) -> int:
    """A cudaStream_t value from None / int / torch.cuda.Stream."""
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _ptr_array(values):
    arr = (ctypes.c_void_p * max(len(values), 1))()
    for i, v in enumerate(values):
        arr[i] = int(v) if v else None
    return arr


def grouped_gemm(problem_sizes, A, B, SFA, SFB, C, stream=None, *, check: bool = True) -> int:
    """nvfp4_grouped_gemm with host lists of device addresses (ints)."""
    G = len(problem_sizes)
    sizes = (ProblemSize * max(G, 1))()
    for g, (m, n, k, l) in enumerate(problem_sizes):
        sizes[g] = ProblemSize(int(m), int(n), int(k), int(l))
    status = lib().nvfp4_grouped_gemm(
        G, sizes, _ptr_array(A), _ptr_array(B), _ptr_array(SFA), _ptr_array(SFB), _ptr_array(C),
        ctypes.c_void_p(_stream_handle(stream) or None))
    if check:
        _check(status)
    return status


def grouped_gemm_batched(problems, stream=None, *, check: bool = True) -> int:
    """nvfp4_grouped_gemm_batched: `problems` is a list of (problem_sizes, A,
    B, SFA, SFB, C) tuples with host lists of device addresses (ints), one
    per independent grouped problem; all run in one launch."""
    counts = (ctypes.c_int * max(len(problems), 1))(*[len(p[0]) for p in problems])
    flat = [[], [], [], [], [], []]
    for p in problems:
        for i in range(6):
            flat[i].extend(p[i])
    G = len(flat[0])
    sizes = (ProblemSize * max(G, 1))()
    for g, (m, n, k, l) in enumerate(flat[0]):
        sizes[g] = ProblemSize(int(m), int(n), int(k), int(l))
    status = lib().nvfp4_grouped_gemm_batched(
        len(problems), counts, sizes, *[_ptr_array(flat[i]) for i in range(1, 6)],
        ctypes.c_void_p(_stream_handle(stream) or None))
    if check:
        _check(status)
    return status


def _dptr(t):
    return 0 if t is None or t.numel() == 0 else int(t.data_ptr())


def grouped_gemm_tensors(problem_sizes, A, B, SFA, SFB, C, stream=None) -> None:
    """Same call with torch CUDA tensors: A/B uint8 [rows, k/2], SFA/SFB uint8
    atom-layout buffers, C float16 [m, n] (written in place)."""
    grouped_gemm(problem_sizes, [_dptr(t) for t in A], [_dptr(t) for t in B], [_dptr(t) for t in SFA],
                 [_dptr(t) for t in SFB], [_dptr(t) for t in C], stream)


def grouped_gemm_device(group_count: int, sizes_ptr: int, A_ptr: int, B_ptr: int, SFA_ptr: int, SFB_ptr: int,
                        C_ptr: int, stream=None, *, check: bool = True) -> int:
    """nvfp4_grouped_gemm_device: every argument but group_count is the device
    address of an array of group_count entries (sizes int32 [G, 4], the others
    uint64 device addresses)."""
    vp = ctypes.c_void_p
    status = lib().nvfp4_grouped_gemm_device(
        int(group_count), vp(int(sizes_ptr) or None), vp(int(A_ptr) or None), vp(int(B_ptr) or None),
        vp(int(SFA_ptr) or None), vp(int(SFB_ptr) or None), vp(int(C_ptr) or None),
        vp(_stream_handle(stream) or None))
    if check:
        _check(status)
    return status


class DeviceGroupTable:
    """Device-resident group table for :func:`grouped_gemm_device`: sizes int32
    [G, 4] and five int64 arrays of device addresses, on `device`. ``set``
    rewrites them (a host-to-device copy on the current stream); ``run``
    issues the call. The arrays keep their addresses, so a captured ``run``
    can be replayed after ``set``."""

    def __init__(self, group_count: int, device="cuda"):
        import torch
        self.group_count = int(group_count)
        self.sizes = torch.zeros((max(self.group_count, 1), 4), dtype=torch.int32, device=device)
        self.ptrs = torch.zeros((5, max(self.group_count, 1)), dtype=torch.int64, device=device)

    def set(self, problem_sizes, A, B, SFA, SFB, C) -> None:
        """problem_sizes: (m, n, k, l) per group; A..C: torch tensors or ints (device addresses)."""
        import torch
        assert len(problem_sizes) == self.group_count
        addr = lambda t: int(t) if isinstance(t, int) else _dptr(t)
        host_sizes = torch.tensor([[int(v) for v in s] for s in problem_sizes], dtype=torch.int32)
        host_ptrs = torch.tensor([[addr(t) for t in col] for col in (A, B, SFA, SFB, C)], dtype=torch.int64)
        self.sizes[: self.group_count].copy_(host_sizes)
        self.ptrs[:, : self.group_count].copy_(host_ptrs)

    def run(self, stream=None, *, check: bool = True) -> int:
        row = lambda i: self.ptrs[i].data_ptr()
        return grouped_gemm_device(self.group_count, self.sizes.data_ptr(), row(0), row(1), row(2), row(3), row(4),
                                   stream, check=check)


DTYPE_BF16, DTYPE_F16 = 0, 1


def quantize_pack(x_ptr: int, x_dtype: int, rows: int, k: int, codes_ptr: int, sf_atoms_ptr: int, stream=None,
                  *, check: bool = True) -> int:
    """nvfp4_quantize_pack with raw device addresses."""
    vp = ctypes.c_void_p
    status = lib().nvfp4_quantize_pack(vp(int(x_ptr) or None), int(x_dtype), int(rows), int(k),
                                       vp(int(codes_ptr) or None), vp(int(sf_atoms_ptr) or None),
                                       vp(_stream_handle(stream) or None))
    if check:
        _check(status)
    return status


def quantize_pack_tensor(x, stream=None):
    """torch bf16 / fp16 CUDA tensor [rows, k] -> (codes uint8 [rows, k/2],
    atom-layout scales uint8 [scale_bytes(rows, k)]), both new tensors."""
    import torch
    assert x.dim() == 2 and x.is_contiguous() and x.dtype in (torch.bfloat16, torch.float16)
    rows, k = x.shape
    codes = torch.empty((rows, k // 2), dtype=torch.uint8, device=x.device)
    sf = torch.empty(scale_bytes(rows, k), dtype=torch.uint8, device=x.device)
    if rows and k:
        quantize_pack(x.data_ptr(), DTYPE_BF16 if x.dtype == torch.bfloat16 else DTYPE_F16, rows, k,
                      codes.data_ptr(), sf.data_ptr(), stream)
    return codes, sf


def scale_bytes(rows: int, k: int) -> int:
    return int(lib().nvfp4_scale_bytes(int(rows), int(k)))


def pack_scales(sf_rowmajor_ptr: int, rows: int, k: int, sf_atoms_ptr: int, stream=None) -> None:
    _check(lib().nvfp4_pack_scales(ctypes.c_void_p(int(sf_rowmajor_ptr) or None), int(rows), int(k),
                                   ctypes.c_void_p(int(sf_atoms_ptr) or None),
                                   ctypes.c_void_p(_stream_handle(stream) or None)))


def pack_scales_tensor(sf_rowmajor, k: int, stream=None):
    """Device uint8 [rows, k/16] -> new device uint8 tensor in the atom layout."""
    import torch
    rows = sf_rowmajor.shape[0]
    out = torch.empty(scale_bytes(rows, k), dtype=torch.uint8, device=sf_rowmajor.device)
    if out.numel():
        pack_scales(sf_rowmajor.data_ptr(), rows, k, out.data_ptr(), stream)
    return out


def pack_scales_batched(entries, stream=None, *, check: bool = True) -> int:
    """nvfp4_pack_scales_batched: entries = [(sf_rowmajor_ptr, rows, k, sf_atoms_ptr), ...]."""
    n = len(entries)
    rows = (ctypes.c_int * max(n, 1))(*[int(e[1]) for e in entries])
    ks = (ctypes.c_int * max(n, 1))(*[int(e[2]) for e in entries])
    st = lib().nvfp4_pack_scales_batched(n, _ptr_array([e[0] for e in entries]), rows, ks,
                                         _ptr_array([e[3] for e in entries]),
                                         ctypes.c_void_p(_stream_handle(stream) or None))
    if check:
        _check(st)
    return st


def pack_scales_tensors(mats, stream=None):
    """[(device uint8 [rows, k/16], k), ...] -> new device uint8 tensors in the
    atom layout, all packed by one launch."""
    import torch
    outs = [torch.empty(scale_bytes(sf.shape[0], k), dtype=torch.uint8, device=sf.device) for sf, k in mats]
    entries = [(sf.data_ptr(), sf.shape[0], k, out.data_ptr()) for (sf, k), out in zip(mats, outs) if out.numel()]
    if entries:
        pack_scales_batched(entries, stream)
    return outs


def device_status(stream=None) -> int:
    """Read and clear the device status word of this stream's workspace."""
    st = ctypes.c_int(0)
    _check(lib().nvfp4_device_status(ctypes.c_void_p(_stream_handle(stream) or None), ctypes.byref(st)))
    return int(st.value)


def set_tile_n(block_n: int) -> None:
    _check(lib().nvfp4_set_tile_n(int(block_n)))
