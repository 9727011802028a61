"""nvfp4_grouped_gemm_noalloc: the grouped GEMM for callers that cannot
allocate device memory (frameworks that own every byte of device memory
through their own arena, latency-critical callers that cannot take a
cudaMalloc, which may synchronise the device, in the middle of their work).
Its scratch is a fixed array inside the library instead of a cudaMalloc'd
buffer, so the results must be those of nvfp4_grouped_gemm.

The check: through the C ABI, two calls in a row with different problems
(the second call sees the array holding the first call's contents), each
compared with nvfp4_grouped_gemm on the same inputs within the parity
tolerance, plus the host-side rejection of a group count above the limit.
Collected last so a stop-at-first-failure run has already run the rest.
"""
import ctypes

import numpy as np
import pytest
import torch

from parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from nvfp4_block_scaled_grouped_gb300 import build
    build.build_library()
    import nvfp4_block_scaled_grouped_gb300 as nv
    L = nv.lib()
    vpp = ctypes.POINTER(ctypes.c_void_p)
    L.nvfp4_grouped_gemm_noalloc.restype = ctypes.c_int
    L.nvfp4_grouped_gemm_noalloc.argtypes = [ctypes.c_int, ctypes.POINTER(nv.ProblemSize), vpp, vpp, vpp, vpp,
                                             vpp, ctypes.c_void_p]
    assert torch.cuda.is_available()
    return L


def _noalloc(L, dp, stream):
    import nvfp4_block_scaled_grouped_gb300 as nv
    G = len(dp.problem_sizes)
    sizes = (nv.ProblemSize * G)(*[nv.ProblemSize(*map(int, s)) for s in dp.problem_sizes])
    arr = lambda ts: (ctypes.c_void_p * G)(*[int(t.data_ptr()) if t.numel() else None for t in ts])
    return L.nvfp4_grouped_gemm_noalloc(G, sizes, arr(dp.A), arr(dp.B), arr(dp.SFA), arr(dp.SFB), arr(dp.C),
                                        ctypes.c_void_p(int(stream.cuda_stream) or None))


def _problem(sizes, seed):
    from nvfp4_block_scaled_grouped_gb300 import workloads
    return workloads.make_problem("ragged", seed=seed, sizes=sizes)


CALLS = [
    [(1, 7168, 2048, 1), (17, 7168, 2048, 1), (0, 256, 2048, 1), (333, 1024, 2048, 1), (200, 96, 288, 1)],
    [(130, 512, 1024, 1), (5, 32, 64, 1)],
]


def test_noalloc_matches_grouped_gemm_on_two_calls_in_a_row(L):
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    stream = torch.cuda.current_stream()
    for call, sizes in enumerate(CALLS):
        prob = _problem(sizes, seed=40 + call)
        ref = DeviceProblem.upload(prob)
        ref.run(stream)
        got = DeviceProblem.upload(prob)   # fresh C buffers holding the NaN sentinel
        assert _noalloc(L, got, stream) == 0, L.nvfp4_last_error_message().decode()
        torch.cuda.synchronize()
        for g, (m, n, k, _) in enumerate(sizes):
            c_ref, c_got = ref.C[g].cpu().numpy(), got.C[g].cpu().numpy()
            if m == 0 or n == 0:
                assert c_got.size == 0
                continue
            assert_parity(c_got, c_ref, f"call {call} group {g}")


def test_noalloc_rejects_more_groups_than_its_workspace(L):
    import nvfp4_block_scaled_grouped_gb300 as nv
    G = 65
    sizes = (nv.ProblemSize * G)(*[nv.ProblemSize(4, 64, 64, 1)] * G)
    ptrs = (ctypes.c_void_p * G)(*[0x10000] * G)
    assert L.nvfp4_grouped_gemm_noalloc(G, sizes, ptrs, ptrs, ptrs, ptrs, ptrs, None) == -1
    assert b"64" in L.nvfp4_last_error_message()
