"""nvfp4_grouped_gemm_noalloc: the grouped GEMM for callers that cannot
allocate device memory (frameworks that own every byte of device memory
through their own arena, latency-critical callers that cannot take a
cudaMalloc, which may synchronise the device, in the middle of their work).
Its scratch is a fixed array inside the library instead of a cudaMalloc'd
buffer, so the results must be those of nvfp4_grouped_gemm.

The checks, through the C ABI: two calls in a row with different problems
(the second call sees the array holding the first call's contents), each
compared with the CPU oracle and with nvfp4_grouped_gemm on the same inputs
within the parity tolerance; a call with the largest group count the array
holds (64 groups, empty and tail groups among them) against the oracle; a
call whose bounded waits run out is reported by nvfp4_device_status and the
next call is correct; and the host-side rejection of a group count above
the limit. Collected last so a stop-at-first-failure run has already run the
rest.
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
    L.nvfp4_device_status.restype = ctypes.c_int
    L.nvfp4_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
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


def _status(L):
    st = ctypes.c_int(99)
    assert L.nvfp4_device_status(ctypes.c_void_p(int(torch.cuda.current_stream().cuda_stream) or None),
                                 ctypes.byref(st)) == 0
    return st.value


def _check_oracle(oracle_mod, prob, got, what):
    ref = oracle_mod.grouped_gemm(prob.problem_sizes, prob.A, prob.B, prob.SFA, prob.SFB)
    for g, (m, n, k, _) in enumerate(prob.problem_sizes):
        c = got.C[g].cpu().numpy()
        if m == 0 or n == 0:
            assert c.size == 0
            continue
        assert_parity(c, ref[g], f"{what} group {g} {(m, n, k)}")


def test_noalloc_matches_oracle_and_grouped_gemm_on_two_calls_in_a_row(L, oracle_mod):
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    stream = torch.cuda.current_stream()
    for call, sizes in enumerate(CALLS):
        prob = _problem(sizes, seed=40 + call)
        ref = DeviceProblem.upload(prob)
        ref.run(stream)
        got = DeviceProblem.upload(prob)   # fresh C buffers holding the NaN sentinel
        assert _noalloc(L, got, stream) == 0, L.nvfp4_last_error_message().decode()
        torch.cuda.synchronize()
        assert _status(L) == 0
        _check_oracle(oracle_mod, prob, got, f"call {call}")
        for g, (m, n, k, _) in enumerate(sizes):
            c_ref, c_got = ref.C[g].cpu().numpy(), got.C[g].cpu().numpy()
            if m == 0 or n == 0:
                continue
            assert_parity(c_got, c_ref, f"call {call} group {g} vs nvfp4_grouped_gemm")


def test_noalloc_64_groups(L, oracle_mod):
    """The largest call the array holds: 64 groups (descriptor slots up to
    the end of the array), with empty groups, k == 0, and M / N / K tails."""
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    rng = np.random.default_rng(64)
    sizes = []
    for g in range(64):
        m = 0 if g % 13 == 5 else int(rng.choice([1, 17, 64, 128, 129, 200, 300]))
        n = 32 * int(rng.integers(1, 13))
        k = 0 if g % 17 == 3 else 32 * int(rng.integers(1, 20))
        sizes.append((m, n, k, 1))
    prob = _problem(sizes, seed=64)
    got = DeviceProblem.upload(prob)
    stream = torch.cuda.current_stream()
    assert _noalloc(L, got, stream) == 0, L.nvfp4_last_error_message().decode()
    torch.cuda.synchronize()
    assert _status(L) == 0
    for g, (m, n, k, _) in enumerate(sizes):
        if m and n and k == 0:
            np.testing.assert_array_equal(got.C[g].cpu().numpy().view(np.uint16), np.zeros((m, n), np.uint16))
    _check_oracle(oracle_mod, prob, got, "64 groups")


def test_noalloc_timeout_is_reported_and_the_next_call_is_correct(L, oracle_mod, monkeypatch):
    """A bounded wait that runs out inside a no-alloc call (the bound set to
    200 ns, shorter than any copy) is reported by nvfp4_device_status; the
    next call with the normal bound matches the oracle."""
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    prob = _problem(CALLS[0], seed=77)
    got = DeviceProblem.upload(prob)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    assert _status(L) == 0
    monkeypatch.setenv("NVFP4_WATCHDOG_MS", "0.0002")
    assert _noalloc(L, got, stream) == 0
    torch.cuda.synchronize()
    assert _status(L) == -5      # NVFP4_ERR_TIMEOUT
    assert _status(L) == 0       # read and cleared
    monkeypatch.delenv("NVFP4_WATCHDOG_MS")
    for c in got.C:
        c.fill_(float("nan"))
    assert _noalloc(L, got, stream) == 0
    torch.cuda.synchronize()
    assert _status(L) == 0
    _check_oracle(oracle_mod, prob, got, "after the timed-out call")


def test_noalloc_rejects_more_groups_than_its_workspace(L):
    import nvfp4_block_scaled_grouped_gb300 as nv
    G = 65
    sizes = (nv.ProblemSize * G)(*[nv.ProblemSize(4, 64, 64, 1)] * G)
    ptrs = (ctypes.c_void_p * G)(*[0x10000] * G)
    assert L.nvfp4_grouped_gemm_noalloc(G, sizes, ptrs, ptrs, ptrs, ptrs, ptrs, None) == -1
    assert b"64" in L.nvfp4_last_error_message()
