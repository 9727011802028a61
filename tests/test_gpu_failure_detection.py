"""Failure detection on the GPU without a fault: every wait in the GEMM
kernel is bounded. With the bound set shorter than any TMA round trip, the
kernel's waits give up, it sets its status word and returns (its copies and
MMAs drained, TMEM freed), nvfp4_device_status reports NVFP4_ERR_TIMEOUT, and
the context stays usable: the next call with the normal bound completes and
matches the oracle."""
import numpy as np
import pytest
import torch

from parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from nvfp4_block_scaled_grouped_gb300 import build
    build.build_library()
    import nvfp4_block_scaled_grouped_gb300 as nv
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()
    return nv


def _status(nv, name):
    return {v: k for k, v in nv.STATUS.items()}[name]


@pytest.mark.parametrize("workload,split,api", [("decode", None, "host"), ("decode", "0", "host"),
                                                ("tiny", None, "host"), ("decode", None, "device")])
def test_bounded_waits_give_up_and_the_context_recovers(nv, oracle_mod, monkeypatch, workload, split, api):
    from nvfp4_block_scaled_grouped_gb300 import workloads
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    if split is not None:
        monkeypatch.setenv("NVFP4_SPLIT", split)
    prob = workloads.make_problem(workload)
    dp = DeviceProblem.upload(prob)
    table = None
    if api == "device":
        table = nv.DeviceGroupTable(len(dp.problem_sizes))
        table.set(dp.problem_sizes, dp.A, dp.B, dp.SFA, dp.SFB, dp.C)
    run = (lambda: table.run()) if table else (lambda: dp.run())
    torch.cuda.synchronize()
    assert nv.device_status() == 0

    monkeypatch.setenv("NVFP4_WATCHDOG_MS", "0.0002")      # 200 ns
    run()
    torch.cuda.synchronize()                                 # the kernel returned on its own
    assert nv.device_status() == _status(nv, "NVFP4_ERR_TIMEOUT")
    assert nv.device_status() == 0                           # read and cleared

    monkeypatch.delenv("NVFP4_WATCHDOG_MS")
    for c in dp.C:
        c.fill_(float("nan"))
    run()
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    rng = np.random.default_rng(3)
    for g, ((m, n, k, _), c) in enumerate(zip(prob.problem_sizes, dp.c_host())):
        if m == 0 or n == 0:
            continue
        rows = rng.integers(0, m, 256).astype(np.int32)
        cols = rng.integers(0, n, 256).astype(np.int32)
        ref = oracle_mod.gemm_sampled(m, n, k, prob.A[g], prob.B[g], prob.SFA[g], prob.SFB[g], rows, cols)
        assert_parity(c[rows, cols], ref, f"{workload} group {g} after the timed-out call")
        assert not np.isnan(c.astype(np.float32)).any()
