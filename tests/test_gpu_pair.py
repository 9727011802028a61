"""GPU parity of the cluster kernels (clusters of two CTAs, 256 x 256 tiles)
against the CPU oracle, through the C ABI: the CTA pair (tcgen05 cta_group::2
MMAs, NVFP4_PAIR=1) and the multicast cluster (each CTA its own 128 x 256
tile, the B tile and its scales multicast to both, NVFP4_PAIR=2).

NVFP4_PAIR selects the cluster kernel on every call that runs whole tiles;
the shapes put the second CTA of a pair on rows past m (groups with m <= 128),
the second half of B past n (n mod 256 <= 128), M / N / K tails, batches
(l > 1), empty groups and k == 0, and compare every output with the oracle.
The failure-detection case makes every bounded wait of a pair call run out
(without any fault) and checks the status and the next call.
"""
import numpy as np
import pytest
import torch

from parity import assert_parity, block_samples

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from nvfp4_block_scaled_grouped_gb300 import build
    build.build_library()
    import nvfp4_block_scaled_grouped_gb300 as nv
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()
    return nv


@pytest.fixture(autouse=True, params=["1", "2"], ids=["pair", "mcast"])
def mode(request, nv, monkeypatch):
    monkeypatch.setenv("NVFP4_PAIR", request.param)
    monkeypatch.delenv("NVFP4_SPLIT", raising=False)
    nv.set_tile_n(256)
    yield request.param
    nv.set_tile_n(0)


def _make(sizes, seed, name="tiny"):
    from nvfp4_block_scaled_grouped_gb300 import workloads
    return workloads.make_problem(name, seed=seed, sizes=sizes)


def _run_full(nv, oracle_mod, prob, what):
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    dp = DeviceProblem.upload(prob)
    dp.run()
    torch.cuda.synchronize()
    assert nv.device_status() == 0, what
    got = dp.c_host()
    ref = oracle_mod.grouped_gemm(prob.problem_sizes, prob.A, prob.B, prob.SFA, prob.SFB)
    for g, ((m, n, k, l), c, r) in enumerate(zip(prob.problem_sizes, got, ref)):
        if m == 0 or n == 0 or l == 0:
            continue
        if k == 0:
            np.testing.assert_array_equal(c.view(np.uint16), np.zeros_like(c.view(np.uint16)), f"{what} group {g}")
            continue
        assert_parity(c, r, f"{what} group {g} {(m, n, k, l)}")
    return dp, got


def test_pair_one_tile(nv, oracle_mod):
    """One 256 x 256 tile, one k-tile: both CTAs' rows, both halves of B."""
    _run_full(nv, oracle_mod, _make([(256, 256, 256, 1)], seed=101), "one pair tile")


@pytest.mark.parametrize("sizes", [
    [(128, 256, 512, 1)],                       # the second CTA has no rows
    [(129, 256, 512, 1)],                       # the second CTA has one row
    [(300, 128, 256, 1)],                       # the second half of B lies past n
    [(256, 384, 1024, 1)],                      # a second n-tile whose second half is past n
    [(1, 32, 32, 1), (255, 96, 96, 1)],         # tails everywhere, k below one MMA
    [(17, 160, 288, 1), (0, 64, 64, 1), (513, 256, 7168, 1)],   # K tail, empty group, long K, 3 m-tiles
    [(3, 32, 0, 1), (200, 32, 7168, 1)],        # k == 0 gives zeros
])
def test_pair_edge_shapes(nv, oracle_mod, sizes):
    _run_full(nv, oracle_mod, _make(sizes, seed=len(sizes) * 7 + sizes[0][0]), f"pair {sizes}")


def test_pair_batches(nv, oracle_mod):
    """l > 1: batch b's rows start at b * m of the stacked operands; a pair
    tile of batch b reads rows of batch b + 1 past m, which are never stored.
    Each batch must match the oracle's product of that batch alone."""
    import test_gpu_batched as tb
    sizes = [(100, 256, 512, 3), (300, 160, 256, 2), (0, 64, 64, 4), (256, 256, 256, 2), (1, 32, 32, 5)]
    groups = tb._batched(nv, sizes, seed=5)
    cols = list(zip(*[(A, B, SFA, SFB, C) for (_, A, B, SFA, SFB, C) in groups]))
    nv.grouped_gemm_tensors(sizes, *cols)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    tb._check(oracle_mod, sizes, groups, "pair batches")


def test_pair_random_shapes(nv, oracle_mod):
    rng = np.random.default_rng(2026)
    for call in range(6):
        G = int(rng.choice([1, 3, 8, 20, 70]))
        sizes = []
        for _ in range(G):
            r = rng.random()
            m = 0 if r < 0.08 else int(rng.integers(1, 600))
            n = 32 * int(rng.integers(1, 13))
            k = 0 if 0.08 <= r < 0.12 else 32 * int(rng.integers(1, 25))
            sizes.append((m, n, k, 1))
        _run_full(nv, oracle_mod, _make(sizes, seed=9000 + call), f"pair random call {call}")


def test_pair_many_waves_and_descriptor_reuse(nv, oracle_mod, mode):
    """More tiles than pairs (several tiles per pair), run twice (cached
    descriptors), then once through the one-CTA kernel on the same buffers
    (the B descriptor box changes) and once more as a pair."""
    sizes = [(1024, 2048, 1024, 1), (700, 1024, 512, 1), (64, 4096, 256, 1)]
    prob = _make(sizes, seed=77)
    dp, first = _run_full(nv, oracle_mod, prob, "pair many waves")
    dp.run()
    torch.cuda.synchronize()
    for g, c in enumerate(dp.c_host()):
        np.testing.assert_array_equal(c.view(np.uint16), first[g].view(np.uint16), f"repeat group {g}")
    import os
    os.environ["NVFP4_PAIR"] = "0"
    try:
        dp.run()
        torch.cuda.synchronize()
        one = dp.c_host()
    finally:
        os.environ["NVFP4_PAIR"] = mode
    ref = oracle_mod.grouped_gemm(prob.problem_sizes, prob.A, prob.B, prob.SFA, prob.SFB)
    for g, (c, r) in enumerate(zip(one, ref)):
        assert_parity(c, r, f"one-CTA kernel on the same buffers, group {g}")
    dp.run()
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    for g, c in enumerate(dp.c_host()):
        np.testing.assert_array_equal(c.view(np.uint16), first[g].view(np.uint16), f"pair again, group {g}")


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_pair_full_size_sampled(nv, oracle_mod, name):
    from nvfp4_block_scaled_grouped_gb300 import workloads
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    prob = workloads.make_problem(name)
    dp = DeviceProblem.upload(prob)
    dp.run()
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    got = dp.c_host()
    rng = np.random.default_rng(31)
    for g, (m, n, k, _) in enumerate(prob.problem_sizes):
        c = got[g]
        assert not np.isnan(c.astype(np.float32)).any(), f"{name} group {g}"
        rows, cols = block_samples(rng, m, n)
        ref = oracle_mod.gemm_sampled(m, n, k, prob.A[g], prob.B[g], prob.SFA[g], prob.SFB[g], rows, cols)
        assert_parity(c[rows, cols], ref, f"pair {name} group {g}")


def test_pair_bounded_waits_give_up_and_the_context_recovers(nv, oracle_mod, monkeypatch):
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    sizes = [(700, 1024, 2048, 1), (100, 512, 1024, 1)]
    prob = _make(sizes, seed=13)
    dp = DeviceProblem.upload(prob)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    monkeypatch.setenv("NVFP4_WATCHDOG_MS", "0.0002")      # 200 ns: every wait gives up
    dp.run()
    torch.cuda.synchronize()                                 # the kernel returned on its own
    assert nv.device_status() == -5                          # NVFP4_ERR_TIMEOUT
    assert nv.device_status() == 0
    monkeypatch.delenv("NVFP4_WATCHDOG_MS")
    for c in dp.C:
        c.fill_(float("nan"))
    dp.run()
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    ref = oracle_mod.grouped_gemm(prob.problem_sizes, prob.A, prob.B, prob.SFA, prob.SFB)
    for g, (c, r) in enumerate(zip(dp.c_host(), ref)):
        assert_parity(c, r, f"after the timed-out pair call, group {g}")
