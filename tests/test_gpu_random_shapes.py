"""Randomised grouped calls against the CPU oracle: seeded random group
counts and shapes (m, n, k, l, including empty groups, K tails and M / N
tails), through both entry points and both schedules, at the group counts
that select each kernel-parameter capacity (8, 64, 512)."""
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


@pytest.fixture(autouse=True)
def _reset(nv, monkeypatch):
    monkeypatch.delenv("NVFP4_SPLIT", raising=False)
    yield
    nv.set_tile_n(0)


def _random_sizes(rng, groups, max_m, max_n, max_k, max_l):
    sizes = []
    for _ in range(groups):
        r = rng.random()
        m = 0 if r < 0.08 else int(rng.integers(1, max_m + 1))
        n = 0 if 0.08 <= r < 0.12 else 32 * int(rng.integers(1, max_n // 32 + 1))
        k = 0 if 0.12 <= r < 0.15 else 32 * int(rng.integers(1, max_k // 32 + 1))
        l = int(rng.integers(1, max_l + 1)) if rng.random() < 0.3 else 1
        sizes.append((m, n, k, l))
    return sizes


def _upload_batched(nv, sizes, seed):
    """Stacked operands (batch-outermost) per group, plus each batch's problem."""
    from nvfp4_block_scaled_grouped_gb300 import workloads
    per_group, dev = [], []
    empty = lambda: torch.empty(0, dtype=torch.uint8, device="cuda")
    for g, (m, n, k, l) in enumerate(sizes):
        batches = [workloads.make_problem("tiny", seed=seed * 7919 + 31 * g + b, sizes=[(m, n, k, 1)])
                   for b in range(max(l, 1))]
        live = m > 0 and n > 0
        cat = lambda xs: torch.from_numpy(np.ascontiguousarray(np.concatenate(xs))).cuda() if live and k else empty()
        pack = lambda sf, rows: nv.pack_scales_tensor(torch.from_numpy(np.ascontiguousarray(sf)).cuda(), k)
        A = cat([p.A[0] for p in batches])
        B = cat([p.B[0] for p in batches])
        SFA = torch.cat([pack(p.SFA[0], m) for p in batches]) if live and k else empty()
        SFB = torch.cat([pack(p.SFB[0], n) for p in batches]) if live and k else empty()
        C = torch.full((max(m * l, 1), max(n, 1)), 0x7E00, dtype=torch.int16, device="cuda").view(torch.float16)
        per_group.append(batches)
        dev.append((A, B, SFA, SFB, C))
    return per_group, dev


def _check(oracle_mod, sizes, per_group, dev, what):
    for g, ((m, n, k, l), batches, (_, _, _, _, C)) in enumerate(zip(sizes, per_group, dev)):
        c = C.cpu().numpy()
        if m == 0 or n == 0:
            assert np.all(c.view(np.uint16) == 0x7E00), f"{what}: empty group {g} was written"
            continue
        c = c.reshape(l, m, n)
        for b, p in enumerate(batches):
            if k == 0:
                np.testing.assert_array_equal(c[b].view(np.uint16), np.zeros((m, n), np.uint16))
                continue
            ref = oracle_mod.grouped_gemm(p.problem_sizes, p.A, p.B, p.SFA, p.SFB)[0]
            assert_parity(c[b], ref, f"{what} group {g} batch {b} {(m, n, k, l)}")


CASES = [  # (seed, groups, max_m, max_n, max_k, max_l)
    (1, 5, 300, 512, 1024, 3),
    (2, 8, 140, 384, 2048, 2),
    (3, 40, 96, 256, 512, 2),
    (4, 100, 40, 128, 256, 1),
    (5, 512, 24, 64, 128, 1),   # the largest call: NVFP4_MAX_GROUPS groups
]


@pytest.mark.parametrize("case", CASES, ids=[f"seed{c[0]}-G{c[1]}" for c in CASES])
@pytest.mark.parametrize("api,block_n,split", [("host", 256, None), ("host", 128, "1"), ("device", 256, "1"),
                                               ("device", 128, "0"), ("host", 256, "2"), ("device", 256, "2")])
def test_random_grouped_calls(nv, oracle_mod, monkeypatch, case, api, block_n, split):
    seed, groups, max_m, max_n, max_k, max_l = case
    if split is not None:
        monkeypatch.setenv("NVFP4_SPLIT", split)
    nv.set_tile_n(block_n)
    rng = np.random.default_rng(seed)
    sizes = _random_sizes(rng, groups, max_m, max_n, max_k, max_l)
    per_group, dev = _upload_batched(nv, sizes, seed)
    cols = list(zip(*dev))
    if api == "host":
        nv.grouped_gemm_tensors(sizes, *cols)
    else:
        t = nv.DeviceGroupTable(len(sizes))
        t.set(sizes, *cols)
        t.run()
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    _check(oracle_mod, sizes, per_group, dev, f"{api} BN={block_n} split={split} seed={seed}")


@pytest.mark.parametrize("extra_tiles", [1, 8])
@pytest.mark.parametrize("api", ["host", "device"])
def test_split_remainder_smaller_than_the_grid(nv, oracle_mod, monkeypatch, extra_tiles, api):
    """Whole waves plus a split remainder (forced) whose schedule units are
    fewer than the CTAs: the remainder must go to as many CTAs as it has
    units, each finishing CTA waiting only for CTAs that hold a piece."""
    monkeypatch.setenv("NVFP4_SPLIT", "2")
    nv.set_tile_n(256)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    m, n, k = 128 * (sms + extra_tiles), 256, 512          # sms + extra tiles of 2 k-tiles each
    from nvfp4_block_scaled_grouped_gb300 import workloads
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    prob = workloads.make_problem("tiny", seed=500 + extra_tiles, sizes=[(m, n, k, 1)])
    dp = DeviceProblem.upload(prob)
    if api == "host":
        dp.run()
    else:
        t = nv.DeviceGroupTable(1)
        t.set(dp.problem_sizes, dp.A, dp.B, dp.SFA, dp.SFB, dp.C)
        t.run()
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    c = dp.c_host()[0]
    rows = np.concatenate([np.arange(m - 128 * extra_tiles, m), np.random.default_rng(1).integers(0, m, 512)])
    rows = rows.astype(np.int32)
    cols = np.random.default_rng(2).integers(0, n, rows.size).astype(np.int32)
    ref = oracle_mod.gemm_sampled(m, n, k, prob.A[0], prob.B[0], prob.SFA[0], prob.SFB[0], rows, cols)
    assert_parity(c[rows, cols], ref, f"remainder of {extra_tiles} tiles")
