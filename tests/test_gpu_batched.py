"""GPU parity of groups with l > 1 batches against the CPU oracle.

A group (m, n, k, l) holds l independent products stacked batch-outermost,
the layout of the submissions' (m, k, l) operands with strides (k, 1, m*k):
A [l*m][k/2], B [l*n][k/2], C [l*m][n], and per-batch scale-atom blocks
(nvfp4_scale_bytes(m, k) bytes each) one after another. Each batch must match
the oracle's product of that batch alone.
"""
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


SIZES = [(130, 96, 288, 3), (1, 32, 32, 5), (0, 64, 64, 2), (64, 256, 512, 2), (200, 160, 7168, 2),
         (77, 64, 0, 2), (40, 64, 256, 0), (129, 384, 1024, 1)]


def _batched(nv, sizes, seed):
    """Per group: the l batch problems (host, row-major scales) and the stacked
    device buffers."""
    from nvfp4_block_scaled_grouped_gb300 import workloads
    groups = []
    for g, (m, n, k, l) in enumerate(sizes):
        batches = [workloads.make_problem("tiny", seed=seed * 1000 + 10 * g + b, sizes=[(m, n, k, 1)])
                   for b in range(l)]
        dev = lambda arrs: torch.from_numpy(np.ascontiguousarray(np.concatenate(arrs))).cuda() if arrs else None
        A = dev([p.A[0] for p in batches]) if l else torch.empty(0, dtype=torch.uint8, device="cuda")
        B = dev([p.B[0] for p in batches]) if l else torch.empty(0, dtype=torch.uint8, device="cuda")
        pack = lambda sf, rows: (nv.pack_scales_tensor(torch.from_numpy(np.ascontiguousarray(sf)).cuda(), k)
                                 if rows > 0 and k > 0 else torch.empty(0, dtype=torch.uint8, device="cuda"))
        SFA = torch.cat([pack(p.SFA[0], m) for p in batches]) if l else torch.empty(0, dtype=torch.uint8,
                                                                                     device="cuda")
        SFB = torch.cat([pack(p.SFB[0], n) for p in batches]) if l else torch.empty(0, dtype=torch.uint8,
                                                                                     device="cuda")
        C = torch.full((max(l * m, 0), n), 0x7E00, dtype=torch.int16, device="cuda").view(torch.float16)
        groups.append((batches, A, B, SFA, SFB, C))
    return groups


def _check(oracle_mod, sizes, groups, what):
    for g, ((m, n, k, l), (batches, _, _, _, _, C)) in enumerate(zip(sizes, groups)):
        if m == 0 or n == 0 or l == 0:
            continue
        c = C.cpu().numpy().reshape(l, m, n)
        for b, p in enumerate(batches):
            if k == 0:
                np.testing.assert_array_equal(c[b].view(np.uint16), np.zeros((m, n), np.uint16))
                continue
            ref = oracle_mod.grouped_gemm(p.problem_sizes, p.A, p.B, p.SFA, p.SFB)[0]
            assert_parity(c[b], ref, f"{what} group {g} batch {b} {(m, n, k, l)}")


@pytest.mark.parametrize("api", ["host", "device"])
@pytest.mark.parametrize("block_n,split", [(128, "0"), (256, "0"), (256, "1"), (128, None)])
def test_batched_groups(nv, oracle_mod, monkeypatch, api, block_n, split):
    if split is not None:
        monkeypatch.setenv("NVFP4_SPLIT", split)
    nv.set_tile_n(block_n)
    groups = _batched(nv, SIZES, seed=7)
    cols = list(zip(*[(A, B, SFA, SFB, C) for (_, A, B, SFA, SFB, C) in groups]))
    if api == "host":
        nv.grouped_gemm_tensors(SIZES, *cols)
    else:
        t = nv.DeviceGroupTable(len(SIZES))
        t.set(SIZES, *cols)
        t.run()
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    _check(oracle_mod, SIZES, groups, f"{api} BN={block_n} split={split}")


@pytest.mark.parametrize("split", ["0", None])
def test_several_problems_in_one_launch(nv, oracle_mod, monkeypatch, split):
    """nvfp4_grouped_gemm_batched over three independent grouped problems
    matches the oracle per problem; with whole-tile schedules it is also
    bit-identical to one call per problem."""
    if split is not None:
        monkeypatch.setenv("NVFP4_SPLIT", split)
    from nvfp4_block_scaled_grouped_gb300 import workloads
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    shapes = [[(100, 256, 512, 1), (7, 128, 256, 1)], [(0, 64, 64, 1), (300, 96, 1024, 1)],
              [(64, 512, 768, 1), (1, 32, 32, 1), (129, 160, 256, 1)]]
    probs = [workloads.make_problem("tiny", seed=90 + i, sizes=s) for i, s in enumerate(shapes)]
    dps = [DeviceProblem.upload(p) for p in probs]
    ptr = lambda t: 0 if t.numel() == 0 else int(t.data_ptr())
    args = [(dp.problem_sizes, [ptr(t) for t in dp.A], [ptr(t) for t in dp.B], [ptr(t) for t in dp.SFA],
             [ptr(t) for t in dp.SFB], [ptr(t) for t in dp.C]) for dp in dps]
    nv.grouped_gemm_batched(args)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    together = [dp.c_host() for dp in dps]
    for p, (prob, got) in enumerate(zip(probs, together)):
        ref = oracle_mod.grouped_gemm(prob.problem_sizes, prob.A, prob.B, prob.SFA, prob.SFB)
        for g, ((m, n, k, _), c, r) in enumerate(zip(prob.problem_sizes, got, ref)):
            if m and n:
                assert_parity(c, r, f"problem {p} group {g}")
    if split == "0":
        for dp in dps:
            for c in dp.C:
                c.fill_(float("nan"))
            dp.run()
        torch.cuda.synchronize()
        for p, dp in enumerate(dps):
            for g, (c, t) in enumerate(zip(dp.c_host(), together[p])):
                np.testing.assert_array_equal(c.view(np.uint16), t.view(np.uint16), err_msg=f"problem {p} group {g}")


def test_scale_descriptor_follows_batch_layout_over_the_same_buffers(nv, oracle_mod):
    """The same B and SFB buffers read first as one batch of n = 256 rows and
    then as l = 4 batches of n = 64 (the same l*n, but 4 instead of 2 blocks of
    128 scale rows): the cached SFB descriptor must be patched again."""
    from nvfp4_block_scaled_grouped_gb300 import workloads
    k, m = 256, 64
    one = workloads.make_problem("tiny", seed=77, sizes=[(m, 256, k, 1)])
    B = torch.from_numpy(np.ascontiguousarray(one.B[0])).cuda()
    sf_rows = one.SFB[0]                                       # [256][k/16] row-major
    sfb = torch.zeros(4 * nv.scale_bytes(64, k), dtype=torch.uint8, device="cuda")
    packed1 = nv.pack_scales_tensor(torch.from_numpy(np.ascontiguousarray(sf_rows)).cuda(), k)
    sfb[: packed1.numel()].copy_(packed1)
    A1 = torch.from_numpy(np.ascontiguousarray(one.A[0])).cuda()
    SFA1 = nv.pack_scales_tensor(torch.from_numpy(np.ascontiguousarray(one.SFA[0])).cuda(), k)
    C1 = torch.full((m, 256), float("nan"), dtype=torch.float16, device="cuda")
    nv.grouped_gemm_tensors([(m, 256, k, 1)], [A1], [B], [SFA1], [sfb], [C1])
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    ref1 = oracle_mod.grouped_gemm(one.problem_sizes, one.A, one.B, one.SFA, one.SFB)[0]
    assert_parity(C1.cpu().numpy(), ref1, "n = 256, l = 1")

    # the same buffers as 4 batches of 64 rows of B (batch b: rows 64b .. 64b+63)
    sfb.copy_(torch.cat([nv.pack_scales_tensor(torch.from_numpy(np.ascontiguousarray(sf_rows[64 * b: 64 * b + 64]))
                                               .cuda(), k) for b in range(4)]))
    batches = [workloads.make_problem("tiny", seed=80 + b, sizes=[(m, 64, k, 1)]) for b in range(4)]
    A4 = torch.from_numpy(np.ascontiguousarray(np.concatenate([p.A[0] for p in batches]))).cuda()
    SFA4 = torch.cat([nv.pack_scales_tensor(torch.from_numpy(np.ascontiguousarray(p.SFA[0])).cuda(), k)
                      for p in batches])
    C4 = torch.full((4 * m, 64), float("nan"), dtype=torch.float16, device="cuda")
    nv.grouped_gemm_tensors([(m, 64, k, 4)], [A4], [B], [SFA4], [sfb], [C4])
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    c4 = C4.cpu().numpy().reshape(4, m, 64)
    for b, p in enumerate(batches):
        ref = oracle_mod.grouped_gemm([(m, 64, k, 1)], p.A, [one.B[0][64 * b: 64 * b + 64]], p.SFA,
                                      [sf_rows[64 * b: 64 * b + 64]])[0]
        assert_parity(c4[b], ref, f"l = 4 batch {b}")
