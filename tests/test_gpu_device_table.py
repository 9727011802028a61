"""GPU parity of nvfp4_grouped_gemm_device (group table in device memory)
against the CPU oracle, its CUDA-graph replay with changing sizes and
pointers, and its device-side group validation.
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


@pytest.fixture(autouse=True)
def _reset(nv, monkeypatch):
    monkeypatch.delenv("NVFP4_SPLIT", raising=False)
    yield
    nv.set_tile_n(0)


def _make(sizes, seed, name="tiny"):
    from nvfp4_block_scaled_grouped_gb300 import workloads
    return workloads.make_problem(name, seed=seed, sizes=sizes)


def _upload(prob):
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    return DeviceProblem.upload(prob)


def _table(nv, dp):
    t = nv.DeviceGroupTable(len(dp.problem_sizes))
    t.set(dp.problem_sizes, dp.A, dp.B, dp.SFA, dp.SFB, dp.C)
    return t


def _check_full(oracle_mod, prob, got, what):
    ref = oracle_mod.grouped_gemm(prob.problem_sizes, prob.A, prob.B, prob.SFA, prob.SFB)
    for g, ((m, n, k, _), c, r) in enumerate(zip(prob.problem_sizes, got, ref)):
        if m == 0 or n == 0:
            continue
        if k == 0:
            np.testing.assert_array_equal(c.view(np.uint16), np.zeros((m, n), np.uint16))
            continue
        assert_parity(c, r, f"{what} group {g} {(m, n, k)}")


EDGE_SIZES = [
    (1, 32, 32, 1), (129, 96, 96, 1), (17, 160, 288, 1), (0, 64, 64, 1), (256, 256, 512, 1),
    (3, 32, 0, 1), (130, 384, 1024, 1), (64, 0, 256, 1), (200, 32, 7168, 1),
]


@pytest.mark.parametrize("block_n,split", [(128, None), (256, None), (256, "1"), (128, "0"), (256, "2")])
def test_device_table_edge_shapes(nv, oracle_mod, monkeypatch, block_n, split):
    """The kernel reads sizes and pointers from device memory, derives the tile
    counts, prefix sums and the schedule itself (split forced either way or
    left to its rule) and matches the oracle on every edge shape."""
    if split is not None:
        monkeypatch.setenv("NVFP4_SPLIT", split)
    nv.set_tile_n(block_n)
    prob = _make(EDGE_SIZES, seed=41)
    dp = _upload(prob)
    _table(nv, dp).run()
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    _check_full(oracle_mod, prob, dp.c_host(), "device table")


@pytest.mark.parametrize("name", ["decode", "zipf64"])
def test_device_table_full_size_sampled(nv, oracle_mod, name):
    from nvfp4_block_scaled_grouped_gb300 import workloads
    prob = workloads.make_problem(name)
    dp = _upload(prob)
    _table(nv, dp).run()
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    got = dp.c_host()
    rng = np.random.default_rng(5)
    for g, (m, n, k, _) in enumerate(prob.problem_sizes):
        if m == 0 or n == 0:
            continue
        c = got[g]
        assert not np.isnan(c.astype(np.float32)).any(), f"{name} group {g}"
        rows, cols = block_samples(rng, m, n)
        ref = oracle_mod.gemm_sampled(m, n, k, prob.A[g], prob.B[g], prob.SFA[g], prob.SFB[g], rows, cols)
        assert_parity(c[rows, cols], ref, f"{name} group {g}")
    # the host-table entry point gives the same bits (same kernel, same schedule rule)
    host = [torch.full_like(c, float("nan")) for c in dp.C]
    nv.grouped_gemm_tensors(dp.problem_sizes, dp.A, dp.B, dp.SFA, dp.SFB, host)
    torch.cuda.synchronize()
    for g, (c, h) in enumerate(zip(got, host)):
        np.testing.assert_array_equal(c.view(np.uint16), h.cpu().numpy().view(np.uint16), err_msg=f"group {g}")


def test_graph_replay_with_new_sizes_and_pointers(nv, oracle_mod):
    """Capture one device-table call in a CUDA graph, then replay it after
    rewriting the device arrays: other m per group (including 0), other
    buffers, and host-table calls on the capturing stream in between (which
    rewrite the shared descriptor slots). Every replay matches the oracle."""
    G, n, k = 4, 256, 512
    big = _make([(300, n, k, 1)] * G, seed=51)
    dp = _upload(big)
    alt = _upload(_make([(300, n, k, 1)] * G, seed=52))
    table = nv.DeviceGroupTable(G)
    s = torch.cuda.Stream()

    def prob_for(base, ms):
        from nvfp4_block_scaled_grouped_gb300.workloads import GroupedProblem
        return GroupedProblem("replay", 0, [(ms[g], n, k, 1) for g in range(G)],
                              [base.A[g][: ms[g]] for g in range(G)], list(base.B),
                              [base.SFA[g][: ms[g]] for g in range(G)], list(base.SFB))

    table.set(dp.problem_sizes, dp.A, dp.B, dp.SFA, dp.SFB, dp.C)
    torch.cuda.synchronize()
    table.run(stream=s)            # allocates the stream's workspace before capture
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        table.run(stream=s)
    torch.cuda.synchronize()

    base_probs = {"dp": big, "alt": _make([(300, n, k, 1)] * G, seed=52)}
    for step, (which, ms) in enumerate([("dp", [300, 300, 300, 300]), ("dp", [7, 0, 129, 256]),
                                        ("alt", [128, 1, 0, 300]), ("dp", [0, 0, 0, 33])]):
        src = dp if which == "dp" else alt
        prob = prob_for(base_probs[which], ms)
        # group g uses the first ms[g] rows of its buffers, with its scales
        # packed for that row count
        sfa = [nv.pack_scales_tensor(torch.from_numpy(np.ascontiguousarray(prob.SFA[g])).cuda(), k)
               if ms[g] > 0 else src.SFA[g] for g in range(G)]
        A = [src.A[g][: ms[g]] for g in range(G)]
        C = [torch.full((ms[g], n), 0x7E00, dtype=torch.int16, device="cuda").view(torch.float16) for g in range(G)]
        table.set(prob.problem_sizes, A, src.B, sfa, src.SFB, C)
        if step == 2:
            # a host-table call on the capturing stream rewrites the descriptor slots
            other = _upload(_make([(77, 128, 256, 1), (5, 64, 512, 1)], seed=53))
            torch.cuda.synchronize()
            other.run(stream=s)
            s.synchronize()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert nv.device_status(s) == 0
        got = [c.cpu().numpy() for c in C]
        _check_full(oracle_mod, prob, got, f"replay {step}")


def test_host_table_capture_survives_slot_reuse(nv, oracle_mod):
    """A captured host-table call patches every descriptor on each replay, so
    other calls that reuse the workspace's descriptor slots between replays
    cannot leave it with stale ones."""
    s = torch.cuda.Stream()
    p1 = _make([(100, 256, 512, 1), (33, 128, 256, 1)], seed=61)
    p2 = _make([(64, 96, 768, 1), (200, 64, 256, 1)], seed=62)
    d1, d2 = _upload(p1), _upload(p2)
    torch.cuda.synchronize()
    d1.run(stream=s)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        d1.run(stream=s)
    for _ in range(2):
        d2.run(stream=s)            # same slot indices, other pointers and shapes
        s.synchronize()
        for c in d1.C:
            c.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        _check_full(oracle_mod, p1, d1.c_host(), "captured host-table call")
    _check_full(oracle_mod, p2, d2.c_host(), "interleaved call")
    assert nv.device_status(s) == 0


def test_device_table_rejects_bad_groups_on_device(nv, oracle_mod):
    """Groups that break the rules (l > 65535, k % 32 != 0, misaligned C) are
    skipped by the kernel -- their C untouched -- while the valid groups are
    computed; the stream's status then reports NVFP4_ERR_INVALID_ARG."""
    sizes = [(40, 64, 256, 1), (16, 64, 256, 70000), (70, 96, 256, 1), (8, 32, 48, 1), (9, 64, 256, 1)]
    prob = _make([(40, 64, 256, 1), (16, 64, 256, 1), (70, 96, 256, 1), (8, 32, 64, 1), (9, 64, 256, 1)],
                 seed=71)
    dp = _upload(prob)
    # group 4: C one fp16 element into its buffer (2-byte aligned only)
    c4 = torch.full((9 * 64 + 8,), 0x7E00, dtype=torch.int16, device="cuda").view(torch.float16)
    C = list(dp.C)
    C[4] = c4[1:]
    table = nv.DeviceGroupTable(len(sizes))
    table.set(sizes, dp.A, dp.B, dp.SFA, dp.SFB, C)
    table.run()
    torch.cuda.synchronize()
    assert nv.device_status() == nv_status(nv, "NVFP4_ERR_INVALID_ARG")
    assert nv.device_status() == 0  # read and cleared
    ref = oracle_mod.grouped_gemm(prob.problem_sizes, prob.A, prob.B, prob.SFA, prob.SFB)
    for g in (0, 2):
        assert_parity(dp.C[g].cpu().numpy(), ref[g], f"valid group {g}")
    for g in (1, 3):
        assert np.all(dp.C[g].cpu().numpy().view(np.uint16) == 0x7E00), f"skipped group {g} was written"
    assert np.all(c4.cpu().numpy().view(np.uint16) == 0x7E00), "misaligned group was written"


def nv_status(nv, name):
    return {v: k for k, v in nv.STATUS.items()}[name]


def test_device_table_host_argument_errors(nv):
    """What the host can check is rejected before anything is enqueued."""
    sizes = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    ptrs = torch.zeros((5, 2), dtype=torch.int64, device="cuda")
    p = [ptrs[i].data_ptr() for i in range(5)]
    assert nv.grouped_gemm_device(0, 0, 0, 0, 0, 0, 0, check=False) == 0
    assert nv.grouped_gemm_device(-1, sizes.data_ptr(), *p, check=False) == nv_status(nv, "NVFP4_ERR_INVALID_ARG")
    assert nv.grouped_gemm_device(513, sizes.data_ptr(), *p, check=False) == nv_status(nv, "NVFP4_ERR_INVALID_ARG")
    assert nv.grouped_gemm_device(2, 0, *p, check=False) == nv_status(nv, "NVFP4_ERR_INVALID_ARG")
    assert nv.grouped_gemm_device(2, sizes.data_ptr() + 4, *p, check=False) == nv_status(nv, "NVFP4_ERR_MISALIGNED")
