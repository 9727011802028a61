"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Small problems are compared element by element over all of C; the full-size
workloads (the five grouped-call shapes of the "nvfp4 group gemm" task) are
compared on sampled outputs plus properties that hold at any size: no NaN in
written groups, empty groups untouched, identical bits on a repeated call.
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
def _reset_tile(nv, monkeypatch):
    monkeypatch.delenv("NVFP4_SPLIT", raising=False)
    yield
    nv.set_tile_n(0)


def _schedule(monkeypatch, split):
    """split: None = library choice, True/False = force the split (stream-K)
    or whole-tile schedule."""
    if split is None:
        monkeypatch.delenv("NVFP4_SPLIT", raising=False)
    elif split == "hybrid":
        monkeypatch.setenv("NVFP4_SPLIT", "2")   # whole tiles for the full waves, the rest split
    else:
        monkeypatch.setenv("NVFP4_SPLIT", "1" if split else "0")


def _run(nv, prob, block_n=128):
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    nv.set_tile_n(block_n)
    dp = DeviceProblem.upload(prob)
    dp.run()
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    return dp, dp.c_host()


def _oracle_full(oracle_mod, prob):
    return oracle_mod.grouped_gemm(prob.problem_sizes, prob.A, prob.B, prob.SFA, prob.SFB)


def _make(sizes, seed=0, name="tiny"):
    from nvfp4_block_scaled_grouped_gb300 import workloads
    return workloads.make_problem(name, seed=seed, sizes=sizes)


# ---------------------------------------------------------------- the packer

@pytest.mark.parametrize("rows,k", [(1, 32), (128, 64), (129, 96), (300, 256), (513, 2048), (4096, 7168),
                                    (1000, 160)])
def test_pack_scales_matches_cpu_packer(nv, oracle_mod, rows, k):
    rng = np.random.default_rng(rows * 7 + k)
    sf = rng.integers(0, 256, (rows, k // 16), dtype=np.uint8)
    got = nv.pack_scales_tensor(torch.from_numpy(sf).cuda(), k).cpu().numpy()
    np.testing.assert_array_equal(got, oracle_mod.pack_scales(sf, k))


def test_batched_packer_matches_cpu_packer(nv, oracle_mod):
    """nvfp4_pack_scales_batched packs every matrix of a mixed batch (ragged
    rows, K tails, empty entries, one large matrix) byte for byte as the CPU
    packer does, padding included, in one launch."""
    shapes = [(1, 32), (0, 64), (128, 64), (129, 96), (300, 256), (5, 0), (4096, 7168), (1000, 160), (77, 16)]
    rng = np.random.default_rng(5)
    mats = [rng.integers(0, 256, (r, k // 16), dtype=np.uint8) for r, k in shapes]
    outs = nv.pack_scales_tensors([(torch.from_numpy(m).cuda(), k) for m, (_, k) in zip(mats, shapes)])
    torch.cuda.synchronize()
    for m, (r, k), out in zip(mats, shapes, outs):
        if r == 0 or k == 0:
            assert out.numel() == 0
            continue
        np.testing.assert_array_equal(out.cpu().numpy(), oracle_mod.pack_scales(m, k), err_msg=f"{(r, k)}")


# ---------------------------------------------------------------- full parity, small shapes

@pytest.mark.parametrize("block_n", [128, 256])
def test_tiny_workload_full(nv, oracle_mod, block_n):
    from nvfp4_block_scaled_grouped_gb300 import workloads
    prob = workloads.make_problem("tiny")
    _, got = _run(nv, prob, block_n)
    for g, (c, r) in enumerate(zip(got, _oracle_full(oracle_mod, prob))):
        assert_parity(c, r, f"tiny group {g}")


EDGE_SIZES = [
    (1, 32, 32, 1),        # one row, one column chunk, k below one MMA
    (129, 96, 96, 1),      # M tail (2 m-tiles), N tail inside a 128/256 tile, K tail (k-block half empty)
    (17, 160, 288, 1),     # two k-tiles, the second with one k-block
    (0, 64, 64, 1),        # empty group between non-empty ones
    (256, 256, 512, 1),    # exact tiles
    (3, 32, 0, 1),         # k == 0: C = 0
    (130, 384, 1024, 1),   # several k-tiles, N = 3 x 128
    (64, 0, 256, 1),       # empty (n == 0)
    (200, 32, 7168, 1),    # long K (28 k-tiles)
]


@pytest.mark.parametrize("block_n,split", [(128, False), (256, False), (128, True), (256, True), (256, "hybrid"),
                                           (128, "hybrid")])
def test_edge_shapes_full(nv, oracle_mod, monkeypatch, block_n, split):
    """All edge shapes in one call; with the split schedule forced, the tiles
    are cut along K over many CTAs (most pieces one k-tile long), so the
    partial-tile hand-off between CTAs is exercised on every group."""
    _schedule(monkeypatch, split)
    prob = _make(EDGE_SIZES, seed=3)
    dp, got = _run(nv, prob, block_n)
    ref = _oracle_full(oracle_mod, prob)
    for g, ((m, n, k, _), c, r) in enumerate(zip(EDGE_SIZES, got, ref)):
        if m == 0 or n == 0:
            assert c.size == 0
            continue
        if k == 0:
            np.testing.assert_array_equal(c.view(np.uint16), np.zeros((m, n), np.uint16))
            continue
        assert_parity(c, r, f"edge group {g} {(m, n, k)}")


@pytest.mark.parametrize("block_n,split", [(128, False), (256, False), (256, True), (128, True)])
def test_c_16_byte_aligned_only(nv, oracle_mod, monkeypatch, block_n, split):
    """C that is 16-byte aligned (what the API requires) but not 32-byte
    aligned: the epilogue then stores 16-byte pieces instead of 32-byte ones.
    Results match the oracle on every path that stores fp16 (whole tiles in
    the main loop and as a CTA's last segment, and the finishing piece of a
    split tile), and the bytes around each C stay untouched."""
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem, SENTINEL_F16
    _schedule(monkeypatch, split)
    sizes = [(200, 320, 512, 1), (64, 256, 768, 1), (300, 512, 256, 1), (129, 96, 7168, 1)]
    prob = _make(sizes, seed=11)
    nv.set_tile_n(block_n)
    dp = DeviceProblem.upload(prob)
    bufs = []
    for g, (m, n, _k, _l) in enumerate(sizes):
        buf = torch.full((m * n + 16,), SENTINEL_F16, dtype=torch.int16, device="cuda")
        c = buf[8:8 + m * n].view(m, n).view(torch.float16)
        assert c.data_ptr() % 32 == 16
        dp.C[g] = c
        bufs.append(buf)
    dp.run()
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    ref = _oracle_full(oracle_mod, prob)
    for g, ((m, n, _k, _l), buf, r) in enumerate(zip(sizes, bufs, ref)):
        raw = buf.cpu().numpy()
        assert np.all(raw[:8].view(np.uint16) == SENTINEL_F16), f"group {g}: bytes before C written"
        assert np.all(raw[8 + m * n:].view(np.uint16) == SENTINEL_F16), f"group {g}: bytes after C written"
        assert_parity(raw[8:8 + m * n].view(np.float16).reshape(m, n), r, f"16-byte aligned C, group {g}")


def test_interior_empty_groups_keep_sentinel(nv, oracle_mod):
    """Empty groups between non-empty ones get no tiles and keep their C; the
    tiles of the neighbours land in the right group."""
    sizes = [(40, 64, 256, 1), (0, 64, 256, 1), (0, 96, 256, 1), (70, 96, 256, 1), (0, 32, 256, 1),
             (5, 128, 256, 1)]
    prob = _make(sizes, seed=5)
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    dp = DeviceProblem.upload(prob)
    # give the empty groups real (non-empty) C buffers to watch
    for g, (m, n, k, _) in enumerate(sizes):
        if m == 0:
            dp.C[g] = torch.full((4, n), 0x7E00, dtype=torch.int16, device="cuda").view(torch.float16)
    dp.run()
    torch.cuda.synchronize()
    ref = _oracle_full(oracle_mod, prob)
    for g, (m, n, k, _) in enumerate(sizes):
        c = dp.C[g].cpu().numpy()
        if m == 0:
            assert np.all(c.view(np.uint16) == 0x7E00), g
        else:
            assert_parity(c, ref[g], f"group {g}")


def test_scale_doubling_moves_one_row(nv, oracle_mod):
    """Doubling one SFA scale block changes only that row of C; each run
    matches the oracle; every other row is bit-identical between runs."""
    m, n, k = 150, 256, 512
    prob = _make([(m, n, k, 1)], seed=9)
    _, base = _run(nv, prob)
    row, blk = 131, 9
    code = int(prob.SFA[0][row, blk])
    assert 1 <= (code >> 3) <= 13
    prob.SFA[0] = prob.SFA[0].copy()
    prob.SFA[0][row, blk] = code + 8
    _, dbl = _run(nv, prob)
    assert_parity(dbl[0], _oracle_full(oracle_mod, prob)[0], "doubled")
    others = np.arange(m) != row
    np.testing.assert_array_equal(dbl[0][others].view(np.uint16), base[0][others].view(np.uint16))
    assert not np.array_equal(dbl[0][row].view(np.uint16), base[0][row].view(np.uint16))


def test_unit_scale_single_element(nv):
    """A single non-zero product lands at exactly one C element, exactly."""
    m, n, k = 130, 160, 256
    a = np.zeros((m, k // 2), np.uint8)
    b = np.zeros((n, k // 2), np.uint8)
    sfa = np.full((m, k // 16), 0x38, np.uint8)
    sfb = np.full((n, k // 16), 0x38, np.uint8)
    i, j, kk = 129, 131, 201                      # row in the 2nd m-tile, col in the 2nd n-tile
    a[i, kk // 2] = 0x7 << (4 * (kk % 2))         # 6.0
    b[j, kk // 2] = 0x5 << (4 * (kk % 2))         # 3.0
    sfa[i, kk // 16] = 0x40                       # 2.0
    sfb[j, kk // 16] = 0x30                       # 0.5
    from nvfp4_block_scaled_grouped_gb300.workloads import GroupedProblem
    prob = GroupedProblem("unit", 0, [(m, n, k, 1)], [a], [b], [sfa], [sfb])
    _, got = _run(nv, prob)
    want = np.zeros((m, n), np.float16)
    want[i, j] = 6.0 * 3.0 * 2.0 * 0.5
    np.testing.assert_array_equal(got[0].view(np.uint16), want.view(np.uint16))


# ---------------------------------------------------------------- full-size workloads, sampled

def _samples(rng, m, n, count=1024):
    """Two random outputs in every 32 x 32 cell of C (so every tile, column
    chunk and TMEM lane quarter of the kernel's tiling is reached), the last
    row and column, and `count` more anywhere."""
    br, bc = block_samples(rng, m, n)
    rows = np.concatenate([br, rng.integers(0, m, count)])
    cols = np.concatenate([bc, rng.integers(0, n, count)])
    return rows.astype(np.int32), cols.astype(np.int32)


_PROBLEMS = {}


def _workload(name):
    if name not in _PROBLEMS:
        from nvfp4_block_scaled_grouped_gb300 import workloads
        _PROBLEMS.clear()
        _PROBLEMS[name] = workloads.make_problem(name)
    return _PROBLEMS[name]


@pytest.mark.parametrize("name,block_n,split", [("decode", 256, None), ("decode", 128, False),
                                                ("prefill", 256, None), ("prefill", 128, True),
                                                ("prefill", 256, "hybrid"), ("ragged", 256, None),
                                                ("ragged", 256, "hybrid"), ("zipf64", 256, None),
                                                ("zipf64", 256, "hybrid")])
def test_full_size_sampled(nv, oracle_mod, monkeypatch, name, block_n, split):
    _schedule(monkeypatch, split)
    prob = _workload(name)
    dp, got = _run(nv, prob, block_n)
    rng = np.random.default_rng(17)
    for g, (m, n, k, _) in enumerate(prob.problem_sizes):
        c = got[g]
        if m == 0 or n == 0:
            assert c.size == 0
            continue
        assert not np.isnan(c.astype(np.float32)).any(), f"{name} group {g}: NaN / untouched entries"
        rows, cols = _samples(rng, m, n)
        ref = oracle_mod.gemm_sampled(m, n, k, prob.A[g], prob.B[g], prob.SFA[g], prob.SFB[g], rows, cols)
        assert_parity(c[rows, cols], ref, f"{name} group {g}")
    # a repeated call gives the same bits
    dp.run()
    torch.cuda.synchronize()
    for g, c in enumerate(dp.c_host()):
        np.testing.assert_array_equal(c.view(np.uint16), got[g].view(np.uint16))


@pytest.mark.parametrize("name", ["decode", "ragged"])
def test_full_size_full_c(nv, oracle_mod, name):
    """Every output of the full-size decode and ragged calls (library-chosen
    tile width and schedule) against the oracle's full C."""
    prob = _workload(name)
    _, got = _run(nv, prob, 256)
    ref = _oracle_full(oracle_mod, prob)
    for g, ((m, n, k, _), c, r) in enumerate(zip(prob.problem_sizes, got, ref)):
        if m == 0 or n == 0:
            assert c.size == 0
            continue
        assert_parity(c, r, f"{name} group {g} (full C)")


def test_two_streams_concurrently(nv, oracle_mod):
    """Calls on two streams use separate workspaces and may overlap."""
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    p1 = _make([(100, 256, 512, 1), (33, 128, 256, 1)], seed=21)
    p2 = _make([(300, 96, 1024, 1)], seed=22)
    d1, d2 = DeviceProblem.upload(p1), DeviceProblem.upload(p2)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        d1.run(s1)
        d2.run(s2)
    torch.cuda.synchronize()
    for dp, prob in ((d1, p1), (d2, p2)):
        for g, (c, r) in enumerate(zip(dp.c_host(), _oracle_full(oracle_mod, prob))):
            assert_parity(c, r, f"stream problem group {g}")
    assert nv.device_status(s1) == 0 and nv.device_status(s2) == 0


def test_descriptor_slots_follow_pointer_and_shape_changes(nv, oracle_mod):
    """A workspace's descriptor slots are reused across calls when a group's
    pointer and shape are unchanged; any change (groups reordered, a smaller m
    over the same buffer, another tile width) must be patched again."""
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem
    sizes = [(130, 256, 512, 1), (64, 128, 256, 1), (200, 384, 768, 1)]
    prob = _make(sizes, seed=31)
    dp = DeviceProblem.upload(prob)
    ref = _oracle_full(oracle_mod, prob)

    def check(order, msg, block_n=256):
        nv.set_tile_n(block_n)
        out = [torch.full_like(dp.C[g], float("nan")) for g in order]
        nv.grouped_gemm([sizes[g] for g in order], [dp.A[g].data_ptr() for g in order],
                        [dp.B[g].data_ptr() for g in order], [dp.SFA[g].data_ptr() for g in order],
                        [dp.SFB[g].data_ptr() for g in order], [o.data_ptr() for o in out])
        torch.cuda.synchronize()
        assert nv.device_status() == 0
        for i, g in enumerate(order):
            assert_parity(out[i].cpu().numpy(), ref[g], f"{msg}: slot {i} = group {g}")

    check([0, 1, 2], "first call")
    check([0, 1, 2], "same pointers and shapes again")
    check([2, 0, 1], "groups moved to other slots")
    check([2, 0, 1], "moved groups, BN=128", block_n=128)
    check([2, 0, 1], "moved groups, back to BN=256")
    # the same A buffer read as fewer rows: only m changes
    m_small = 70
    sub = _make([(m_small, 256, 512, 1)], seed=31)  # same seed/stream: rows are a prefix of group 0
    np.testing.assert_array_equal(sub.A[0], prob.A[0][:m_small])
    out = torch.full((m_small, 256), float("nan"), dtype=torch.float16, device="cuda")
    sfa_small = nv.pack_scales_tensor(torch.from_numpy(prob.SFA[0][:m_small]).cuda(), 512)
    nv.grouped_gemm([(m_small, 256, 512, 1)], [dp.A[0].data_ptr()], [dp.B[0].data_ptr()],
                    [sfa_small.data_ptr()], [dp.SFB[0].data_ptr()], [out.data_ptr()])
    torch.cuda.synchronize()
    assert_parity(out.cpu().numpy(), ref[0][:m_small], "m shrunk over the same A buffer")
