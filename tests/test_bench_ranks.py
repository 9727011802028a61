"""The multi-rank (replica) path of bench.py on CPU: world size 2 over gloo.

The grouped GEMM has no exchange step, so N GPUs run N independent replicas;
what bench.py adds for N > 1 is host logic -- every rank takes part in the
max-over-ranks reductions of the timed region, rank 0 alone prints, and the
whole-job rate is all ranks' work over the slowest rank's time.
"""
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parent.parent


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, str(ROOT))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [37.5, 41.0][rank]                     # this rank's mean step time (ms)
        t_max = bench.max_over_ranks(local, world, "cpu")
        e_max = bench.max_over_ranks(10.0 * (rank + 1), world, "cpu")
        value = bench.replica_throughput(4.0e10, world, t_max * 1e-3)
        Path(out_dir, f"rank{rank}.json").write_text(json.dumps({"t_max": t_max, "e_max": e_max, "value": value}))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_replica_rate_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    got = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in range(world)]
    for g in got:
        assert g["t_max"] == 41.0                      # the slowest rank's time, on every rank
        assert g["e_max"] == 20.0
        assert g["value"] == pytest.approx(2 * 4.0e10 / 41.0e-3)


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.replica_throughput(10.0, 1, 2.0) == 5.0


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank_zero_only(rank):
    """Under torchrun the reference arm (the CPU oracle) runs on rank 0 alone;
    the other ranks exit 0 without work or output."""
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "0", "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank == 0:
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
        assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    else:
        assert lines == []


def test_profile_summary_lookup(tmp_path, monkeypatch):
    """The roofline's `traffic` comes from a committed ncu summary only when
    the summary names the kernel code as it is now (comments do not count)."""
    sys.path.insert(0, str(ROOT))
    import bench
    src = tmp_path / "k.cu"
    src.write_text("int x; // a comment\n\n__global__ void k() {}\n")
    d = bench.kernel_code_digest(src)
    src.write_text("int x; // another comment\n// more\n__global__ void k() {}\n")
    assert bench.kernel_code_digest(src) == d
    src.write_text("int y;\n__global__ void k() {}\n")
    assert bench.kernel_code_digest(src) != d
    cur = bench.kernel_code_digest(ROOT / "nvfp4_block_scaled_grouped_gb300" / "csrc" / "gemm.cu")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "nvfp4_block_scaled_grouped_gb300" / "csrc").mkdir(parents=True)
    (tmp_path / "nvfp4_block_scaled_grouped_gb300" / "csrc" / "gemm.cu").write_text(
        (ROOT / "nvfp4_block_scaled_grouped_gb300" / "csrc" / "gemm.cu").read_text())
    summ = tmp_path / "profiles" / "gemm_kernel_decode.txt"
    summ.write_text(f"gemm.cu code sha256[:16]: {cur} (comments and blank lines stripped)\ntile_n: 256\n"
                    "dram bytes per launch: 123456\n")
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    assert bench.stored_traffic("decode", 256) == 123456.0
    assert bench.stored_traffic("decode", 128) is None
    summ.write_text("gemm.cu code sha256[:16]: 0000000000000000\ntile_n: 256\ndram bytes per launch: 1\n")
    assert bench.stored_traffic("decode", 256) is None


def test_quantize_traffic_names_its_own_source(tmp_path, monkeypatch):
    """The quantise line's `traffic` checks quantize.cu's digest and the
    profiled shape, not the GEMM kernel's."""
    sys.path.insert(0, str(ROOT))
    import bench
    csrc = tmp_path / "nvfp4_block_scaled_grouped_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "quantize.cu").write_text("__global__ void q() {}\n")
    (csrc / "gemm.cu").write_text("__global__ void g() {}\n")
    dq = bench.kernel_code_digest(csrc / "quantize.cu")
    dg = bench.kernel_code_digest(csrc / "gemm.cu")
    summ = tmp_path / "profiles" / "quantize_pack_kernel_prefill.txt"
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    shape = {"rows": "8192", "k": "7168"}
    summ.write_text(f"quantize.cu code sha256[:16]: {dq}\nrows: 8192\nk: 7168\ndram bytes per launch: 777\n")
    assert bench.profile_traffic("quantize_pack_kernel_prefill.txt", "quantize.cu", shape) == 777.0
    assert bench.profile_traffic("quantize_pack_kernel_prefill.txt", "quantize.cu", {"rows": "732", "k": "7168"}) is None
    summ.write_text(f"gemm.cu code sha256[:16]: {dg}\nrows: 8192\nk: 7168\ndram bytes per launch: 777\n")
    assert bench.profile_traffic("quantize_pack_kernel_prefill.txt", "quantize.cu", shape) is None
