"""Host-side checks of bench.py: the multi-rank combination (gloo, world size 2) and the
reference arm's JSON line (the CPU oracle; no GPU needed)."""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    el, units = bench.combine_over_ranks(1.0 + rank, 100.0 * (rank + 1), world)
    bench.barrier(world)
    q.put((rank, el, units))
    dist.destroy_process_group()


def test_combine_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, el, units in res:
        assert el == 2.0          # max over ranks
        assert units == 300.0     # summed over ranks


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["unit"] == "GB/s" and line["value"] > 0
    import oracle
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] == oracle.threads(openmp=True) >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_cpu_baseline_single_and_all_core():
    """The CPU baseline reports the all-core rate with its thread count and the single-thread
    rate beside it, measured on a bounded row sample of the workload's layer."""
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    assert bench.sample_rows(13824, 2560, 1) == 7812
    assert bench.sample_rows(2560, 6912, 256) == 16 and bench.sample_rows(256, 256, 1) == 256
    cb = bench.cpu_baseline_for("2B", 1, 0.0, 0.0)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["value"] > 0
    assert cb["cores"] == oracle.threads(openmp=True)
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
    assert "rows multiplied per matrix" in cb["sample"]


def test_step_bytes_match_layer_shapes():
    sys.path.insert(0, ROOT)
    import bench
    # 2B layer: q|k|v 3840x2560, o 2560x2560, gate|up 13824x2560, down 2560x6912
    packed = (3840 * 2560 + 2560 * 2560 + 13824 * 2560 + 2560 * 6912) // 4
    assert packed == 17_367_040
    acts = 2560 * 3 + 6912
    scales = 4 * (4 + 4)
    assert bench.step_bytes(1) == 30 * (packed + acts + scales)


def test_recorded_traffic_needs_matching_source_hash(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    f = tmp_path / "traffic.md"
    monkeypatch.setitem(bench.TRAFFIC_FILES, "2b", str(f))
    assert bench.recorded_traffic("2b") is None  # no summary
    f.write_text("# summary\n- source_hash: `%s`\n- dram_bytes_per_launch_avg: 4321.5\n"
                 % bench.source_hash(bench.GEMV_SOURCES))
    assert bench.recorded_traffic("2b") == 4321.5
    f.write_text("- source_hash: `0000000000000000`\n- dram_bytes_per_launch_avg: 4321.5\n")
    assert bench.recorded_traffic("2b") is None  # taken on another kernel
    assert bench.recorded_traffic("8b_m1") is None
