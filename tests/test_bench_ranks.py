"""The multi-replica path of bench.py on CPU (no GPU): two gloo ranks agree
on the slowest replica's time and the whole-job rate, and the reference arm
runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    ms = [3.0, 5.0][rank]                      # rank 1 is the slow replica
    m = bench.max_over_ranks(ms, world, "cpu")
    q.put((rank, m, bench.whole_job_rate(world, 100, m)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_replica():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [5.0, 5.0]
    # 2 replicas x 100 units in 5 ms
    assert got[0][2] == pytest.approx(40000.0)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.whole_job_rate(1, 4096, 2.0) == pytest.approx(2048000.0)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "3", "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if rank == 0:
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    else:
        assert lines == []


def test_tensor_peak_follows_the_sampled_clocks():
    """The bench holds a kernel to the burst bf16 peak at full clocks, and to
    the sustained one once the power cap (or a lowered clock) shows."""
    import bench
    pk = {"bf16_tflops": 1957.4, "bf16_tflops_sustained": 1729.1}
    assert bench.tensor_peak(pk, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}) == (1957.4, "burst")
    assert bench.tensor_peak(pk, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}) == \
        (1729.1, "sustained")
    assert bench.tensor_peak(pk, {"sm_mhz": 1650.0, "sm_max_mhz": 2070.0, "reasons": []}) == (1729.1, "sustained")
    assert bench.tensor_peak(pk, {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]})[1] == "burst"


def test_traffic_figure_only_for_its_workload_and_source(tmp_path, monkeypatch):
    """roofline.traffic is reported only for the workload the ncu capture was
    taken on, and only while the profiled kernel source is unchanged."""
    import hashlib
    import bench
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel\n")
    h = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    entry = {"source": "kernel.cu", "source_sha256_16": h, "workload": "w: T=1", "bytes_per_launch": 1234}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"k": entry}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("k", "w: T=1") == 1234
    assert bench.traffic_for("k", "w: T=2") is None       # another workload
    assert bench.traffic_for("other", "w: T=1") is None   # another kernel
    src.write_text("// changed\n")
    assert bench.traffic_for("k", "w: T=1") is None       # the source changed since the capture
