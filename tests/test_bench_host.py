"""Host-side logic of bench.py without a GPU: the max-over-ranks timing
reduction on two gloo ranks, the JSON line of the CPU reference arm, and the
traffic record lookup."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_path):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([10.0 * (rank + 1), 5.0 - rank], world, torch.device("cpu"))
        if rank == 0:
            with open(out_path, "w") as f:
                json.dump(got, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    import socket

    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    out = tmp_path / "max.json"
    mp.spawn(_rank_main, args=(2, port, str(out)), nprocs=2, join=True)
    assert json.loads(out.read_text()) == [20.0, 5.0]


def test_max_over_ranks_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1, None) == [1.5, 2.5]


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_record_follows_kernel_source(tmp_path):
    """A traffic line counts only while the kernel source has the hash it was
    measured with."""
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "tc.cu"
    src.write_text("// kernel source, revision 1\n")
    sha = hashlib.sha1(src.read_bytes()).hexdigest()[:12]
    prof = tmp_path / "traffic.md"
    prof.write_text(f"traffic: workload=aero kernel=encode source_sha1={sha} bytes_per_launch=1234\n"
                    f"traffic: workload=aero kernel=decode source_sha1=0123456789ab bytes_per_launch=9\n")
    assert bench.measured_traffic("aero", "encode", str(src), str(prof)) == 1234
    assert bench.measured_traffic("aero", "decode", str(src), str(prof)) is None  # other revision
    assert bench.measured_traffic("aero", "no-such-kernel", str(src), str(prof)) is None
    src.write_text("// kernel source, revision 2\n")
    assert bench.measured_traffic("aero", "encode", str(src), str(prof)) is None
    # the committed record parses (lines may be stale while the kernels change)
    bench.measured_traffic("aero", "encode")


def test_variant_stage_costs():
    """Algorithmic bytes per pass follow each variant's inputs: the synthesis
    reads Ks_raw (D per token), Ks and Vs (2D), or nothing (FLARE)."""
    sys.path.insert(0, ROOT)
    import bench
    from rank_latent_routing_gb300 import workloads
    s = workloads.Shape(2, 3, 100, 64, 16)
    th = 2 * 3 * 100
    assert bench.stage_costs(s, 2)["synthesis"]["bytes"] == th * 16 * 2
    assert bench.stage_costs(s, 2, "unshared")["synthesis"]["bytes"] == 2 * th * 16 * 2
    assert bench.stage_costs(s, 2, "simplified")["synthesis"]["bytes"] == 2 * th * 16 * 2
    flare = bench.stage_costs(s, 2, "flare")
    assert flare["synthesis"] == {"bytes": 0, "flops": 0.0, "exps": 0.0}
    assert flare["encode"]["bytes"] == 2 * th * 16 * 2


@pytest.mark.parametrize("variant", ["flare", "simplified"])
def test_reference_arm_variant(variant):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3", "--workload", "tiny",
                        "--variant", variant], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.strip()][-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert f"{variant} mixer" in line["config"]["workload"]
