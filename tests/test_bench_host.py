"""CPU tests of the benchmark's host logic: byte accounting (pinned to the
sizes the source post prints), the multi-rank reduction over gloo, and the
reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

GOLDEN = os.path.join(ROOT, "tests", "golden", "paper_sizes.txt")


def paper_sizes():
    out = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        key, val, tol = line.split()[:3]
        out[key] = (float(val), float(tol.split("=")[1]))
    return out


def test_router_bytes_match_the_post():
    val, tol = paper_sizes()["router_bytes_bf16"]
    b = bench.algorithmic_bytes(2560, 512, 8, 512, M=1, n_active=0) - 2 * 2560 * 2 - 8 * 4
    assert b == 2560 * 512 * 2
    assert abs(b - val) <= tol * val


def test_expert_traffic_matches_the_post():
    # six-token verify chain x top-8, all 48 experts distinct, inter split over 4 GPUs
    val, tol = paper_sizes()["expert_traffic_per_layer_step_tp4"]
    full = bench.algorithmic_bytes(2560, 512, 8, 512 // 4, M=6, n_active=48)
    experts = full - bench.algorithmic_bytes(2560, 512, 8, 512 // 4, M=6, n_active=0)
    assert experts == 48 * 3 * 2560 * 128 * 2
    assert abs(experts - val) <= tol * val


def test_call_bytes_count_router_and_io_once():
    # no expert chosen: the router weight once, x in, out out, the indices out
    base = bench.algorithmic_bytes(2560, 512, 8, 512, M=6, n_active=0)
    assert base == 512 * 2560 * 2 + 2 * 6 * 2560 * 2 + 6 * 8 * 4
    # each distinct expert adds its gate, up and down weights exactly once
    assert bench.algorithmic_bytes(2560, 512, 8, 512, M=6, n_active=46) - base == 46 * 3 * 2560 * 512 * 2


@pytest.mark.parametrize("fp8", [False, True])
def test_traffic_record_is_complete_and_near_the_algorithmic_bytes(fp8):
    # the committed ncu records the bench scales into roofline.traffic
    if not os.path.exists(bench.TRAFFIC_FILES[fp8]):
        pytest.skip("no record for this weight type")
    with open(bench.TRAFFIC_FILES[fp8]) as f:
        tr = json.load(f)
    assert bool(tr.get("fp8", False)) == fp8
    for key in ("source_hash", "shape", "M", "bytes_per_launch", "algorithmic_bytes_per_launch", "launches", "command"):
        assert key in tr
    reads = [l["dram_read"] + l["dram_write"] for l in tr["launches"]]
    assert abs(sum(reads) / len(reads) - tr["bytes_per_launch"]) <= 1e-6 * tr["bytes_per_launch"] + 1
    # DRAM traffic of a cold call is its algorithmic bytes, give or take a few per cent
    assert 0.97 <= tr["bytes_per_launch"] / tr["algorithmic_bytes_per_launch"] <= 1.05


def test_layer_count_keeps_l2_cold():
    from weight_streaming_expert_gb300 import workloads as wl
    l2 = 126 * 1024 * 1024
    for M in (1, 6, 16, 64):
        n = bench.n_layers_for(M, wl.LING, l2, 0)
        per = bench.algorithmic_bytes(2560, 512, 8, 512, M, min(8 * M, 512) * 0.85 + 1)
        assert n >= 4 and (n - 1) * per >= 3 * l2


WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import bench
rank, ws, local, pg = bench.dist_setup(2)
assert ws == 2 and pg is not None
bench.barrier(pg)
v = bench.max_over_ranks(pg, 1.0 + rank)
assert v == 2.0, v
print("ok", rank, v)
pg.destroy_process_group()
"""


def test_two_rank_max_over_ranks_gloo(tmp_path):
    script = tmp_path / "w.py"
    script.write_text(WORKER.format(root=ROOT))
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
                        "--master-addr=127.0.0.1", "--master-port=29533", str(script)],
                       capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.count("ok") == 2


def test_reference_arm_prints_one_json_line(tmp_path):
    """The oracle arm on a reduced workload shape, through bench's own code."""
    from weight_streaming_expert_gb300 import workloads as wl
    us, n, host = bench.oracle_call_us(wl.TINY, M=6, zipf=False, budget_s=0.5, max_calls=5)
    assert us > 0 and 1 <= n <= 5


def test_crossover_summary_finds_the_first_lasting_tensor_core_win():
    import bench
    Ms = (1, 2, 3, 4)
    res = {(1, "cuda_cores"): 9.6, (1, "tensor_cores"): 10.0,   # CUDA cores 4 % faster
           (2, "cuda_cores"): 10.0, (2, "tensor_cores"): 9.8,   # within the margin
           (3, "cuda_cores"): 12.0, (3, "tensor_cores"): 10.0,
           (4, "cuda_cores"): 14.0, (4, "tensor_cores"): 10.0}
    s = bench.crossover_summary(res, Ms)
    assert s["tensor_cores_faster_from_M_e"] == 3
    assert s["cuda_cores_faster_at_M_e"] == [1]
    assert s["ratio_cuda_over_tensor"]["4"] == 1.4
    res[(4, "tensor_cores")] = 14.0  # a tie at the largest M_e: no lasting win
    assert bench.crossover_summary(res, Ms)["tensor_cores_faster_from_M_e"] is None
