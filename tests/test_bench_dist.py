"""Multi-replica host logic of bench.py on CPU (gloo, world size 2).

Verification shards by sequence with no exchange, so several GPUs run
independent replicas: each rank verifies its own seeded batch, the slowest
rank's time is the job's time, and the job's rate counts every rank's rows.
These tests run that logic as two gloo ranks without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_verification_59_gb300 import workloads as W  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank times: rank 1 is the slow one
        ms = [12.5, 20.0][rank]
        ms_max = bench.max_over_ranks(ms, world, "cpu")
        x = W.make_chain("chain-small", seed=bench.rank_seed(W.WORKLOADS["chain-small"].seed, rank))
        rows = bench.step_accounting(x)["rows"]
        rate = bench.job_rate(world, rows, 10, ms_max)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms_max": ms_max, "rate": rate, "rows": rows,
                       "target_sum": float(np.asarray(x.target, dtype=np.float64).sum())}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_max_time_and_sum_rows(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    # both ranks see the slowest rank's time
    assert r[0]["ms_max"] == r[1]["ms_max"] == 20.0
    # whole-job rate: both ranks' rows over the slowest time
    expect = world * r[0]["rows"] * 10 / 20.0e-3
    assert r[0]["rate"] == pytest.approx(expect) and r[1]["rate"] == pytest.approx(expect)
    # each replica verified its own batch
    assert r[0]["target_sum"] != r[1]["target_sum"]


def test_single_rank_helpers_need_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_rate(1, 1536, 100, 50.0) == pytest.approx(1536 * 100 / 0.05)
    assert bench.rank_seed(2, 0) == 2 and bench.rank_seed(2, 3) == 3002


def test_reference_arm_on_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert p.returncode == 0
    assert p.stdout.strip() == ""


def test_reference_arm_prints_the_contract_line():
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1", "--workload", "chain-small"],
                       capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    line = json.loads(p.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["config"]["workload"] == "chain-small"


def test_lazy_rows_read_accounting():
    """Rows the lazy pass reads per sequence, as bench.py reports them: every
    group up to the one holding the sequence's rejection (or the bonus row),
    target and draft rows of its positions (the last position has no draft
    row)."""
    import bench
    groups = [(0, 2), (2, 8)]                          # chain-b64's schedule, gamma = 7
    assert [bench.lazy_rows_read(k, groups) for k in (-1, 0, 1)] == [4, 4, 4]
    assert all(bench.lazy_rows_read(k, groups) == 4 + 6 + 5 for k in range(2, 8))
    assert bench.lazy_rows_read(0, [(0, 1)]) == 1       # gamma = 0: the bonus row only
    assert bench.lazy_rows_read(4, [(0, 2), (2, 5)]) == 4 + 3 + 2


def test_kernel_hash_ignores_comments_but_not_code(tmp_path):
    """The traffic figure recorded under profiles/ stays valid across an edit of comments
    alone, and is dropped after any change of the streaming kernel's code."""
    import shutil
    src = os.path.join(bench.ROOT, "speculative_decoding_verification_59_gb300", "csrc")
    for f in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(src, f), tmp_path / f)
    h0 = bench.kernel_source_hash(str(tmp_path))
    assert h0 == bench.kernel_source_hash()
    p = tmp_path / "sv_stream.cuh"
    text = p.read_text(encoding="utf-8")
    p.write_text("// a new comment line\n\n" + text.replace("namespace sv {", "namespace sv {  // same code"),
                 encoding="utf-8")
    assert bench.kernel_source_hash(str(tmp_path)) == h0
    p.write_text(text.replace("constexpr int kStages = 3;", "constexpr int kStages = 4;"), encoding="utf-8")
    assert bench.kernel_source_hash(str(tmp_path)) != h0


def test_recorded_traffic_matches_the_committed_kernel():
    """profiles/stats_traffic.txt carries the hash of the code it was captured on; the
    bench line reports its traffic only while that hash is the current one."""
    t = bench.recorded_traffic("chain-b64")
    assert t is None or t >= 291717120
