"""Host-side logic of bench.py on CPU: the multi-rank timing reduction over a
world-size-2 gloo group, the reference arm under torchrun, and the byte
accounting the roofline numbers rest on.

The data path has no exchange step (rows are independent units), so N ranks
are N replicas: each verifies its own cohort, the job's time is the slowest
rank's, and the job's throughput is N cohorts over that time.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, per_rank_ms, out_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(per_rank_ms[rank], "cpu", world)
        rate = bench.job_rate(world, 16, ms)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "rate": rate, "seed": bench.rank_seed(2, rank)}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    world, per_rank = 2, [0.25, 0.40]
    mp.start_processes(_rank_main, args=(world, _free_port(), per_rank, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["ms"] == pytest.approx(max(per_rank)), "every rank sees the slowest rank's time"
        assert r["rate"] == pytest.approx(world * 16 / (max(per_rank) * 1e-3))
    assert res[0]["seed"] != res[1]["seed"], "ranks draw distinct cohorts"


def test_single_rank_reduction_is_identity():
    assert bench.max_over_ranks(1.5, "cpu", 1) == 1.5
    assert bench.job_rate(1, 16, 0.5) == pytest.approx(32000.0)


def test_reference_arm_under_torchrun_world2(tmp_path):
    """Rank 0 alone times the oracle and prints one JSON line; rank 1 exits 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--B", "2", "--layers", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2 and d["warmup"] == 1
    for key in ("metric", "value", "unit", "ms_per_step", "higher_is_better", "scaling", "vs_baseline", "dtype",
                "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert "workload" in d["config"]


def _geom():
    from speculative_decode_gated_gdn_gb300 import synth
    return synth.Geometry(B=8, T=2, H_k=16, H_v=32, d=128)


def test_byte_accounting():
    g = _geom()
    row = 32 * 128 * 128 * 4
    assert bench.state_row_bytes(g) == row
    base = bench.verify_bytes(g, 6)
    assert base > 6 * row and base < 6 * row + (1 << 20), "state dominates a verify's bytes"
    assert bench.verify_bytes(g, 6, "snapshot") == base + 2 * 6 * row
    assert bench.verify_bytes(g, 6, "deferred", 4) == base + 4 * row
    shift = bench.ring_shift_bytes(g, 4, 30)
    assert bench.commit_bytes(g, 4, 30, "recompute") == 2 * row * 4 * 30 + shift
    assert bench.commit_bytes(g, 4, 30, "deferred") == shift
    # whatever the strategy, a cycle moves at least the path's minimum, and
    # DEFERRED moves exactly that when the same rows are kept every cycle
    mn = bench.path_min_bytes(g, 6, 4, 30)
    for mode in ("recompute", "snapshot"):
        step = 30 * bench.verify_bytes(g, 6, mode) + bench.commit_bytes(g, 4, 30, mode)
        assert step > mn
    assert 30 * bench.verify_bytes(g, 6, "deferred", 4) + bench.commit_bytes(g, 4, 30, "deferred") == mn


def test_source_hash_follows_code_not_comments():
    src = ('int a = 1;  // a note\n/* a block\n   comment */ const char *s = "// kept";\n'
           "char q = '\"';\n\n  x = y; /* inline */ z;\n")
    code = bench.code_only(src)
    assert "note" not in code and "block" not in code and "inline" not in code
    assert '"// kept"' in code and "'\"'" in code and "x = y;" in code and "z;" in code
    # comments, trailing blanks and empty lines do not move the hash; code does
    assert bench.code_only(src.replace("a note", "another note") + "\n\n// tail\n") == code
    assert bench.code_only(src.replace("x = y;", "x = w;")) != code


def test_profiled_figures_need_a_matching_code_hash(monkeypatch):
    # a committed ncu figure is reported only while the code it was taken on
    # is the current code
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    key = next(iter(rec["verify"]))
    monkeypatch.setattr(bench, "source_hash", lambda kind: rec[kind]["source_hash"] if kind == "prefill"
                        else rec[kind][key]["source_hash"])
    assert bench.profiled_traffic("verify", key) == rec["verify"][key]["dram_bytes_per_launch"]
    assert bench.profiled_tensor_pipe() == rec["prefill"]["tensor_pipe"]
    monkeypatch.setattr(bench, "source_hash", lambda kind: "0" * 16)
    assert bench.profiled_traffic("verify", key) is None
    assert bench.profiled_tensor_pipe() is None
