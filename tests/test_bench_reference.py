"""bench.py's reference arm (the oracle timed on the host cores) on CPU: the JSON line it prints
and, under two gloo ranks, that rank 0 alone runs and prints while the other rank exits cleanly."""
import contextlib
import io
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _check_line(d, n_gpus):
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["n_gpus"] == n_gpus and d["steps"] == 2 and d["warmup"] == 3
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"].startswith("tiny")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_prints_one_contract_line():
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
                          "--warmup", "1"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [x for x in res.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    _check_line(json.loads(lines[0]), 1)   # a warm-up count below 3 is raised to 3


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    os.chdir(ROOT)
    import bench
    sys.argv = ["bench.py", "--impl", "reference", "--workload", "tiny", "--gpus", str(world), "--steps", "2",
                "--warmup", "3"]
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main()
    out[rank] = buf.getvalue()


def test_reference_arm_two_ranks_rank0_only():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(600)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    lines0 = [x for x in out[0].splitlines() if x.startswith("{")]
    assert len(lines0) == 1
    _check_line(json.loads(lines0[0]), 2)
    assert not [x for x in out[1].splitlines() if x.startswith("{")]


def test_stored_dram_counters_match_the_kernel_sources():
    """profiles/traffic.json (the ncu DRAM bytes the bench line's roofline `traffic` reports) is
    keyed to a hash of the kernel sources' code; a kernel edit without a new capture would make
    the bench report null traffic, so the committed state must match."""
    sys.path.insert(0, ROOT)
    import bench

    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        stored = json.load(f)
    assert stored["kernel_hash"] == bench.kernel_hash()
    t = bench.load_traffic()
    for key in ("grouped_linear1_bytes_per_launch", "grouped_linear2_bytes_per_launch", "quantize_bytes_per_launch"):
        assert t[key] == stored[key] and t[key] > 0
