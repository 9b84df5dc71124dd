"""Multi-process (gloo, world size 2, CPU) coverage of the benchmark's replica path:
every rank runs its own copy of the workload (no exchange in the data path), the
timing is the maximum over ranks and the throughput is summed over replicas."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    vals = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)])
    gbs = bench.aggregate_throughput(1e9, vals[0], world)
    q.put((rank, vals, gbs))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, vals, gbs in out:
        assert vals == [2.0, 5.0, 0.5]                 # max over the two ranks
        assert gbs == pytest.approx(2 * 1e9 / 2e-3 / 1e9)   # two replicas, slowest rank's 2 ms


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.aggregate_throughput(2e9, 1.0, 1) == pytest.approx(2000.0)


def test_kernel_hash_ignores_comments_but_not_code():
    """The committed DRAM counters stay valid across comment edits, never across code edits."""
    import bench
    code = "int f(int x) {\n    return x + 1;   // add one\n}\n"
    commented = "// header\n/* block\n   comment */\nint f(int x) {\n\n    return x + 1;\n}\n"
    assert bench._code_only(code) == bench._code_only(commented)
    assert bench._code_only(code) != bench._code_only(code.replace("x + 1", "x + 2"))
    h = bench.kernel_source_hash()
    assert len(h) == 16 and h == bench.kernel_source_hash()


def test_reference_arm_json_line():
    """bench.py --impl reference (the fp64 oracle on this host's cores) prints the bench
    contract's JSON line; a non-zero rank prints nothing and exits 0."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--config", "c1",
           "--steps", "2", "--warmup", "1"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=root)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"] and line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] >= 1 and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    other = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=root,
                           env=dict(os.environ, RANK="1", WORLD_SIZE="2"))
    assert other.returncode == 0 and other.stdout.strip() == ""
