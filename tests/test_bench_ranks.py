"""Host logic of the multi-replica bench (torchrun, one process per GPU) on two CPU ranks over gloo: rank
environment, distinct per-rank seeds, the max-over-ranks time and the whole-job value. No GPU is involved; the
block itself has no exchange step, so this is the whole of its N > 1 path besides the per-rank GPU work."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.rank_env()
    elapsed = 10.0 + 5.0 * r                      # rank 1 is the slow one
    m = bench.max_over_ranks(elapsed)
    q.put({"rank": r, "world": w, "local": lr, "seed": bench.rank_seed(r), "max": m,
           "value": bench.whole_job_value(w, 100, m)})
    dist.destroy_process_group()


def test_two_ranks_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort(key=lambda d: d["rank"])
    assert [d["world"] for d in out] == [2, 2] and [d["local"] for d in out] == [0, 1]
    assert out[0]["seed"] != out[1]["seed"]
    assert out[0]["max"] == out[1]["max"] == 15.0
    assert out[0]["value"] == pytest.approx(2 * 100 / 15e-3)


def test_single_process_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.rank_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_value(1, 1000, 20.0) == pytest.approx(50000.0)


def test_reference_arm_other_ranks_do_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    """The reference arm (the oracle on the host cores) prints one JSON line with the contract's keys, on the
    same metric, unit and workload as the main arm."""
    sys.path.insert(0, ROOT)
    import bench
    env = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 3
    assert d["ms_per_step"] == pytest.approx(1e3 / d["value"])
    assert d["config"]["workload"] == bench.WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
