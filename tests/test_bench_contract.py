"""bench.py's contract on the CPU: the reference arm (the fp64 oracle on the
host cores) prints one JSON line with the keys the measurement contract asks
for, non-zero ranks of a launch print nothing, the warm-up floor is enforced,
and the algorithmic byte and flop counts match the workload's definition
(q, k, v read and o written in bf16, beta and gamma in fp32, the state in and
out; 6 N D^2 + 2 D^3 flops per frame-head)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env=None, timeout=600):
    e = dict(os.environ, **(env or {}))
    return subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, env=e, capture_output=True, text=True,
                          timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "layer_60s_720p"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]


def test_reference_arm_other_ranks_print_nothing():
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "3"], env={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_floor():
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "2"])
    assert r.returncode != 0


def test_algorithmic_counts():
    sys.path.insert(0, ROOT)
    import bench
    a = bench.algorithmic(1, 20, 121, 880, 112)
    per_fh = 880 * 112 * (3 * 2 + 2) + 4 * 880 + 4          # q, k, v in, o out, beta, gamma
    assert a["stats"] + a["out"] == 20 * 121 * per_fh == 20 * 121 * 792004
    assert a["state"] == 2 * 20 * 112 * 112 * 4
    assert a["flops"] == 20 * 121 * (6 * 880 * 112 ** 2 + 2 * 112 ** 3)
    assert bench.step_bytes(1, 20, 880, 112) == 17847120


def _max_rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        bench.barrier(world)
        v = bench.max_over_ranks(world, 1.5 + rank)   # per-rank step times
        with open(os.path.join(out, f"r{rank}.txt"), "w") as fh:
            fh.write(repr(v))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_on_cpu_ranks(tmp_path):
    """The timing reduction of a multi-rank run: every rank sees the slowest rank's time."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.spawn(_max_rank, args=(3, port, str(tmp_path)), nprocs=3, join=True)
    for r in range(3):
        assert float(open(tmp_path / f"r{r}.txt").read()) == 3.5
