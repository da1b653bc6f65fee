"""bench.py on CPU.  Its launcher: ``--gpus N`` started without a launcher
starts N ranks itself (through torch.distributed.run on 127.0.0.1), rank 0
alone prints the JSON line, and a launcher whose WORLD_SIZE disagrees with
``--gpus`` is refused.  The reference arm (the oracle on host cores) needs no
GPU, so it stands in for the flce arm here.  And its traffic records, which
follow the kernels' code, not their comments."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--impl", "reference", "--steps", "1", "--warmup", "0", "--ref-tokens", "1",
        "--workload", "tiny_worked_4x128x256_fp32"]


def _bench(extra, env=None):
    e = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        e.pop(k, None)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *ARGS, *extra],
                          capture_output=True, text=True, timeout=600, cwd=ROOT, env=e)


def test_gpus_2_starts_two_ranks_and_prints_one_line():
    r = _bench(["--gpus", "2"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["value"] > 0 and d["unit"] == "tokens/s"


def test_world_size_mismatch_is_refused():
    r = _bench(["--gpus", "3"], env={"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode != 0
    assert "WORLD_SIZE" in r.stderr


def test_traffic_records_follow_the_code_not_the_comments():
    """A recorded DRAM-traffic figure stays valid across comment-only edits of
    its kernel's sources and is dropped after a change to their code."""
    import bench
    src = {n: "// header\nint f(int a) { return a + 1; } /* note */\n"
           for n in bench.KERNEL_SOURCES["dx"]}
    base = bench.kernel_source_hash("dx", src.__getitem__)
    name = sorted(src)[0]
    recommented = dict(src)
    recommented[name] = "// other words\n/* block\n comment */ int f(int a)  {\n return a + 1;\n}\n"
    assert bench.kernel_source_hash("dx", recommented.__getitem__) == base
    changed = dict(src)
    changed[name] = src[name].replace("a + 1", "a + 2")
    assert bench.kernel_source_hash("dx", changed.__getitem__) != base
