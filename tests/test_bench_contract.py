"""bench.py's JSON line, checked without a GPU: the reference arm (the fp64
oracle on the host cores) on the tiny workload prints one line with every key
the benchmark contract names, and its values are consistent with each other."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_prints_the_contract_line():
    d = _run("--impl", "reference", "--workload", "tiny_fp32", "--steps", "2", "--warmup", "3",
             "--cpu-seconds", "1")
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None
    assert d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "tiny_fp32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_kernel_source_hash_ignores_comments_only():
    """The traffic table is keyed by a hash of the decode sources without
    their comments: a comment edit keeps it, a code edit changes it."""
    import bench
    base = b"int f(int x) {\n  return x + 1;  // one more\n}\n/* block\n comment */\n"
    assert bench._strip_comments(base) == bench._strip_comments(
        base.replace(b"one more", b"the successor").replace(b"block", b"another"))
    assert bench._strip_comments(base) != bench._strip_comments(base.replace(b"x + 1", b"x + 2"))
    assert bench._strip_comments(b"a = 1;\n\n// only a comment\nb = 2;\n") == b"a = 1;\nb = 2;"
