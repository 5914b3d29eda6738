"""bench.py's reference arm (the fp64 oracle on the host cores) runs without a GPU: its JSON
line carries the keys the benchmark contract asks for, on the forward, the projection and
the backward."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("extra", [[], ["--pass", "proj"], ["--pass", "bwd"], ["--alibi"]])
def test_reference_arm_line(extra):
    d = run_bench("--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3", *extra)
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["gpu_launches"] == 0 and d["config"]["workload"] == "tiny"


def test_bench_rejects_too_few_warmup_steps():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], capture_output=True,
                         text=True, timeout=120, cwd=ROOT)
    assert out.returncode != 0 and "warmup" in out.stderr


def test_profile_hash_ignores_comments_but_not_code():
    sys.path.insert(0, ROOT)
    import bench
    src = 'int a = 1;  // one\n/* block\ncomment */\n\nasm("x // y" : "=r"(a));\nchar c = \'"\';\n'
    assert bench.code_only(src) == 'int a = 1;\nasm("x // y" : "=r"(a));\nchar c = \'"\';'
    assert bench.code_only(src.replace("// one", "// two")) == bench.code_only(src)
    assert bench.code_only(src.replace("a = 1", "a = 2")) != bench.code_only(src)


def test_reference_arm_line_for_decode():
    d = run_bench("--impl", "reference", "--workload", "pythia160m-decode", "--steps", "3", "--warmup", "3")
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0 and d["steps"] == 3
    assert d["e2e"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle" and d["gpu_launches"] == 0
    assert d["config"]["workload"] == "pythia160m-decode" and 1 <= d["config"]["sample_sequences_per_step"] <= 64
