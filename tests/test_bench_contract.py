"""bench.py's output contract, checked on the arm that runs without a GPU
(--impl reference: the float64 oracle on the host cores)."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line_with_the_contract_keys():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("gqa_32x4k")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_warmup_below_three_is_rejected():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "--warmup must be >= 3" in r.stderr


def test_reference_arm_under_torchrun_prints_once_from_rank_zero():
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and "rank 0 of 2" in d["cpu_baseline"]["sample"]


def test_kernel_digest_ignores_comments_and_tracks_code(tmp_path):
    """The digest that keys the committed ncu traffic figures: a comment or blank-line edit keeps it (the
    compiled kernel is the same), a code edit changes it (the counters no longer describe the kernel)."""
    import shutil
    sys.path.insert(0, ROOT)
    import bench
    src = os.path.join(ROOT, "paged_kv_cache_144_gb300", "csrc")
    dst = tmp_path / "paged_kv_cache_144_gb300" / "csrc"
    shutil.copytree(src, dst)
    base = bench.kernel_source_digest(str(tmp_path))
    assert base == bench.kernel_source_digest()
    f = dst / "pa_kernels.h"
    text = f.read_text()
    f.write_text("// an added comment\n\n" + text.replace("{", "{  /* inline comment */", 1) + "\n\n")
    assert bench.kernel_source_digest(str(tmp_path)) == base
    f.write_text(text.replace("{", "{ int added_field_for_the_test; ", 1))
    assert bench.kernel_source_digest(str(tmp_path)) != base
    # a string literal that looks like a comment is code
    assert bench._code_only('const char* s = "a // b";  // c') == 'const char* s = "a // b";'
