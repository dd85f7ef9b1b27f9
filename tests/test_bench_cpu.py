"""bench.py contract checks that run without a GPU: the reference arm (the
float64 oracle) on one process and as two gloo ranks under torchrun."""
import json
import os
import subprocess
import sys

from conftest import ROOT

TINY = "batch=2,len_lo=64,len_hi=200,pool_pages=64,h_q=8,h_kv=2"


def _json_lines(text):
    return [json.loads(l) for l in text.splitlines() if l.startswith("{")]


def test_reference_arm_single_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--override", TINY,
                        "--steps", "2", "--warmup", "1"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["steps"] == 2 and d["warmup"] >= 3


def test_reference_arm_two_gloo_ranks():
    """Under torchrun with two ranks only rank 0 prints (one line); the other
    rank exits 0 without work."""
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", "29531", "bench.py", "--impl", "reference",
                        "--gpus", "2", "--override", TINY, "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def test_reference_arm_does_not_load_the_cuda_library():
    """The reference arm runs the oracle only: after it ran in this process,
    the package's CUDA library has not been loaded."""
    code = (
        "import sys, runpy; sys.argv = ['bench.py', '--impl', 'reference', '--override', "
        f"'{TINY}', '--steps', '1', '--warmup', '1']; "
        "runpy.run_path('bench.py', run_name='__main__'); "
        "import paged_kv_cache_203_gb300 as pkv; "
        "maps = open('/proc/self/maps').read(); "
        "assert pkv._LIB is None and 'libpkv.so' not in maps, 'libpkv loaded'; print('CLEAN')")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "CLEAN" in r.stdout
