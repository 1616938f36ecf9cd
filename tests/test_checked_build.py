"""The checked build (PA_CHECKED): every kernel range-checks the global
indices it computes (block-table entries, lengths, q and out rows, workspace
slots and counters) and reports a violation through PA_DEV_OOB instead of
making the access.  compute-sanitizer is not available on the GPUs these
tests run on, so this build is how the index arithmetic is checked on the
device: the small-shape parity suites run against it and must report no
status bit beyond the ones each test expects.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from paged_kv_gqa_02_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# small-shape suites: decode (split counts, partial, combine, bad pages and
# lengths, graph replay), prefill, several rows, windows, append, head_dim
# 256, the single launch
SELECT = ("not workload_full and not run_to_run_bitwise_deterministic")
FILES = ["tests/test_gpu_parity.py", "tests/test_single_launch.py", "tests/test_multi_row_decode.py",
         "tests/test_sliding_window.py", "tests/test_decode_append.py", "tests/test_head_dim_256.py"]


def test_parity_suites_pass_on_the_checked_build():
    lib = build.build(checked=True)
    probe = subprocess.run(
        [sys.executable, "-c",
         "from paged_kv_gqa_02_gb300 import ops; L = ops.load(); print(L.pa_build_flags(), ops.LIB_PATH)"],
        cwd=ROOT, env=dict(os.environ, PA_GQA_LIB=lib), capture_output=True, text=True, timeout=600)
    assert probe.returncode == 0, probe.stderr
    flags, path = probe.stdout.split()
    assert int(flags) == 1 and os.path.samefile(path, lib)
    r = subprocess.run([sys.executable, "-m", "pytest", *FILES, "-q", "-x", "-m", "gpu", "-k", SELECT,
                        "-p", "no:cacheprovider"],
                       cwd=ROOT, env=dict(os.environ, PA_GQA_LIB=lib), capture_output=True, text=True,
                       timeout=3000)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
