"""The forward's odd-shaped parity cases rerun on the bounds-checked debug
build of the library (FA_DEBUG): there, the tensor-core forward checks every
shared-memory, tensor-memory and output index range before using it and
reports a failed check as FA_ERR_DEVICE_BOUNDS.  The cases run in a child
pytest process that loads the debug library (FA_GB300_LIBRARY); each of
them compares its outputs with the oracle and requires a clean device
status, so a range error anywhere in those launches fails this test.  (The
memory checker of the CUDA toolkit is closed on this GPU pool; these checks
stand in for it.)"""
import os
import re
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Small odd shapes: single rows, ragged tails, both head dims, causal and
# not, packed sequences of lengths 0, 1, 127..129, window edges, sentinel
# tails, the moving reference maximum, the timeout path, and the persistent
# launch (B=4 H=16 N=2048: 1024 items on one CTA per SM).
CASES = ("test_bf16_small or test_varlen_small or test_output_tail_untouched or "
         "test_reference_moves or test_scale_zero_prefix_means or test_window or "
         "test_wait_timeout_unwinds or test_config2_full or test_forward_deterministic")


def test_forward_cases_clean_under_debug_checks():
    import exact_io_aware_15_gb300 as fa
    if not os.path.exists(fa.DEBUG_LIB_PATH):
        from exact_io_aware_15_gb300 import build
        build.build()
    env = dict(os.environ, FA_GB300_LIBRARY=fa.DEBUG_LIB_PATH)
    # the child's binding loads the debug library
    which = subprocess.run([sys.executable, "-c",
                            "import exact_io_aware_15_gb300 as fa; print(fa.LIB_PATH)"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert which.stdout.strip() == fa.DEBUG_LIB_PATH, which.stdout + which.stderr
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu",
         os.path.join(ROOT, "tests", "test_gpu_prefill.py"),
         os.path.join(ROOT, "tests", "test_gpu_variants.py"),
         os.path.join(ROOT, "tests", "test_gpu_failure.py"),
         "-k", CASES],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 30, r.stdout[-2000:]
