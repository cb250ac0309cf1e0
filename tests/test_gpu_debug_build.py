"""The tiny and mid-size parity suites under the bound-checking build.

The V4_DEBUG build checks every gather row, selection-list slot, P-buffer
offset and TMEM column of the tensor-core kernels against its bound; a
failed check records V4_ERR_BOUND in the device status word and skips the
access.  The parity tests (which also assert a clean status word) run in a
child process that loads that build through V4ATTN_LIB.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suites_pass_under_the_bound_checking_build():
    from sparse_compressed_attention_gb300 import build
    lib = build.build(debug=True)
    env = dict(os.environ, V4ATTN_LIB=lib)
    probe = subprocess.run([sys.executable, "-c", "import sparse_compressed_attention_gb300 as V; "
                            "print(V.v4_build_info())"], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=300)
    assert "V4_DEBUG" in probe.stdout, probe.stdout + probe.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_parity.py", "tests/test_gpu_tc.py",
                        "tests/test_gpu_kl_target.py", "-m", "gpu", "-x", "-q", "-p", "no:cacheprovider",
                        "-k", "not full_size and not every_row"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
