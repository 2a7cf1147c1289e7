"""The bounds-checked build: every index the kernels compute from data before an access
(request lists, tokens used as row indices, partial slots, list slots) is checked against
its buffer when the library is compiled with -DDSPARK_BOUNDS, and a miss is reported as
DSPARK_ERR_BOUNDS.  The guard-region, recompute-verification and chained-step tests run
again against that build (in a child process, selected by DSPARK_LIBRARY) and must see
DSPARK_OK and the same parity throughout.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounds_checked_build_runs_clean():
    sys.path.insert(0, ROOT)
    from speculative_decoding_draft_gb300 import build

    lib = build.build(bounds=True)
    assert lib.endswith("libdspark_bounds.so")
    env = dict(os.environ, DSPARK_LIBRARY=lib)
    probe = subprocess.run([sys.executable, "-c",
                            "import speculative_decoding_draft_gb300 as ds; ds.lib(); print(ds.library_path())"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert probe.returncode == 0 and probe.stdout.strip().endswith("libdspark_bounds.so"), probe.stderr[-2000:]
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                        "tests/test_gpu_canary.py", "tests/test_gpu_verify_markov.py", "tests/test_gpu_chain.py",
                        "-k", "not full_size"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
