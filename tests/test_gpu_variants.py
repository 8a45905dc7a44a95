"""Parity with programmatic dependent launch switched off (PKV_PDL=0, read once per
process, so it runs in a child process): every kernel then starts only after the
previous one on the stream has finished. Results must not depend on how soon a
kernel starts, so the child reruns existing parity tests (tests/test_gpu_parity.py,
test_gpu_prefill.py) under the variable, decode and prefill.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_child(env_var, value, selection, test_file="test_gpu_parity.py"):
    env = dict(os.environ, **{env_var: value})
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", test_file),
                        "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider", "-k", selection],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, f"{env_var}={value}:\n{r.stdout[-3000:]}\n{r.stderr[-2000:]}"
    assert " passed" in r.stdout and " failed" not in r.stdout, r.stdout[-2000:]


@pytest.mark.parametrize("test_file,selection", [
    ("test_gpu_parity.py", "decode_small_cases or shared_prefix_plan or graph_replay"),
    ("test_gpu_prefill.py", "small_cases or graph_replay"),
])
def test_without_programmatic_dependent_launch(test_file, selection):
    run_child("PKV_PDL", "0", selection, test_file)
