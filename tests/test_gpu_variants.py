"""Parity of the decode kernel's opt-in instances, which the library selects from
environment variables read once per process (so each runs in a child process):

* PKV_SHARED_ROW_BLOCKS=2: the two-row-block shared-prefix kernel (32 query rows per
  KV head, one CTA per SM, units of one row block dealt by stages);
* PKV_HEADS_PER_CTA=2 and 1: narrower head groups per CTA (512 B and 256 B rows);
* PKV_PDL=0: every kernel launched without programmatic dependent launch (each starts
  after the previous one has finished), decode and prefill.

Each child runs existing parity tests (tests/test_gpu_parity.py, test_gpu_prefill.py)
under the variable.
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


def test_two_row_block_shared_prefix_kernel():
    run_child("PKV_SHARED_ROW_BLOCKS", "2", "shared_prefix_plan or early_gather")


@pytest.mark.parametrize("heads", ["2", "1"])
def test_narrow_head_groups(heads):
    run_child("PKV_HEADS_PER_CTA", heads, "decode_small_cases or fused_append_attention")


@pytest.mark.parametrize("test_file,selection", [
    ("test_gpu_parity.py", "decode_small_cases or shared_prefix_plan or graph_replay"),
    ("test_gpu_prefill.py", "small_cases or graph_replay"),
])
def test_without_programmatic_dependent_launch(test_file, selection):
    run_child("PKV_PDL", "0", selection, test_file)
