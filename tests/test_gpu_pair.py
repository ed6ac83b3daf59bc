"""The backward's dQ on CTA pairs (tcgen05 cta_group::2, replay_bwd_dq_pair.cu), selected
with LS_BWD_PAIR=1: the attention parity cases (ragged shapes, grouped-query packing,
P = 0, more splits than tiles) and the ragged-members cases rerun against the fp64 oracle
in a fresh process with the pair kernel selected.  The default path (one CTA per unit)
is covered by the same tests in this process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_pair_kernel_parity(cuda):
    env = dict(os.environ, LS_BWD_PAIR="1")
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_gpu_attention.py"),
         os.path.join(ROOT, "tests", "test_gpu_ragged.py"),
         "-k", "ragged or packed or small_workload or deterministic or accumulate"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert " passed" in r.stdout
