"""The failure path of the pipelines' bounded waits, on the GPU without a fault: a wait
on a barrier that nothing completes must give up, report LS_ERR_TIMEOUT through the
device error word, and leave the context usable for the next replay."""
import time

import numpy as np
import pytest

import oracle
from parity_util import TOL_LSE, TOL_O, Case, rel_err
from response_replay_gb300 import binding as B

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_the_context_survives(cuda):
    assert B.ls_last_device_error(0) == B.LS_OK
    t0 = time.perf_counter()
    B.ls_selftest_wait_timeout(0)
    assert B.ls_last_device_error(0) == B.LS_ERR_TIMEOUT
    waited = time.perf_counter() - t0
    assert 0.5 < waited < 60, waited           # the limit is about 2 s of SM clock
    assert B.ls_last_device_error(0) == B.LS_OK  # reading the word cleared it

    # the same context still runs the replay pipelines correctly
    case = Case(1000, 200, 6, 2, 16, 3, 4242, cuda, sharp=True)
    o, lse = case.fwd()
    o_ref, lse_ref = oracle.attn_fwd(case.problem())
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL_O
    assert float(np.abs(lse.cpu().numpy() - lse_ref).max()) <= TOL_LSE
    assert B.ls_last_device_error(0) == B.LS_OK
