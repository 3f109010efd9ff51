"""Failure detection without a GPU fault.

Every device wait in the library is bounded (a cycle budget), and a wait that
runs out records the timeout in an error word the host reads, then lets the
kernel end.  The test makes one such wait run out -- on a barrier that no
thread completes -- and checks the reported status and that the context still
runs a full step correctly afterwards.  Nothing here faults, traps or hangs.
"""
import pytest

from newton_schulz_bucket_gb300 import _capi
from newton_schulz_bucket_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    from parity import GpuRun, check_all
    L = _capi.load()
    limit = 1 << 20  # ~0.5 ms of SM cycles
    assert L.muon_testing_wait_probe(1, limit, None) == _capi.MUON_OK
    assert L.muon_testing_wait_probe(0, limit, None) == _capi.MUON_ERR_TIMEOUT
    assert L.muon_testing_wait_probe(0, 0, None) == _capi.MUON_ERR_INVALID_ARG
    run = GpuRun(W.custom([[24, 2048], [256, 384]], seed=31))
    check_all(run)
    run.close()
