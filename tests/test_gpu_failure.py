"""Failure detection without a GPU fault: a bounded wait that nothing will
satisfy gives up, reports PHOTON_DEVERR_WAIT_TIMEOUT through the sticky error
word, and leaves the context usable for the next step."""
import time

import numpy as np
import pytest

import synth
from tests.helpers import ensure_built, gpu_step, host_inputs, oracle_step

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports():
    pk = ensure_built()
    pk.photon_device_errors(clear=True)
    t0 = time.perf_counter()
    pk.photon_selftest_wait_timeout(2_000_000)  # ~1 ms of SM cycles
    flags = pk.photon_device_errors(clear=True)
    assert flags & pk.DEVERR_WAIT_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    assert pk.photon_device_errors(clear=True) == 0  # cleared


def test_context_usable_after_a_timeout():
    pk = ensure_built()
    pk.photon_selftest_wait_timeout(1_000_000)
    assert pk.photon_device_errors(clear=True) & pk.DEVERR_WAIT_TIMEOUT
    wl = synth.make("cb_batch16")
    vals = synth.make_values(wl, device="cuda")
    h = host_inputs(wl, vals)
    ref, _, _, _ = oracle_step(wl, h)
    out, _ = gpu_step(wl, vals)
    assert np.abs(out.cpu().numpy() - ref).max() <= 5e-3
    assert pk.photon_device_errors() == 0
