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


@pytest.mark.parametrize("case", ["tiny_fp32", "bf16_d256", "cb_batch16"])
def test_stale_timeout_bit_does_not_stop_later_steps(case):
    """The sticky word only reports: with PHOTON_DEVERR_WAIT_TIMEOUT left set
    by an earlier launch (not cleared), later decode steps on the CUDA-core
    kernel (fp32, bf16 head_dim 256) and the tensor-core kernel must still
    compute every row, equal to the oracle."""
    pk = ensure_built()
    pk.photon_device_errors(clear=True)
    pk.photon_selftest_wait_timeout(1_000_000)
    if case == "bf16_d256":
        wl = synth.make_custom([3, 200, 700, 1300], 8, 2, 256, kv_dtype="bf16", seed=3, value_std=0.5)
    else:
        wl = synth.make(case)
    vals = synth.make_values(wl, device="cuda")
    h = host_inputs(wl, vals)
    ref, _, _, _ = oracle_step(wl, h)
    out, _ = gpu_step(wl, vals, partition_size=256 if case == "bf16_d256" else None)
    tol = 1e-5 if wl.kv_dtype == "f32" else 5e-3
    got = out.cpu().numpy()
    assert np.isfinite(got).all() and np.abs(got - ref).max() <= tol
    assert pk.photon_device_errors(clear=True) == pk.DEVERR_WAIT_TIMEOUT  # still only the old bit
