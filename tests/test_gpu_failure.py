"""Failure detection on the GPU without a fault: every pipeline wait in the
library is bounded, and a wait that runs out sets the device error word,
lets its kernel return and is reported by repro_device_check() as
REPRO_ERR_TIMEOUT.  Here a barrier phase that nothing completes makes the
library's own bounded wait run out; the status is read on the host and the
context must stay usable (later calls still give the oracle's bits)."""
import time

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import gpu_helpers as G  # noqa: E402
import bitwise_reproducible_int8_gb300 as R  # noqa: E402

ERR_TIMEOUT = -6


def _scale_matches_oracle(orc, seed):
    x = np.random.default_rng(seed).standard_normal(70_001).astype(np.float32)
    G.assert_bits_equal(G.gpu_scale(x, 0), orc.wscale(x, 0), "scale after a timeout")


def test_satisfied_wait_reports_nothing():
    assert R.repro_device_check() == R.REPRO_OK
    assert R.repro_wait_probe(1) == R.REPRO_OK
    assert R.repro_device_check() == R.REPRO_OK


def test_wait_that_runs_out_is_reported_and_cleared(orc):
    assert R.repro_device_check() == R.REPRO_OK
    t0 = time.monotonic()
    assert R.repro_wait_probe(0) == R.REPRO_OK          # enqueueing succeeds
    assert R.repro_device_check() == ERR_TIMEOUT         # the wait gave up, the host sees it
    waited = time.monotonic() - t0
    assert 0.2 < waited < 30.0, waited                   # bounded: about two seconds
    assert R.repro_device_check() == R.REPRO_OK          # reading cleared the word
    # the context is intact: ordinary calls still run and match the oracle
    _scale_matches_oracle(orc, 11)
    assert R.repro_device_check() == R.REPRO_OK


def test_timeout_on_a_side_stream_leaves_other_work_intact(orc):
    side = torch.cuda.Stream()
    assert R.repro_wait_probe(0, stream=side) == R.REPRO_OK
    _scale_matches_oracle(orc, 12)                            # runs on the current stream meanwhile
    assert R.repro_device_check(side) == ERR_TIMEOUT
    assert R.repro_device_check(side) == R.REPRO_OK
    _scale_matches_oracle(orc, 13)


def test_repeated_timeouts_each_reported_once():
    for _ in range(2):
        assert R.repro_wait_probe(0) == R.REPRO_OK
        assert R.repro_device_check() == ERR_TIMEOUT
        assert R.repro_device_check() == R.REPRO_OK
        assert R.repro_wait_probe(1) == R.REPRO_OK
        assert R.repro_device_check() == R.REPRO_OK
