"""Failure detection without a GPU fault: a device wait that can never be
satisfied expires, the device error word reports it to the host, and the
context keeps working.  Host-side argument failures are covered on CPU in
test_host_abi.py."""
import time

import pytest
import torch

from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def test_expired_device_wait_is_reported_and_context_survives():
    import headwise_chunked_attention_gb300 as u
    from tests.test_parity_fwd import run_fwd
    w = WORKLOADS["tiny-s2048"]
    t = make_inputs(w, seed=0)
    out0, lse0, _ = run_fwd(w, 2, t, debug=False)
    assert u.last_error() == 0
    t0 = time.time()
    u.selftest_wait_timeout(50_000)          # 50 ms
    assert u.last_error() == 5               # UPIPE_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 30
    assert u.last_error() == 0               # reading clears it
    # the context still works: the same forward gives the same bits
    out1, lse1, _ = run_fwd(w, 2, t, debug=False)
    assert u.last_error() == 0
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_selftest_rejects_bad_limits():
    import headwise_chunked_attention_gb300 as u
    with pytest.raises(u.UpipeError):
        u.selftest_wait_timeout(0)
