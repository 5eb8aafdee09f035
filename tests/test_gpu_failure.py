"""Device-side failure reporting, tested without faulting the GPU: a bounded wait that nothing
completes must give up, record DLR_ERR_TIMEOUT in the status word, and leave the context usable."""
import numpy as np
import pytest
import torch

import oracle
from state_space_sequence_gb300 import dlr, inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert dlr.device_status() == dlr.DLR_OK
    dlr.selftest_timeout(50)
    assert dlr.device_status() == dlr.DLR_ERR_TIMEOUT
    assert dlr.device_status() == dlr.DLR_OK  # reading clears it
    # the context still computes correctly afterwards
    w = inputs.make_dlr(1, 2, 8, 300, seed=3)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    y = dlr.dlr_layer(dev(w.u), (dev(w.fwd.log_re), dev(w.fwd.log_im), dev(w.fwd.W)))
    torch.cuda.synchronize()
    ref = oracle.dlr_layer(w.u, (w.fwd.log_re, w.fwd.log_im, w.fwd.W))
    assert oracle.rel_l2(y.cpu().numpy(), ref) <= 1e-5


def test_selftest_rejects_bad_limits():
    with pytest.raises(dlr.DLRError):
        dlr.selftest_timeout(0)
    with pytest.raises(dlr.DLRError):
        dlr.selftest_timeout(5000)
