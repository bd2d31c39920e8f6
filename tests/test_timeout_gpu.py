"""A bounded wait that runs out reports a timeout and leaves the context usable.

Every kernel waits on its mbarriers with the same bounded wait (include/ffpa.h,
ffpa_check_status).  ffpa_selftest_wait_timeout launches one warp whose wait
nothing completes, so the wait runs out without any copy or MMA in flight.
The test checks that the status comes back once as FFPA_ERR_TIMEOUT, is then
cleared, and that a normal call on the same context still matches the oracle.
"""
import pytest
import torch

from head_dim_attention_gb300 import _lib, ffpa_check_status
from parity import check_fwd_full

pytestmark = pytest.mark.gpu
FFPA_ERR_TIMEOUT = 5


def test_wait_runs_out_and_context_survives():
    _lib.load()
    torch.cuda.synchronize()
    assert ffpa_check_status() == 0
    _lib.ffpa_selftest_wait_timeout()
    assert ffpa_check_status() == FFPA_ERR_TIMEOUT
    assert ffpa_check_status() == 0  # read once, then cleared
    check_fwd_full(1, 1, 1, 256, 256, 512, torch.float16)
    check_fwd_full(1, 2, 2, 129, 129, 512, torch.bfloat16, causal=True)
