"""Failure detection without a GPU fault.

Every spin-wait of the tcgen05 kernels is bounded; an expired wait records a code in a
device word, the kernel returns, and medusa_poll_errors reports MEDUSA_ERR_TIMEOUT. The
self-test kernel waits on an mbarrier that nothing completes, for a budget of a few
milliseconds, so the expiry path runs for real and the GPU context stays usable.
"""
import numpy as np
import pytest
import torch

from medusa_speculative_decoding_heads_gb300 import binding as mb, configs
from medusa_speculative_decoding_heads_gb300.configs import GREEDY

from _helpers import gpu_ready


def test_selftest_budget_is_checked_on_the_host():
    mb.load()
    for bad in (0, 1_000_001):
        assert mb.load().medusa_selftest_wait_timeout(bad, 0) == -1   # invalid argument, nothing enqueued


@pytest.mark.gpu
def test_expired_wait_is_reported_once_and_the_context_stays_usable():
    gpu_ready()
    mb.poll_errors()                                  # start from clear words
    mb.selftest_wait_timeout(3000)                    # ~3 ms bounded wait that nothing completes
    status, heads, attn = mb.poll_errors()
    assert status == mb.STATUS_TIMEOUT and heads == 0 and attn == mb.WAIT_SELFTEST_CODE
    assert mb.poll_errors() == (0, 0, 0)              # read-and-clear
    # a whole step afterwards runs and checks out against the oracle, and leaves no error behind
    import test_gpu_parity as parity
    w = configs.scaled(configs.get("gqa7b_b32"), B=4, d=512, V=1000, Hq=8, Hkv=2, L_range=(40, 300),
                       modes=(GREEDY,), target_corr=0.0)
    parity.check_step(w, torch.device("cuda"))
    assert mb.poll_errors() == (0, 0, 0)
