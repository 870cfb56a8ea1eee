"""Failure detection on the GPU without a fault.

The library's self-test launches a bounded wait that nothing satisfies: it must
give up after the limit, record DIT_ERR_TIMEOUT with its wait site in the
device status word, return normally, and leave the context usable (a normal
attention call afterwards runs clean and matches the oracle).
"""
import time

import numpy as np
import pytest
import torch

import parity
from dit_long_sequence_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    import dit_long_sequence_gb300 as dl
    rc, info = dl.check_watchdog()
    assert rc == 0, info
    t0 = time.perf_counter()
    dl.watchdog_selftest(limit_us=50_000)
    rc, info = dl.check_watchdog()          # synchronises
    elapsed = time.perf_counter() - t0
    assert rc == dl.binding.DIT_ERR_TIMEOUT, (rc, info)
    assert info[0] == dl.binding.DIT_ERR_TIMEOUT and info[3] == 99, info
    assert 0.04 < elapsed < 5.0, elapsed
    # the word was cleared and the context still works
    rc, info = dl.check_watchdog()
    assert rc == 0, info
    q, k, v, _ = wl.make_qkv(1, 300, 2, 128, seed=3, device=torch.device("cuda:0"))
    O, L = dl.attn_fwd(q, k, v)
    rc, info = dl.check_watchdog()
    assert rc == 0, info
    Or, Lr = parity.oracle_full(q, k, v)
    parity.compare(O.double().cpu().numpy(), L.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))


def test_selftest_rejects_bad_limits():
    import dit_long_sequence_gb300 as dl
    for bad in (0, 999, 2_000_001):
        with pytest.raises(dl.DitError):
            dl.watchdog_selftest(limit_us=bad)
