"""Failure detection without a GPU fault: a wait that nothing completes.

The library's kernels bound every wait on an asynchronous copy or MMA by wall
time and report an expired wait through the device error word instead of
trapping or hanging.  q4k_selftest_wait_timeout runs that same bounded wait on
an mbarrier nothing arrives at; the test checks that the timeout bit comes back,
that the word is cleared by the read, and that the context still computes
correct results afterwards.
"""
from __future__ import annotations

import time

import pytest
import torch

import oracle
import synth
from _gpu import DEV, check_bound, xbits

pytestmark = pytest.mark.gpu
Q4K_DEVERR_TIMEOUT = 1


@pytest.fixture(scope="module")
def q4k():
    from bit_block_quantized_q4_gb300 import build
    build.build()
    import bit_block_quantized_q4_gb300 as m
    return m


def test_bounded_wait_reports_timeout_and_context_survives(q4k):
    assert q4k.q4k_get_device_error() == 0
    t0 = time.time()
    q4k.q4k_selftest_wait_timeout()
    bits = q4k.q4k_get_device_error()          # synchronizes the stream
    elapsed = time.time() - t0
    assert bits & Q4K_DEVERR_TIMEOUT
    assert 0.5 < elapsed < 30.0                # gave up after its limit, did not hang
    assert q4k.q4k_get_device_error() == 0     # the read cleared the word
    # the context is still usable: an ordinary projection matches the oracle
    n, k = 300, 2048
    w = synth.q4k_weight(n, k, seed=77)
    x = synth.bf16_normal((1, k), seed=78)
    y = q4k.q4k_gemv(w.to(DEV), n, k, x.to(DEV))
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
    check_bound(y.cpu().numpy(), yref, s, 2e-3, "after timeout")
