"""Failure detection without a GPU fault.

Every pipelined kernel waits on mbarriers with a wall-clock bound; when a wait
runs out it records a timeout flag in the device error word and returns.  The
self-test kernel runs that same bounded wait on a barrier that nothing
completes, with a 1 ms budget, and the host reads FQ_ERR_DEVICE_TIMEOUT back.
The context must stay usable: a parity-checked call runs right after.
"""
import time

import numpy as np
import pytest
import torch

from oracle import int8 as oi8
from fp8_dynamic_quant_gb300 import synth
import fp8_dynamic_quant_gb300 as fq
from _util import bf16_to_dev, bf16_to_np

pytestmark = pytest.mark.gpu

FQ_OK, FQ_ERR_DEVICE_TIMEOUT = 0, 7


def test_wait_timeout_is_reported_and_context_survives():
    assert fq.device_error()[0] == FQ_OK  # start clean
    t0 = time.perf_counter()
    fq.selftest_wait_timeout(budget_ns=1_000_000, arrive=False)
    st, word = fq.device_error()
    dt = time.perf_counter() - t0
    assert st == FQ_ERR_DEVICE_TIMEOUT and word & 1
    assert dt < 5.0  # the wait gave up on its own
    assert fq.device_error() == (FQ_OK, 0)  # reading clears the word

    # the context is still usable: a W8A8 call right after is bit-exact
    c = synth.int8_linear_case(4, 1024, 256, 77)
    y = fq.w8a8_quant_linear(bf16_to_dev(c["x"]), torch.from_numpy(c["w_nk"]).cuda(),
                             torch.from_numpy(c["sw"]).cuda())
    want, _, _ = oi8.w8a8_quant_linear(c["x"], c["w_nk"], c["sw"])
    assert np.array_equal(bf16_to_np(y), want)
    assert fq.device_error() == (FQ_OK, 0)


def test_wait_completes_when_arrived():
    fq.selftest_wait_timeout(budget_ns=1_000_000, arrive=True)
    assert fq.device_error() == (FQ_OK, 0)


def test_budget_is_clamped():
    # a huge budget is clamped to 1 s; with the arrival it returns at once
    fq.selftest_wait_timeout(budget_ns=10 ** 15, arrive=True)
    assert fq.device_error() == (FQ_OK, 0)
