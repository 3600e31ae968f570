"""The failure path on the GPU without a fault: a bounded wait that nobody satisfies
runs out after about one second, the kernel records its site in the device error
word and returns; the host reads ATTN_ERR_DEVICE_TIMEOUT with that site, the word is
cleared, and the same context then runs attention correctly."""
import time

import numpy as np
import pytest
import torch

from parity_util import compare, gpu_run, oracle_run
from scaled_dot_product_tmem_gb300.inputs import Shape, make_inputs

pytestmark = pytest.mark.gpu

TIMEOUT = 5  # ATTN_ERR_DEVICE_TIMEOUT


def test_bounded_wait_reports_and_the_context_stays_usable():
    import scaled_dot_product_tmem_gb300 as sdpa
    assert sdpa.attn_last_device_error() == (0, 0)
    t0 = time.perf_counter()
    sdpa.attn_selftest_wait_timeout(0x5A)
    st, site = sdpa.attn_last_device_error()  # synchronises the stream
    dt = time.perf_counter() - t0
    assert st == TIMEOUT and site == 0x100 + 0x5A, (st, hex(site))
    assert 0.5 < dt < 30.0, dt                 # the wait limit, not a hang
    assert sdpa.attn_last_device_error() == (0, 0)  # reading cleared the word
    # the context is intact: a normal call runs and matches the oracle
    x = make_inputs(Shape(1, 200, 200, 4, 2, 64, 64), 13)
    kw = dict(causal=True, window=50, softmax_type=0, scale=None)
    compare(gpu_run(x, **kw), oracle_run(x, **kw), "after the self-test")
