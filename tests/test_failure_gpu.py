"""Failure detection on the GPU without a GPU fault: a bounded device-side wait
that nothing completes runs out after its limit, the kernel records
FA_ERR_TIMEOUT in the device error word and returns, the host reads it through
fa_get_last_device_error, and the device keeps working."""
import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_21_gb300 import synthetic as syn
from oracle import naive
from tests.parity import check_out, f64

pytestmark = pytest.mark.gpu

SITE_SELFTEST = 19


def test_bounded_wait_times_out_and_device_stays_usable(cuda_lib):
    fa = cuda_lib
    assert fa.fa_get_last_device_error()[0] == fa.FA_OK     # start clean
    fa.fa_selftest_wait_timeout(2_000_000)                   # a 2 ms limit
    st, detail = fa.fa_get_last_device_error()
    assert st == fa.FA_ERR_TIMEOUT, detail
    assert detail[0] == fa.FA_ERR_TIMEOUT and detail[1] == SITE_SELFTEST
    assert fa.fa_get_last_device_error()[0] == fa.FA_OK     # reading cleared the word
    # the context is intact: a forward afterwards is still right
    q, k, v = (syn.bhnd(21, t, 1, 2, 300, 128) for t in (syn.TAG_Q, syn.TAG_K, syn.TAG_V))
    dev = torch.device("cuda", 0)
    o, lse = fa.forward(q.to(dev), k.to(dev), v.to(dev), causal=True)
    o_ref, lse_ref = naive.forward(f64(q), f64(k), f64(v), 1 / math.sqrt(128), True)
    check_out(f64(o.cpu()), f64(lse.cpu()), o_ref, lse_ref, "after timeout")
    assert fa.fa_get_last_device_error()[0] == fa.FA_OK
