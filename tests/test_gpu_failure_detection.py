"""Failure detection without a GPU fault: every device-side wait of the library is bounded.

dsa_check_bounded_wait runs the library's bounded wait on barriers that nothing completes.  The
first wait must give up after about one second, leave a timeout in the device error word and
raise the CTA's abort flag; the second must then return at once.  Afterwards the error is
reported once by dsa_get_device_error, and the context still runs the fused path correctly.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import overlap, to_dev

pytestmark = pytest.mark.gpu

DSA_OK, DSA_ERR_TIMEOUT = 0, 5


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_indexer_e4m3_gb300 as m
    from sparse_attention_indexer_e4m3_gb300 import build

    build.build()
    m.load()
    return m


def test_expired_wait_is_reported_and_context_survives(dsa):
    wl = W.make_config("tiny")
    t = to_dev(wl)
    before = dsa.index_topk(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], wl.topk).cpu().numpy()
    assert dsa.get_device_error() == DSA_OK

    first, second = dsa.check_bounded_wait()
    assert 0.9e9 <= first <= 3e9, first      # gave up after the limit, not before and not never
    assert second < 5e6, second              # saw the abort flag instead of waiting its own limit
    assert dsa.get_device_error() == DSA_ERR_TIMEOUT
    assert dsa.get_device_error() == DSA_OK  # read once, then cleared

    after = dsa.index_topk(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], wl.topk).cpu().numpy()
    assert dsa.get_device_error() == DSA_OK
    assert np.array_equal(before, after)
    ref = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke)
    assert overlap(after, O.topk(ref, wl.topk)) >= 0.999
