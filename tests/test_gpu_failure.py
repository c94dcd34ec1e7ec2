"""Failure detection without a GPU fault.

Every mbarrier wait in the library's pipelines is bounded; when one runs out
the kernel sets a bit in the device error word and returns instead of
hanging, and the host reads BW_ERR_TIMEOUT.  The same holds for the
persistent decoder's polls for another CTA's output.  The self-test makes
one wait of each kind run out on purpose (an arrival that never comes, and
exchange entries that nothing writes; ~10 ms limits); the context must stay
usable afterwards.
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import build_lib

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def bw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib()
    import bit_gemv_bitlinear_gb300 as mod
    return mod


def test_bounded_wait_reports_timeout_and_context_survives(bw):
    assert bw.bw_device_error() == 0          # nothing pending
    status, bits = bw.bw_selftest_wait_timeout()
    assert status == 6 and bits == 8 | 64     # BW_ERR_TIMEOUT, self-test bits
    assert bw.bw_device_error() == 0          # the word was cleared
    # the context still runs the real path correctly
    N, K = 64, 256
    case = synth.gemv_case(1, N, K, synth.base_seed(11))
    packed = bw.bw_repack(torch.from_numpy(case["canon"]).cuda(), N, K)
    acc = bw.bw_gemv_w2a8_acc(torch.from_numpy(case["q"]).cuda(), packed, N, K)
    torch.cuda.synchronize()
    ref = oracle.gemv_acc(case["q"], case["canon"], N, K)
    assert (acc.cpu().numpy() == ref).all()
    assert bw.bw_device_error() == 0
