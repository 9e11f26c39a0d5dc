"""Failure detection on the GPU without a fault: a bounded device wait is made
to run out (an mbarrier nothing arrives on), the host reads the error status,
and the context keeps working."""
import ctypes

import pytest
import torch

import gated_delta_rule_37_gb300 as gdr
import oracle
from gated_delta_rule_37_gb300 import workloads
from tests.gpu_util import check_out, check_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdr.load()


def test_bounded_wait_gives_up_and_context_stays_usable():
    lib = gdr.load()
    assert gdr.device_status() == 0, "error word not clean before the test"
    assert lib.gdr_selftest_bounded_wait(None) == 0
    torch.cuda.synchronize()
    w = ctypes.c_int(0)
    assert lib.gdr_get_device_status(None, ctypes.byref(w)) == 5      # GDR_ERR_DEVICE_TIMEOUT
    assert w.value & 0x100
    assert b"device error word" in lib.gdr_last_error()
    assert gdr.device_status() == 0, "reading the status clears the word"
    # the context is intact: a prefill call still matches the oracle
    case = workloads.chunk_case(71, [130, 3], 2, 2, 128, 128, gate="g", g_range=(-1.0, 0.0), h0_std=0.1)
    dev = torch.device("cuda:0")
    o, sf = gdr.chunk_fwd(case.q.to(dev), case.k.to(dev), case.v.to(dev), case.beta.to(dev), case.cu_seqlens.to(dev),
                          g=case.g.to(dev), initial_state=case.initial_state.to(dev), scale=case.scale)
    torch.cuda.synchronize()
    assert gdr.device_status() == 0
    ro, rs = oracle.tokenwise(case.q, case.k, case.v, case.beta, case.cu_seqlens, g=case.g,
                              initial_state=case.initial_state, scale=case.scale)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")
