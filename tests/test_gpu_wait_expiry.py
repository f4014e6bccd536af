"""Failure detection on the GPU without a fault: a bounded in-kernel wait that runs out.

Every mbarrier wait in the layer's kernels gives up after about one second, sets
MOE_DEVERR_TIMEOUT in the device error word and lets the kernel return.  moe_selftest_wait_expiry
waits on a barrier phase that nothing completes while holding TMEM, then takes the GEMM kernels'
abort teardown; the test checks the status it leaves, then runs a layer step on the same context
against the oracle."""
import ctypes

import pytest

import synth
from moe_helpers import TOL_BF16, bf16_tensor_to_f64, compare_layer, make_plan, oracle_layer, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_expired_wait_sets_the_timeout_bit_and_leaves_the_context_usable():
    from decode_batches_gb300 import DEVERR_TIMEOUT, load_library
    lib = load_library()
    lib.moe_selftest_wait_expiry.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.moe_selftest_wait_expiry.restype = ctypes.c_int
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = torch.zeros(3, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert lib.moe_selftest_wait_expiry(ctypes.c_void_p(err.data_ptr()), ctypes.c_void_p(res.data_ptr()),
                                        ctypes.c_void_p(st)) == 0
    torch.cuda.synchronize()                 # raises if the context were lost
    completed, waited_ms, aborted = res.cpu().tolist()
    assert completed == 2                    # the wait gave up
    assert 900 <= waited_ms <= 5000          # after the ~1 s limit, not at once and not much later
    assert aborted == 1                      # and raised the CTA's abort flag
    assert int(err.item()) & DEVERR_TIMEOUT
    assert lib.moe_selftest_wait_expiry(None, None, None) == 1     # MOE_ERR_INVALID_ARG, no launch

    w = synth.workload("tiny")
    plan = make_plan(w)
    out = bf16_tensor_to_f64(plan.forward(to_dev(w.x(), "bf16"), n_prefill=w.T))
    compare_layer(out, oracle_layer(w), w.spec.k, TOL_BF16)
    assert plan.device_error() == 0
