"""The allocation-free grouping call (moe_permute_static) against moe_permute.

moe_permute_static is for callers that cannot allocate device memory (a memory planner that
owns the device, latency-critical paths where cudaMalloc would synchronise the device): it uses a fixed scratch array inside
the library instead of a plan workspace.  This file is collected last; it must pass on its own
in a fresh process and after every other test.  Grouping is integer work, so the comparison is
bit-exact, on two calls in a row with different ids (the scratch keeps the previous call's
contents, which must not leak into the next result)."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _lib():
    from decode_batches_gb300 import load_library
    lib = load_library()
    lib.moe_permute_static.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.moe_permute_static.restype = ctypes.c_int
    return lib


def _static_permute(lib, E, k, ids):
    T = ids.shape[0]
    dev = ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    inv = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    st = lib.moe_permute_static(E, k, ctypes.c_void_p(ids.data_ptr()), T, ctypes.c_void_p(counts.data_ptr()),
                                ctypes.c_void_p(offsets.data_ptr()), ctypes.c_void_p(perm.data_ptr()),
                                ctypes.c_void_p(inv.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return counts, offsets, perm, inv


def _ids(rng, T, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("E,k,T1,T2", [(256, 8, 2051, 37), (384, 8, 48, 4099), (8, 2, 16, 1)])
def test_static_permute_matches_moe_permute_twice(E, k, T1, T2):
    from decode_batches_gb300 import MoePlan
    lib = _lib()
    rng = np.random.default_rng(E + T1)
    plan = MoePlan(E, k, 64, 64, 0, "bf16")
    plan.allocate_workspace(max(T1, T2))
    for T in (T1, T2):                       # two calls in a row on the shared scratch
        ids = torch.from_numpy(_ids(rng, T, E, k)).cuda()
        got = _static_permute(lib, E, k, ids)
        want = plan.permute(ids)
        torch.cuda.synchronize()
        for g, w in zip(got, want):
            assert torch.equal(g, w)


def test_static_permute_rejects_oversized_inputs_without_launching():
    lib = _lib()
    E, k, T = 256, 8, 32 * 1024 + 1          # ceil(T / 32) * E > 262144
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(z.data_ptr())
    assert lib.moe_permute_static(E, k, p, T, p, p, p, p, None) == 4      # MOE_ERR_WORKSPACE
    assert lib.moe_permute_static(0, k, p, 4, p, p, p, p, None) == 1      # MOE_ERR_INVALID_ARG
