"""The allocation-free grouping call (moe_permute_static) against the oracle and moe_permute.

moe_permute_static is for callers that cannot allocate device memory (a memory planner that
owns the device, latency-critical paths where cudaMalloc would synchronise the device): it uses a
fixed scratch array inside the library instead of a plan workspace.  This file is collected last;
it must pass on its own in a fresh process and after every other test.  Grouping is integer
work, so every comparison is bit-exact: against the oracle's histogram, scan and stable
permutation, and against moe_permute, on two calls in a row with different ids (the scratch keeps
the previous call's contents, which must not leak into the next result)."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
    counts = torch.full((E,), -7, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    perm = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    inv = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    st = lib.moe_permute_static(E, k, ctypes.c_void_p(ids.data_ptr()), T, ctypes.c_void_p(counts.data_ptr()),
                                ctypes.c_void_p(offsets.data_ptr()), ctypes.c_void_p(perm.data_ptr()),
                                ctypes.c_void_p(inv.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return counts, offsets, perm, inv


def _ids(rng, T, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


def _oracle_grouping(ids, E):
    """The oracle's counts, offsets, perm and inv of the assignments that are kept: an id in
    [0, E) that no earlier slot of its token already holds.  Dropped assignments sort last (key
    E) and get inv = -1; perm holds the kept rows only."""
    ids = np.asarray(ids)
    T, k = ids.shape
    keep = (ids >= 0) & (ids < E)
    for j in range(k):
        for q in range(j):
            keep[:, j] &= ids[:, q] != ids[:, j]
    key = np.where(keep, ids, E)
    counts = oracle.expert_histogram(key[keep], E) if keep.any() else np.zeros(E, np.int32)
    offsets = oracle.exclusive_offsets(counts)
    perm, inv = oracle.stable_permutation(key)
    n = int(offsets[-1])
    inv = np.where(keep.ravel(), inv, -1).astype(np.int32)
    return counts, offsets, perm[:n], inv


def _check_vs_oracle(got, ids, E):
    counts, offsets, perm, inv = (t.cpu().numpy() for t in got)
    oc, oo, op, oi = _oracle_grouping(ids, E)
    n = int(oo[-1])
    assert np.array_equal(counts, oc)
    assert np.array_equal(offsets, oo)
    assert np.array_equal(perm[:n], op)
    assert np.all(perm[n:] == -7)              # rows past the kept ones are not written
    assert np.array_equal(inv, oi)


@pytest.mark.parametrize("E,k,T1,T2", [(256, 8, 2051, 37), (384, 8, 48, 4099), (8, 2, 16, 1)])
def test_static_permute_matches_oracle_and_moe_permute_twice(E, k, T1, T2):
    from decode_batches_gb300 import MoePlan
    lib = _lib()
    rng = np.random.default_rng(E + T1)
    plan = MoePlan(E, k, 64, 64, 0, "bf16")
    plan.allocate_workspace(max(T1, T2))
    for T in (T1, T2):                       # two calls in a row on the shared scratch
        ids_np = _ids(rng, T, E, k)
        ids = torch.from_numpy(ids_np).cuda()
        got = _static_permute(lib, E, k, ids)
        want = plan.permute(ids)
        torch.cuda.synchronize()
        _check_vs_oracle(got, ids_np, E)
        for g, w in zip(got[:2], want[:2]):
            assert torch.equal(g, w)
        assert torch.equal(got[3], want[3])


def test_static_permute_empty_step():
    lib = _lib()
    E, k = 64, 4
    ids = torch.empty((0, k), dtype=torch.int32, device="cuda")
    counts, offsets, perm, inv = _static_permute(lib, E, k, ids)
    torch.cuda.synchronize()
    assert torch.all(counts == 0) and torch.all(offsets == 0)


def test_static_permute_drops_invalid_and_repeated_ids():
    """Out-of-range and repeated ids are dropped (inv = -1), the kept ones grouped as the oracle
    groups them; moe_permute agrees, and there it also raises the plan's error bit."""
    from decode_batches_gb300 import DEVERR_EXPERT_RANGE, MoePlan
    lib = _lib()
    E, k, T = 48, 4, 301
    rng = np.random.default_rng(5)
    ids_np = _ids(rng, T, E, k)
    ids_np[3, 1] = E                       # out of range
    ids_np[7, 0] = -1
    ids_np[10, 2] = ids_np[10, 0]          # repeat of an earlier slot
    ids_np[200, 3] = ids_np[200, 1]
    ids_np[299, :] = 5                     # one token with a single valid slot
    ids = torch.from_numpy(ids_np).cuda()
    got = _static_permute(lib, E, k, ids)
    torch.cuda.synchronize()
    _check_vs_oracle(got, ids_np, E)
    plan = MoePlan(E, k, 64, 64, 0, "bf16")
    plan.allocate_workspace(T)
    want = plan.permute(ids)
    for g, w in zip(got[:2], want[:2]):
        assert torch.equal(g, w)
    assert torch.equal(got[3], want[3])
    assert plan.device_error() & DEVERR_EXPERT_RANGE


def test_static_permute_at_the_capacity_limit():
    """ceil(T / 32) * E == 262144 exactly (1024 chunks, a multiple of 4): the mask array is
    filled completely."""
    from decode_batches_gb300 import MoePlan
    lib = _lib()
    E, k, T = 256, 8, 32768
    rng = np.random.default_rng(11)
    ids_np = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    ids = torch.from_numpy(ids_np).cuda()
    got = _static_permute(lib, E, k, ids)
    torch.cuda.synchronize()
    _check_vs_oracle(got, ids_np, E)
    plan = MoePlan(E, k, 64, 64, 0, "bf16")
    plan.allocate_workspace(T)
    want = plan.permute(ids)
    for g, w in zip(got, want):
        assert torch.equal(g, w)


def test_static_permute_rejects_oversized_inputs_without_launching():
    lib = _lib()
    E, k, T = 256, 8, 32 * 1024 + 1          # ceil(T / 32) * E > 262144
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(z.data_ptr())
    assert lib.moe_permute_static(E, k, p, T, p, p, p, p, None) == 4      # MOE_ERR_WORKSPACE
    assert lib.moe_permute_static(0, k, p, 4, p, p, p, p, None) == 1      # MOE_ERR_INVALID_ARG


# A fresh process (no torch CUDA state) that calls moe_permute_static, destroys its CUDA context
# with cudaDeviceReset, and calls it again in the new context: the scratch address must be looked
# up again there.  Device memory comes from the CUDA runtime directly (ctypes), not from torch.
_RESET_SCRIPT = r"""
import ctypes, sys
import numpy as np
sys.path.insert(0, ROOT)
import oracle
from decode_batches_gb300 import load_library
lib = load_library()
lib.moe_permute_static.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 5
rt = ctypes.CDLL("libcudart.so.13")
E, k, T = 64, 4, 777
rng = np.random.default_rng(3)

def run():
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    sizes = [ids.nbytes, 4 * E, 4 * (E + 1), 4 * T * k, 4 * T * k]
    ptrs = [ctypes.c_void_p() for _ in sizes]
    for p, n in zip(ptrs, sizes):
        assert rt.cudaMalloc(ctypes.byref(p), ctypes.c_size_t(n)) == 0
    assert rt.cudaMemcpy(ptrs[0], ids.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(ids.nbytes), 1) == 0
    assert lib.moe_permute_static(E, k, ptrs[0], T, ptrs[1], ptrs[2], ptrs[3], ptrs[4], None) == 0
    assert rt.cudaDeviceSynchronize() == 0
    out = [np.empty(n // 4, np.int32) for n in sizes[1:]]
    for o, p in zip(out, ptrs[1:]):
        assert rt.cudaMemcpy(o.ctypes.data_as(ctypes.c_void_p), p, ctypes.c_size_t(o.nbytes), 2) == 0
    counts, offsets, perm, inv = out
    oc = oracle.expert_histogram(ids, E)
    op, oi = oracle.stable_permutation(ids)
    assert np.array_equal(counts, oc) and np.array_equal(offsets, oracle.exclusive_offsets(oc))
    assert np.array_equal(perm, op) and np.array_equal(inv, oi)
    for p in ptrs:
        assert rt.cudaFree(p) == 0

assert rt.cudaSetDevice(0) == 0
run()
assert rt.cudaDeviceReset() == 0
run()
print("reset-ok")
"""


def test_static_permute_after_context_reset():
    code = _RESET_SCRIPT.replace("ROOT", repr(ROOT))
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300,
                         env=dict(os.environ, CUDA_VISIBLE_DEVICES=os.environ.get("CUDA_VISIBLE_DEVICES", "0")))
    assert res.returncode == 0 and "reset-ok" in res.stdout, res.stdout[-2000:] + res.stderr[-2000:]
