"""GPU parity of the routing and grouping steps against the fp64 oracle (bit-exact where the
step is integer work, stated tolerances for floating point).  All calls go through the C ABI."""
import functools

import numpy as np
import pytest

import oracle
import synth
from moe_helpers import TOL_GATES, TOL_LOGITS, make_plan, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ROUTE_CASES = [("tiny", 0), ("decode", 0), ("mixed", 128), ("mixed", 2048), ("mixed", 8192), ("fp4_zipf", 0),
               ("verify", 0)]


@functools.lru_cache(maxsize=None)
def workload(name, q):
    return synth.workload(name, quantum=q or 2048)


@functools.lru_cache(maxsize=None)
def router_plan(spec):
    """A plan with this spec's router and tiny stand-in experts (routing needs only W_r, b)."""
    from decode_batches_gb300 import MoePlan

    wl = {synth.TINY: workload("tiny", 0), synth.QWEN_A3B_LIKE: workload("mixed", 8192),
          synth.FP4_ZIPF: workload("fp4_zipf", 0)}[spec]
    plan = MoePlan(spec.E, spec.k, spec.d, 64, 0, "bf16")
    z = torch.zeros((spec.E, 64, spec.d), dtype=torch.bfloat16, device="cuda")
    b = wl.router_bias()
    plan.set_weights(to_dev(wl.router_weight()), to_dev(b) if b is not None else None, z, z,
                     torch.zeros((spec.E, spec.d, 64), dtype=torch.bfloat16, device="cuda"))
    plan.allocate_workspace(8195)
    return plan


def _oracle_logits(w):
    x = oracle.bf16_to_f64(w.x())
    b = w.router_bias()
    return oracle.router_logits(x, w.router_weight().astype(np.float64), None if b is None else b.astype(np.float64))


@pytest.mark.parametrize("name,q", ROUTE_CASES)
def test_route_logits_bit_exact(name, q):
    """Given identical fp32 logits, ids match the oracle's selection exactly; gates to fp32 rounding."""
    w = workload(name, q)
    plan = router_plan(w.spec)
    l32 = _oracle_logits(w).astype(np.float32)
    ids, gates = plan.route_logits(to_dev(l32))
    ids = ids.cpu().numpy()
    want = oracle.select_topk(l32, w.spec.k)
    np.testing.assert_array_equal(ids, want)
    g_ref = oracle.topk_gates(l32, want)
    np.testing.assert_allclose(gates.cpu().numpy(), g_ref, rtol=TOL_GATES, atol=1e-7)
    assert plan.device_error() == 0


@pytest.mark.parametrize("name,q", ROUTE_CASES)
def test_route_from_x(name, q):
    """GPU logits vs fp64 within 1e-5 RMS; ids/gates are the oracle's selection on the GPU logits."""
    w = workload(name, q)
    plan = router_plan(w.spec)
    logits, ids, gates = plan.route(to_dev(w.x(), "bf16"))
    lg = logits.cpu().numpy()
    ref = _oracle_logits(w)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.abs(lg - ref).max() <= TOL_LOGITS * rms, np.abs(lg - ref).max() / rms
    want = oracle.select_topk(lg, w.spec.k)
    np.testing.assert_array_equal(ids.cpu().numpy(), want)
    np.testing.assert_allclose(gates.cpu().numpy(), oracle.topk_gates(lg, want), rtol=TOL_GATES, atol=1e-7)


def _route_only_plan(E, k):
    from decode_batches_gb300 import MoePlan
    return MoePlan(E, k, 64, 64, 0, "bf16")


@pytest.mark.parametrize("E,k,T", [(8, 2, 1), (40, 8, 33), (32, 32, 5), (33, 32, 5), (256, 8, 70), (1024, 32, 3), (384, 8, 31)])
def test_route_logits_adversarial(E, k, T):
    plan = _route_only_plan(E, k)
    rng = np.random.default_rng(E * 7 + k)
    cases = [
        np.zeros((T, E), np.float32),                                        # the tie-break decides all
        np.where(rng.random((T, E)) < 0.5, -0.0, 0.0).astype(np.float32),    # signed zeros are equal
        rng.integers(-3, 4, size=(T, E)).astype(np.float32),                 # many ties
        rng.normal(size=(T, E)).astype(np.float32) * 30,                     # wide range
        np.broadcast_to(np.arange(E, dtype=np.float32), (T, E)).copy(),      # ascending: picks the top indices
    ]
    for L in cases:
        ids, gates = plan.route_logits(to_dev(L))
        want = oracle.select_topk(L, k)
        np.testing.assert_array_equal(ids.cpu().numpy(), want)
        np.testing.assert_allclose(gates.cpu().numpy(), oracle.topk_gates(L, want), rtol=TOL_GATES, atol=1e-7)
    assert plan.device_error() == 0


def test_route_logits_nonfinite_flags_device_error():
    plan = _route_only_plan(16, 4)
    L = np.zeros((3, 16), np.float32)
    L[1, 5] = np.nan
    L[2, 0] = np.inf
    ids, _ = plan.route_logits(to_dev(L))
    # NaN ranks below every number (row 1 never selects expert 5); +inf is selected first (row 2)
    np.testing.assert_array_equal(ids.cpu().numpy(), oracle.select_topk(L, 4))
    assert plan.device_error() & 0x2


def _distinct_ids(rng, T, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else np.zeros((0, k), np.int32)


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (31, 8, 2), (32, 8, 2), (33, 256, 8), (100, 5, 5), (1000, 384, 8),
                                   (4099, 1024, 32), (8195, 256, 8)])
def test_permute_bit_exact(T, E, k):
    plan = _route_only_plan(E, k)
    plan.allocate_workspace(T)
    ids = _distinct_ids(np.random.default_rng(T), T, E, k)
    counts, offsets, perm, inv = plan.permute(to_dev(ids))
    c_ref = oracle.expert_histogram(ids, E)
    p_ref, i_ref = oracle.stable_permutation(ids)
    np.testing.assert_array_equal(counts.cpu().numpy(), c_ref)
    np.testing.assert_array_equal(offsets.cpu().numpy(), oracle.exclusive_offsets(c_ref))
    np.testing.assert_array_equal(perm.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(inv.cpu().numpy(), i_ref)
    assert plan.device_error() == 0


@pytest.mark.parametrize("name,q", [("mixed", 2048), ("fp4_zipf", 0), ("verify", 0)])
def test_permute_of_workload_routing(name, q):
    w = workload(name, q)
    plan = router_plan(w.spec)
    _, ids, _ = plan.route(to_dev(w.x(), "bf16"), want_logits=False)
    ids_np = ids.cpu().numpy()
    counts, offsets, perm, inv = plan.permute(ids)
    p_ref, i_ref = oracle.stable_permutation(ids_np)
    np.testing.assert_array_equal(counts.cpu().numpy(), oracle.expert_histogram(ids_np, w.spec.E))
    np.testing.assert_array_equal(perm.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(inv.cpu().numpy(), i_ref)
    assert int(counts.sum()) == w.T * w.spec.k


def test_permute_flags_and_drops_invalid_ids():
    E, k, T = 6, 3, 5
    plan = _route_only_plan(E, k)
    plan.allocate_workspace(T)
    ids = np.array([[0, 1, 2], [3, -1, 4], [5, 5, 0], [1, 6, 2], [2, 3, 4]], np.int32)
    counts, offsets, perm, inv = plan.permute(to_dev(ids))
    assert plan.device_error() & 0x1
    valid = np.array([[True, True, True], [True, False, True], [True, False, True], [True, False, True],
                      [True, True, True]])
    flat = ids.ravel()
    kept = np.where(valid.ravel())[0]
    want_perm = [a for e in range(E) for a in kept if flat[a] == e]
    n = len(want_perm)
    assert offsets.cpu().numpy()[-1] == n
    np.testing.assert_array_equal(perm.cpu().numpy()[:n], want_perm)
    inv_np = inv.cpu().numpy()
    assert np.all(inv_np[~valid.ravel()] == -1)
    assert np.all(perm.cpu().numpy()[inv_np[valid.ravel()]] == kept)
