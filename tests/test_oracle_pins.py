"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test checks one oracle function against the pages' printed numbers, a closed form,
brute force on tiny inputs, or an invariant of the mathematics, chosen so that a plausible
mistake (a dropped term, a wrong sign or index, a transposed operand, silu on the wrong
projection, an unstable sort) fails at least one of them.  CPU only.
"""
import itertools
import math
import os

import numpy as np
import pytest
from scipy.special import softmax as scipy_softmax

import oracle
from oracle import moe_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_to_bf16_bits_exact(v):
    """bf16 bits of values that are exactly representable in bf16 (checked)."""
    a = np.asarray(v, dtype=np.float32)
    bits = a.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not representable in bf16"
    return (bits >> 16).astype(np.uint16)


# ------------------------------------------------------------------------------------------
# number formats
# ------------------------------------------------------------------------------------------

def test_bf16_known_patterns():
    pats = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000, 0x3E80, 0x4049], np.uint16)
    want = [1.0, -2.0, 2.0 ** -133, (2.0 - 2.0 ** -7) * 2.0 ** 127, 0.0, 0.25, 3.140625]
    got = oracle.bf16_to_f64(pats)
    assert list(got) == want
    assert math.copysign(1.0, got[4]) == -1.0


def _e2m1_from_bitfields(c):
    # OCP MX v1.0 FP4 E2M1: S EE M, exponent bias 1; E = 0 is subnormal (M * 2^-1).
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    mag = (m * 0.5) if e == 0 else (2.0 ** (e - 1)) * (1.0 + m / 2.0)
    return -mag if s else mag


def test_e2m1_all_codes_match_bitfield_definition():
    for c in range(16):
        assert oracle.e2m1_value(c) == _e2m1_from_bitfields(c), c
    assert [abs(oracle.e2m1_value(c)) for c in range(8)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_mxfp4_decode_nibble_order_and_scale():
    # one 32-element block: bytes 0x21 -> element0 = code 1 (0.5), element1 = code 2 (1.0)
    codes = np.zeros((1, 16), np.uint8)
    codes[0, 0] = 0x21
    codes[0, 1] = 0x9F        # element2 = code 15 (-6), element3 = code 9 (-0.5)
    codes[0, 15] = 0x70       # element30 = 0, element31 = code 7 (6)
    for s in (1, 100, 120, 127, 130, 200, 254):
        scale = 2.0 ** (s - 127)
        got = oracle.mxfp4_decode(codes, np.array([[s]], np.uint8))[0]
        want = np.zeros(32)
        want[0], want[1], want[2], want[3], want[31] = 0.5, 1.0, -6.0, -0.5, 6.0
        np.testing.assert_array_equal(got, want * scale)
    # the all-6 row at scale 2^0 decodes to 6.0 everywhere
    got = oracle.mxfp4_decode(np.full((2, 16), 0x77, np.uint8), np.full((2, 1), 127, np.uint8))
    assert np.all(got == 6.0)
    # two blocks per row: the second block's scale applies to elements 32..63 only
    codes2 = np.full((1, 32), 0x22, np.uint8)
    got = oracle.mxfp4_decode(codes2, np.array([[127, 129]], np.uint8))[0]
    assert np.all(got[:32] == 1.0) and np.all(got[32:] == 4.0)


# ------------------------------------------------------------------------------------------
# router
# ------------------------------------------------------------------------------------------

def test_router_logits_hand_example_nonsquare():
    x = np.array([[1.0, 2.0]])
    w = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])      # [E=3][d=2]
    b = np.array([0.0, 0.5, -1.0])
    np.testing.assert_array_equal(moe_ref.router_logits(x, w, b), [[1.0, 2.5, 2.0]])
    np.testing.assert_array_equal(moe_ref.router_logits(x, w, None), [[1.0, 2.0, 3.0]])


def _is_valid_topk(v, ids, k):
    """Brute-force property: S beats every unselected expert, and S is listed in order."""
    E = len(v)
    S = list(ids)
    if len(set(S)) != k:
        return False

    def beats(a, b):  # a strictly before b in the total order; NaN below everything
        va, vb = v[a], v[b]
        if math.isnan(va) and math.isnan(vb):
            return a < b
        if math.isnan(va):
            return False
        if math.isnan(vb):
            return True
        return va > vb or (va == vb and a < b)

    for a in S:
        for b in range(E):
            if b not in S and not beats(a, b):
                return False
    return all(beats(S[i], S[i + 1]) for i in range(k - 1))


def test_select_topk_bruteforce_with_ties():
    rng = np.random.default_rng(1)
    for E, k in [(5, 2), (8, 3), (9, 9), (33, 8), (40, 1)]:
        vals = rng.integers(-2, 3, size=(60, E)).astype(np.float32)  # many ties
        ids = oracle.select_topk(vals, k)
        for t in range(vals.shape[0]):
            assert _is_valid_topk(vals[t].tolist(), ids[t].tolist(), k), (E, k, vals[t], ids[t])


def test_select_topk_special_values():
    assert oracle.select_topk(np.zeros((1, 6)), 3).tolist() == [[0, 1, 2]]
    assert oracle.select_topk(np.array([[-0.0, 0.0, -1.0]]), 2).tolist() == [[0, 1]]
    assert oracle.select_topk(np.array([[0.0, -0.0, -1.0]]), 2).tolist() == [[0, 1]]
    assert oracle.select_topk(np.array([[np.nan, 1.0, -np.inf, np.nan]]), 4).tolist() == [[1, 2, 0, 3]]
    assert oracle.select_topk(np.array([[1.0, 3.0, 2.0, 3.0]]), 3).tolist() == [[1, 3, 2]]


def test_gates_closed_form():
    logits = np.array([[math.log(3.0), 0.0, -5.0, math.log(1.0) - 0.0]])
    ids = oracle.select_topk(logits, 2)        # ln3 then 0 (index 1 beats index 3 on the tie)
    assert ids.tolist() == [[0, 1]]
    np.testing.assert_allclose(oracle.topk_gates(logits, ids), [[0.75, 0.25]], rtol=0, atol=1e-15)
    # k = 1 -> gate 1; a constant shift of every logit leaves gates unchanged
    rng = np.random.default_rng(2)
    L = rng.normal(size=(7, 11))
    ids = oracle.select_topk(L, 4)
    g = oracle.topk_gates(L, ids)
    np.testing.assert_allclose(oracle.topk_gates(L + 123.25, oracle.select_topk(L + 123.25, 4)), g, rtol=1e-12)
    np.testing.assert_allclose(g.sum(axis=1), 1.0, rtol=1e-15)
    assert np.all(np.diff(g, axis=1) <= 0)  # slot order is value order
    np.testing.assert_array_equal(oracle.topk_gates(L, oracle.select_topk(L, 1)), 1.0)


def test_gates_equal_renormalised_full_softmax():
    rng = np.random.default_rng(3)
    L = rng.normal(size=(5, 16)) * 3
    ids = oracle.select_topk(L, 5)
    full = scipy_softmax(L, axis=1)
    sel = np.take_along_axis(full, ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(oracle.topk_gates(L, ids), sel / sel.sum(axis=1, keepdims=True), rtol=1e-13)


def test_topk_margin_hand_example():
    L = np.array([[5.0, 1.0, 3.0, 2.5], [0.0, 0.0, 0.0, 0.0]])
    np.testing.assert_array_equal(oracle.topk_margin(L, 2), [0.5, 0.0])
    assert np.isinf(oracle.topk_margin(L, 4)).all()


# ------------------------------------------------------------------------------------------
# grouping
# ------------------------------------------------------------------------------------------

def _distinct_ids(rng, T, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


def test_histogram_scan_permutation_bruteforce():
    rng = np.random.default_rng(4)
    for T, E, k in [(1, 4, 4), (7, 5, 2), (13, 16, 3), (40, 9, 8)]:
        ids = _distinct_ids(rng, T, E, k)
        flat = ids.ravel().tolist()
        counts = oracle.expert_histogram(ids, E)
        off = oracle.exclusive_offsets(counts)
        perm, inv = oracle.stable_permutation(ids)
        # nested-loop construction of the stable grouping
        want_perm = [a for e in range(E) for a in range(T * k) if flat[a] == e]
        want_counts = [sum(1 for a in flat if a == e) for e in range(E)]
        assert perm.tolist() == want_perm
        assert counts.tolist() == want_counts
        assert off.tolist() == [sum(want_counts[:e]) for e in range(E + 1)]
        assert int(counts.sum()) == T * k and off[-1] == T * k
        assert np.all(inv[perm] == np.arange(T * k)) and np.all(perm[inv] == np.arange(T * k))
        for e in range(E):
            seg = perm[off[e]:off[e + 1]]
            assert all(flat[a] == e for a in seg)
            assert np.all(np.diff(seg) > 0)


# ------------------------------------------------------------------------------------------
# expert FFN
# ------------------------------------------------------------------------------------------

def test_swiglu_closed_form_gate_first():
    # d = f = 1: y = W_d * silu(W_g x) * (W_u x); silu(ln 3) = ln 3 * sigmoid(ln 3) = 0.75 ln 3
    x = np.array([[1.0]])
    y = moe_ref.swiglu_ffn(x, np.array([[math.log(3.0)]]), np.array([[2.0]]), np.array([[5.0]]))
    assert abs(y[0, 0] - 7.5 * math.log(3.0)) < 1e-14
    # gate and up swapped: 5 * silu(2) * ln 3, which differs
    y2 = moe_ref.swiglu_ffn(x, np.array([[2.0]]), np.array([[math.log(3.0)]]), np.array([[5.0]]))
    silu2 = 2.0 / (1.0 + math.exp(-2.0))
    assert abs(y2[0, 0] - 5.0 * silu2 * math.log(3.0)) < 1e-13
    assert abs(y2[0, 0] - y[0, 0]) > 0.1
    # silu(0) = 0 whatever the up projection is
    assert moe_ref.swiglu_ffn(x, np.array([[0.0]]), np.array([[9.0]]), np.array([[1.0]]))[0, 0] == 0.0


def test_swiglu_nonsquare_orientation():
    # d = 2, f = 3: gate/up are [f][d], down is [d][f]
    x = np.array([[1.0, -1.0]])
    wg = np.array([[math.log(3.0) + 1.0, 1.0], [0.0, 0.0], [1.0, 1.0]])   # u = [ln3, 0, 0]
    wu = np.array([[2.0, 0.0], [1.0, 0.0], [0.0, -4.0]])                   # v = [2, 1, 4]
    wd = np.array([[1.0, 10.0, 100.0], [-1.0, 0.0, 0.0]])                  # y = [h0, -h0] (h1=h2=0)
    y = moe_ref.swiglu_ffn(x, wg, wu, wd)
    h0 = 0.75 * math.log(3.0) * 2.0
    np.testing.assert_allclose(y, [[h0, -h0]], rtol=1e-14)


# ------------------------------------------------------------------------------------------
# combine and the whole layer
# ------------------------------------------------------------------------------------------

def test_combine_hand_example():
    # T = 2, k = 2, d = 1; assignment a = t*k + j lives at row inv[a] of y
    y = np.array([[10.0], [20.0], [30.0], [40.0]])
    inv = np.array([2, 0, 3, 1], np.int32)
    g = np.array([[0.25, 0.75], [0.5, 0.5]])
    out = moe_ref.combine(y, g, inv, np.array([[1.0], [2.0]]))
    np.testing.assert_array_equal(out, [[0.25 * 30 + 0.75 * 10 + 1.0], [0.5 * 40 + 0.5 * 20 + 2.0]])


def _rand_layer(rng, T, E, k, d, f, n_shared=0, f_s=0, bias=False):
    x = f32_to_bf16_bits_exact(np.round(rng.normal(size=(T, d)) * 8) / 8)
    wr = (rng.normal(size=(E, d)) * 0.3).astype(np.float32)
    b = (rng.normal(size=E) * 0.1).astype(np.float32) if bias else None
    q = lambda *s: f32_to_bf16_bits_exact(np.round(rng.normal(size=s) * 16) / 64)
    ex = oracle.DecodedExperts(q(E, f, d), q(E, f, d), q(E, d, f))
    sh = (q(n_shared, f_s, d), q(n_shared, f_s, d), q(n_shared, d, f_s)) if n_shared else None
    return x, wr, b, ex, sh


def _dense_masked(x_bits, wr, b, k, ex, sh):
    """All experts on all tokens, weighted by a gate matrix that is zero off the top-k."""
    x = oracle.bf16_to_f64(x_bits)
    L = x @ wr.astype(np.float64).T + (0 if b is None else b.astype(np.float64))
    E = wr.shape[0]
    G = np.zeros((x.shape[0], E))
    for t in range(x.shape[0]):
        order = sorted(range(E), key=lambda e: (-L[t, e], e))[:k]
        w = np.exp(np.array([L[t, e] for e in order]) - L[t, order[0]])
        G[t, order] = w / w.sum()
    out = np.zeros_like(x)
    for e in range(E):
        wg, wu, wd = ex.expert(e)
        u = np.einsum("td,fd->tf", x, wg)
        v = np.einsum("td,fd->tf", x, wu)
        out += G[:, e:e + 1] * np.einsum("tf,df->td", u * (1 / (1 + np.exp(-u))) * v, wd)
    if sh is not None:
        for s in range(sh[0].shape[0]):
            wg, wu, wd = (oracle.bf16_to_f64(w[s]) for w in sh)
            u, v = x @ wg.T, x @ wu.T
            out += (u * (1 / (1 + np.exp(-u))) * v) @ wd.T
    return out


@pytest.mark.parametrize("T,E,k,d,f,ns,fs,bias", [(5, 6, 2, 16, 8, 0, 0, False), (9, 7, 3, 8, 24, 1, 16, True),
                                                  (4, 5, 5, 8, 8, 2, 8, False)])
def test_dense_masked_equals_sparse(T, E, k, d, f, ns, fs, bias):
    rng = np.random.default_rng(T * 100 + E)
    x, wr, b, ex, sh = _rand_layer(rng, T, E, k, d, f, ns, fs, bias)
    res = oracle.moe_layer(x, wr, b, k, ex, sh)
    dense = _dense_masked(x, wr, b, k, ex, sh)
    np.testing.assert_allclose(res["out"], dense, rtol=1e-12, atol=1e-12 * np.abs(dense).max())


def test_k_equals_E_single_token_is_dense_softmax_mixture():
    rng = np.random.default_rng(5)
    E, d, f = 6, 8, 12
    x, wr, b, ex, _ = _rand_layer(rng, 1, E, E, d, f)
    res = oracle.moe_layer(x, wr, None, E, ex)
    xv = oracle.bf16_to_f64(x)[0]
    p = scipy_softmax(xv @ wr.astype(np.float64).T)
    want = np.zeros(d)
    for e in range(E):
        wg, wu, wd = ex.expert(e)
        u, v = wg @ xv, wu @ xv
        want += p[e] * (wd @ (u * v / (1.0 + np.exp(-u))))
    np.testing.assert_allclose(res["out"][0], want, rtol=1e-12, atol=1e-13)


def test_layer_token_permutation_and_prefill_independence():
    rng = np.random.default_rng(6)
    x, wr, b, ex, sh = _rand_layer(rng, 11, 9, 3, 16, 8, 1, 8, True)
    res = oracle.moe_layer(x, wr, b, 3, ex, sh, n_prefill=0)
    p = rng.permutation(11)
    res_p = oracle.moe_layer(x[p], wr, b, 3, ex, sh, n_prefill=7)
    np.testing.assert_allclose(res_p["out"], res["out"][p], rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(res_p["ids"], res["ids"][p])


def test_layer_gate_up_swap_changes_output():
    rng = np.random.default_rng(7)
    x, wr, b, ex, _ = _rand_layer(rng, 6, 4, 2, 8, 8)
    swapped = oracle.DecodedExperts(ex.up, ex.gate, ex.down)
    a = oracle.moe_layer(x, wr, None, 2, ex)["out"]
    c = oracle.moe_layer(x, wr, None, 2, swapped)["out"]
    assert np.abs(a - c).max() > 1e-3 * np.abs(a).max()


def test_shared_experts_sum_with_weight_one():
    rng = np.random.default_rng(8)
    x, wr, b, ex, sh = _rand_layer(rng, 5, 4, 2, 8, 8, 1, 16)
    two = tuple(np.concatenate([w, w]) for w in sh)
    one = oracle.moe_layer(x, wr, None, 2, ex, sh)
    both = oracle.moe_layer(x, wr, None, 2, ex, two)
    none = oracle.moe_layer(x, wr, None, 2, ex, None)
    np.testing.assert_allclose(both["out"] - none["out"], 2 * (one["out"] - none["out"]), rtol=1e-12, atol=1e-13)


def test_fp4_experts_equal_bf16_experts_holding_decoded_values():
    # every e2m1 value times a power of two is exact in bf16, so both storage forms must agree
    rng = np.random.default_rng(9)
    E, d, f, T, k = 3, 64, 32, 5, 2
    codes = lambda *s: rng.integers(0, 256, size=s, dtype=np.uint8)
    scales = lambda *s: rng.integers(118, 134, size=s, dtype=np.uint8)
    gc, uc, dc = codes(E, f, d // 2), codes(E, f, d // 2), codes(E, d, f // 2)
    gs, us, ds = scales(E, f, d // 32), scales(E, f, d // 32), scales(E, d, f // 32)
    fp4 = oracle.DecodedExperts(gc, uc, dc, gs, us, ds)
    bf = oracle.DecodedExperts(*(f32_to_bf16_bits_exact(oracle.mxfp4_decode(c, s).astype(np.float32))
                                 for c, s in ((gc, gs), (uc, us), (dc, ds))))
    x = f32_to_bf16_bits_exact(np.round(rng.normal(size=(T, d)) * 4) / 4)
    wr = rng.normal(size=(E, d)).astype(np.float32)
    np.testing.assert_array_equal(oracle.moe_layer(x, wr, None, k, fp4)["out"],
                                  oracle.moe_layer(x, wr, None, k, bf)["out"])


# ------------------------------------------------------------------------------------------
# the pages' worked numbers
# ------------------------------------------------------------------------------------------

def _golden_rows():
    rows, inv = [], []
    with open(os.path.join(GOLDEN, "p1_table9.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "INV":
                inv.append(tuple(float(p) for p in parts[1:]))
            else:
                rows.append(tuple(float(p) for p in parts))
    return rows, inv


def test_table9_unique_experts_and_tokens_per_expert():
    rows, inv = _golden_rows()
    assert rows and inv
    for E, k, Q, uniq, tpe in rows:
        u = oracle.expected_unique_experts(int(E), int(k), int(Q))
        if uniq == 256:
            assert round(u) == 256          # printed as the whole number from Q = 512 on
        else:
            assert round(u, 1) == uniq
        assert oracle.tokens_per_expert(int(Q), int(k), int(E)) == tpe
    for target, E, k, Q in inv:
        assert oracle.quantum_for_tokens_per_expert(target, int(E), int(k)) == Q


def test_selection_wakes_the_expected_number_of_experts():
    """Uniform routing (iid logits) through select_topk wakes E(1-(1-k/E)^Q) experts on average."""
    rng = np.random.default_rng(10)
    E, k, Q, draws = 256, 6, 128, 400
    uniq = np.empty(draws)
    for i in range(draws):
        ids = oracle.select_topk(rng.normal(size=(Q, E)), k)
        uniq[i] = len(np.unique(ids))
    want = oracle.expected_unique_experts(E, k, Q)          # 243.7 per the page
    assert abs(uniq.mean() - want) < 4 * uniq.std() / math.sqrt(draws) + 0.05
    # tokens per expert: counts average Q*k/E (Table 9: 3.0 at Q = 128)
    counts = oracle.expert_histogram(oracle.select_topk(rng.normal(size=(Q, E)), k), E)
    assert counts.sum() == Q * k and counts.mean() == 3.0


# ---------------------------------------------------------------------------------------
# Prefill chunking of the serving loop ("moe-prefill-quantum": the cause section's source
# excerpt, the prefill_cap section and Table 11)
# ---------------------------------------------------------------------------------------
def _golden_calls():
    seq, t11 = [], []
    for line in open(os.path.join(GOLDEN, "p1_prefill_calls.txt")):
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        if f[0] == "SEQ":
            seq.append((int(f[1]), int(f[2]), int(f[3]), int(f[4]), [int(v) for v in f[5:]]))
        elif f[0] == "T11":
            t11.append(tuple(int(v) for v in f[1:]))
    return seq, t11


def test_prefill_calls_reproduce_the_pages_sequences():
    seq, _ = _golden_calls()
    assert len(seq) == 2
    for start, q, cap, n, want in seq:
        got = [c for _, c in oracle.prefill_calls(start, n, q, True, cap)]
        assert got == want


def test_prefill_calls_reproduce_table_11():
    """Table 11 prints calls and mean chunk per boundary for an 8,478-token span at a context of
    about 82K.  Reading: the span starts at 81,920 (= 20 x 4096), the only start between 78,000
    and 86,000 that gives the printed call counts for all three boundaries."""
    _, t11 = _golden_calls()
    assert len(t11) == 3
    for n, cap, calls, mean in t11:
        c = oracle.prefill_calls(81920, n, 2048, True, cap)
        assert len(c) == calls and n // len(c) == mean
    hits = [s for s in range(78000, 86000)
            if all(len(oracle.prefill_calls(s, n, 2048, True, cap)) == calls for n, cap, calls, _ in t11)]
    assert hits == [81920]


def test_prefill_calls_ignore_the_quantum_when_nothing_generates():
    """Table 1's first row: without decoding load quantum 128 and 2048 run identically (the
    hard-coded 2048 piece)."""
    for start in (0, 1539, 81920):
        assert oracle.prefill_calls(start, 5964, 128, False) == oracle.prefill_calls(start, 5964, 2048, False)
        assert oracle.prefill_calls(start, 5964, 128, False) == oracle.prefill_calls(start, 5964, 2048, True)
    assert len(oracle.prefill_calls(0, 5964, 128, True)) == 47


@pytest.mark.parametrize("seed", range(6))
def test_prefill_calls_invariants(seed):
    rng = np.random.default_rng(seed)
    for _ in range(200):
        start = int(rng.integers(0, 300000))
        n = int(rng.integers(0, 40000))
        q = int(rng.choice([1, 7, 128, 512, 1000, 2048, 4096, 8192, 100000]))
        cap = int(rng.choice([1, 64, 2560, 3072, 4096, 8192]))
        active = bool(rng.integers(0, 2))
        piece = q if active else 2048
        calls = oracle.prefill_calls(start, n, q, active, cap)
        assert sum(c for _, c in calls) == n
        pos = start
        for p, c in calls:
            assert p == pos and 1 <= c <= min(piece, cap)
            assert (p % cap) + c <= cap  # never crosses a boundary
            pos += c
        # every piece edge (multiples of the piece from the prompt start) is a call edge
        edges = {p - start for p, _ in calls} | {n}
        assert all(e in edges for e in range(0, n, piece))
