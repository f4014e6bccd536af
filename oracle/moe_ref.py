"""Plain fp64 definition of one MoE expert layer on a serving step's token batch.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Nothing here is tuned.

Sources (pages, by title):
  [P1] "moe-prefill-quantum" (DeepSeek V4 Flash on ds4-server, M3 Ultra): the section on the
       cause (the model is MoE), the expected-unique-experts formula, Figure 5 and Table 9
       (tokens per expert = Q*k/E), and the quantum inversion Q = target*E/k.
  [P2] "DeepSeek V4.1F Q4 with native DSpark MTP on M3 Ultra": the Decode paragraph (a
       384-expert router computed in one dispatch; a shared expert whose gate+up+SwiGLU is
       always run; bf16 rounding inside producer kernels) and the DSpark paragraph (6 verify
       rows share one weight stream).
  [P4] "Why SSD-streamed MoE was slow: 8GB Jetson Orin Nano, part 2": the section re-checking
       part 1 (expert FFN executes gate -> up -> down as SwiGLU(gate, up)), the experiment
       table (256 experts, 8 used per token), the `mul_mat_id` grouped expert matmul in the
       first-cache section, and the section on generated text changing between runs (every
       selected expert must be computed exactly once).

Readings where the pages are silent (each is the plainest one the rest supports):
  * top-k order: a total order on (value, index) -- larger value first, lower index first on
    equal values; +0 == -0; NaN ranks below -inf, NaNs ordered by index.
  * gates: softmax over the k selected logits ("normalised top-k"), identical to a softmax
    over all experts renormalised on the selected set.
  * the shared expert is added with weight 1; several shared experts are summed.
  * the grouping order is a stable counting sort of the assignments a = t*k + j by expert.
  * 4-bit weights: OCP MX v1.0 e2m1 elements with an e8m0 scale per 32 consecutive K
    elements, the even element in the low nibble.
"""
from __future__ import annotations

import math
from typing import Callable, Optional, Sequence

import numpy as np


# ---------------------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns: bf16 is the top half of an IEEE binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def e2m1_value(code: int) -> float:
    """OCP MX v1.0 FP4 (E2M1) element: sign bit 3, 2 exponent bits (bias 1), 1 mantissa bit.

    Magnitudes of codes 0..7 are 0, 0.5, 1, 1.5, 2, 3, 4, 6 (code 1 is the subnormal 0.5)."""
    table = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
    mag = table[code & 7]
    return -mag if (code & 8) else mag


_E2M1 = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def mxfp4_decode(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Decode block-scaled 4-bit weights to fp64.

    codes  uint8 [..., K/2]: element 2i in the low nibble, 2i+1 in the high nibble.
    scales uint8 [..., K/32]: e8m0, value 2^(s-127) (s = 255 is NaN and never produced).
    Returns fp64 [..., K] with value = e2m1(code) * 2^(s - 127)   (OCP MX v1.0).
    [P1] hardware check (MXFP4 unpack, multiply by scale, accumulate); [P4] TL;DR (MXFP4 model).
    """
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    lo = _E2M1[codes & 0x0F]
    hi = _E2M1[codes >> 4]
    vals = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
    s = np.where(scales == 255, np.nan, np.ldexp(1.0, scales.astype(np.int64) - 127))
    return vals * np.repeat(s, 32, axis=-1)


# ---------------------------------------------------------------------------------------
# Router: logits, top-k, gates            [P2] Decode paragraph (router + top-k in one pass)
# ---------------------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_router: np.ndarray, b_router: Optional[np.ndarray]) -> np.ndarray:
    """l[t, e] = sum_i x[t, i] * W_r[e, i] + b[e], in fp64.

    x fp64 [T][d]; W_r fp64 [E][d]; b fp64 [E] or None."""
    logits = x @ w_router.T
    if b_router is not None:
        logits = logits + b_router[None, :]
    return logits


def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    """S_t = the k first experts of row t under the total order (value desc, index asc).

    Works on fp32 or fp64 logits (the comparison is exact either way).  Slot 0 holds the
    largest logit.  A stable sort of the negated values keeps equal values in index order;
    numpy places NaN last (below -inf) and treats -0 and +0 as equal.
    [P1] cause section: DeepSeek V4 Flash picks 6 of its 256 experts for each token;
    [P4] experiment table: 8 of 256 experts per token."""
    logits = np.asarray(logits)
    order = np.argsort(-logits, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def topk_gates(logits: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """g[t, j] = exp(l[t, S_j] - l[t, S_0]) / sum_j' exp(l[t, S_j'] - l[t, S_0]), fp64."""
    sel = np.take_along_axis(np.asarray(logits, dtype=np.float64), ids.astype(np.int64), axis=1)
    ex = np.exp(sel - sel[:, :1])
    return ex / ex.sum(axis=1, keepdims=True)


def topk_margin(logits: np.ndarray, k: int) -> np.ndarray:
    """l_(k) - l_(k+1): gap between the k-th and (k+1)-th largest logit of each row (inf if k = E)."""
    logits = np.asarray(logits, dtype=np.float64)
    if k >= logits.shape[1]:
        return np.full(logits.shape[0], np.inf)
    srt = -np.sort(-logits, axis=1)
    return srt[:, k - 1] - srt[:, k]


# ---------------------------------------------------------------------------------------
# Grouping: histogram, exclusive scan, stable permutation   ([P4] `mul_mat_id`, and the
# section on generated text changing between runs: every selected expert computed once)
# ---------------------------------------------------------------------------------------

def expert_histogram(ids: np.ndarray, E: int) -> np.ndarray:
    """counts[e] = #{(t, j) : ids[t, j] = e}."""
    return np.bincount(np.asarray(ids).ravel().astype(np.int64), minlength=E).astype(np.int32)


def exclusive_offsets(counts: np.ndarray) -> np.ndarray:
    """off[e] = sum_{e' < e} counts[e'];  off[E] = total."""
    return np.concatenate([[0], np.cumsum(counts, dtype=np.int64)]).astype(np.int32)


def stable_permutation(ids: np.ndarray):
    """Stable counting sort of the assignments a = t*k + j by expert id.

    perm[r] = a (the r-th row of the grouped problem), inv[a] = r.  Inside one expert's
    segment rows ascend by assignment index, hence by token."""
    flat = np.asarray(ids).ravel().astype(np.int64)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int32)
    return perm, inv


# ---------------------------------------------------------------------------------------
# Expert FFN: SwiGLU(gate, up) then down        [P4] gate -> up -> down, SwiGLU(gate, up)
# ---------------------------------------------------------------------------------------

def swiglu_ffn(x_rows: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """y = W_d (silu(W_g x) * (W_u x)) for each row of x, silu(z) = z / (1 + e^-z).

    x_rows fp64 [n][d]; w_gate, w_up fp64 [f][d]; w_down fp64 [d][f]; returns fp64 [n][d].
    The hidden vector h is kept in fp64 (no intermediate rounding)."""
    u = x_rows @ w_gate.T
    v = x_rows @ w_up.T
    with np.errstate(over="ignore"):
        h = u / (1.0 + np.exp(-u)) * v
    return h @ w_down.T


class DecodedExperts:
    """Per-expert fp64 weights, decoded on demand from the stored format.

    Stored as bf16 bits ([E][f][d] gate/up, [E][d][f] down) or 4-bit codes + e8m0 scales."""

    def __init__(self, gate, up, down, gate_scale=None, up_scale=None, down_scale=None):
        self.gate, self.up, self.down = gate, up, down
        self.gate_scale, self.up_scale, self.down_scale = gate_scale, up_scale, down_scale
        self.fp4 = gate_scale is not None
        self.E = gate.shape[0]

    def expert(self, e: int):
        if self.fp4:
            return (mxfp4_decode(self.gate[e], self.gate_scale[e]),
                    mxfp4_decode(self.up[e], self.up_scale[e]),
                    mxfp4_decode(self.down[e], self.down_scale[e]))
        return bf16_to_f64(self.gate[e]), bf16_to_f64(self.up[e]), bf16_to_f64(self.down[e])


def shared_ffn(x: np.ndarray, shared) -> np.ndarray:
    """Sum over the always-on shared experts (weight 1 each) of SwiGLU FFN(x).

    shared = (gate [n_s][f_s][d], up [n_s][f_s][d], down [n_s][d][f_s]) bf16 bits, or None.
    [P2] Decode paragraph: the shared expert's gate+up+SwiGLU runs for every token."""
    out = np.zeros_like(x)
    if shared is None:
        return out
    g, u, dn = shared
    for s in range(g.shape[0]):
        out += swiglu_ffn(x, bf16_to_f64(g[s]), bf16_to_f64(u[s]), bf16_to_f64(dn[s]))
    return out


# ---------------------------------------------------------------------------------------
# Combine
# ---------------------------------------------------------------------------------------

def combine(y_perm: np.ndarray, gates: np.ndarray, inv: np.ndarray, shared_y: Optional[np.ndarray]) -> np.ndarray:
    """out[t] = sum_{j=0..k-1} g[t, j] * y[inv[t*k + j]]  (+ shared_y[t]), in fp64, j ascending."""
    T, k = gates.shape
    out = np.zeros((T, y_perm.shape[1]), dtype=np.float64)
    for j in range(k):
        out += gates[:, j:j + 1] * y_perm[inv[np.arange(T) * k + j]]
    if shared_y is not None:
        out += shared_y
    return out


# ---------------------------------------------------------------------------------------
# The whole layer
# ---------------------------------------------------------------------------------------

def moe_layer(x_bits: np.ndarray, w_router: np.ndarray, b_router: Optional[np.ndarray], k: int,
              experts: DecodedExperts, shared=None, logits_override: Optional[np.ndarray] = None,
              n_prefill: int = 0) -> dict:
    """One MoE layer on T tokens, all in fp64.

    x_bits bf16 bits [T][d]; w_router fp32 [E][d]; b_router fp32 [E] or None.
    ``logits_override`` (e.g. fp32 logits taken from another implementation) replaces the
    computed logits for selection and gates; the returned 'logits' are always the fp64 ones.
    ``n_prefill`` marks the first rows as prefill; the layer is per token, so it is unused
    (it exists so tests can show the output does not depend on it).
    Returns a dict with logits, ids, gates, counts, offsets, perm, inv, y_perm, shared_y, out.
    """
    del n_prefill
    x = bf16_to_f64(x_bits)
    T = x.shape[0]
    E = w_router.shape[0]
    wr = np.asarray(w_router, dtype=np.float64)
    br = None if b_router is None else np.asarray(b_router, dtype=np.float64)
    logits = router_logits(x, wr, br)
    sel_logits = logits if logits_override is None else logits_override
    ids = select_topk(sel_logits, k)
    gates = topk_gates(sel_logits, ids)
    counts = expert_histogram(ids, E)
    offsets = exclusive_offsets(counts)
    perm, inv = stable_permutation(ids)
    y_perm = np.zeros((T * k, x.shape[1]), dtype=np.float64)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 == r0:
            continue
        tok = perm[r0:r1] // k
        wg, wu, wd = experts.expert(e)
        y_perm[r0:r1] = swiglu_ffn(x[tok], wg, wu, wd)
    shared_y = shared_ffn(x, shared) if shared is not None else None
    out = combine(y_perm, gates, inv, shared_y)
    return dict(logits=logits, ids=ids, gates=gates, counts=counts, offsets=offsets, perm=perm,
                inv=inv, y_perm=y_perm, shared_y=shared_y, out=out)


# ---------------------------------------------------------------------------------------
# Chunk arithmetic from [P1] (used for workload design and checked against Table 9)
# ---------------------------------------------------------------------------------------

def expected_unique_experts(E: int, k: int, Q: int) -> float:
    """[P1] expected distinct experts woken by a Q-token chunk: E * (1 - (1 - k/E)^Q)."""
    return E * (1.0 - (1.0 - k / E) ** Q)


def tokens_per_expert(Q: int, k: int, E: int) -> float:
    """[P1] Table 9: tokens per expert = Q * k / E."""
    return Q * k / E


def quantum_for_tokens_per_expert(target: float, E: int, k: int) -> float:
    """[P1] the inversion: quantum = target * E / k."""
    return target * E / k


# ---------------------------------------------------------------------------------------
# Prefill chunking of the serving loop from [P1] (the step composer's definition)
# ---------------------------------------------------------------------------------------

def prefill_piece_size(quantum: int, generation_active: bool) -> int:
    """[P1] the cause section's source excerpt: the server's prefill piece is the configured
    quantum only while some request is generating tokens; otherwise it is a fixed 2048."""
    return quantum if generation_active else 2048


def prefill_calls(start_pos: int, n_tokens: int, quantum: int, generation_active: bool,
                  prefill_cap: int = 4096) -> list:
    """[P1] the GPU calls that prefill ``n_tokens`` prompt tokens starting at context position
    ``start_pos``, as (pos, n) pairs in order.

    Two levels, as the page describes them:
      * the server hands the prompt over in pieces of ``prefill_piece_size`` tokens, counted
        from the start of the prompt;
      * the engine cuts each piece at the multiples of ``prefill_cap`` in absolute position (the
        section on ``prefill_cap`` boundaries and its code excerpt): a call starting at ``pos``
        with ``pos % prefill_cap != 0`` ends at the next multiple at the latest.
    Reading where the excerpt is silent: a call also never exceeds ``prefill_cap`` tokens (the
    engine's batch buffer is sized by it), so a piece larger than ``prefill_cap`` is cut at the
    boundaries too.  With a prompt starting at 1539 modulo 4096 and pieces of 2048 this gives
    the page's repeating 2048, 509, 1539."""
    if n_tokens < 0 or quantum < 1 or prefill_cap < 1 or start_pos < 0:
        raise ValueError("bad arguments")
    piece = prefill_piece_size(quantum, generation_active)
    calls = []
    pos, left = start_pos, n_tokens
    while left > 0:
        rem = min(piece, left)
        while rem > 0:
            n = min(rem, prefill_cap)
            mod = pos % prefill_cap
            if mod != 0:
                n = min(n, prefill_cap - mod)
            calls.append((pos, n))
            pos += n
            rem -= n
            left -= n
    return calls
