"""fp64 CPU oracle of the MoE expert layer -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import or run anything in this package.  The product path (the C-ABI library and its Python
binding) never imports it, and this package imports nothing from the product path: the two
share no code.  Both consume the arrays produced by the separate ``synth`` generator.

Every function is the plain definition of one step, written in float64 with numpy; matmul,
argsort and bincount are the only library primitives used.  Each step cites the passage of
the source pages it follows (pages are named by title; sections, tables and formulas by their
caption).

Parity status: every function here is pinned by tests in ``tests/test_oracle_pins.py``
(closed forms, brute force on tiny inputs, invariants and the pages' worked numbers).
"""
from .moe_ref import (  # noqa: F401
    bf16_to_f64,
    mxfp4_decode,
    e2m1_value,
    router_logits,
    select_topk,
    topk_gates,
    topk_margin,
    expert_histogram,
    exclusive_offsets,
    stable_permutation,
    swiglu_ffn,
    DecodedExperts,
    shared_ffn,
    combine,
    moe_layer,
    expected_unique_experts,
    tokens_per_expert,
    quantum_for_tokens_per_expert,
    prefill_piece_size,
    prefill_calls,
)
