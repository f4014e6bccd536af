"""Helpers shared by the tests: build plans from synthetic workloads, run the oracle on the
same arrays, and compare with the tolerances the layer is specified with."""
from __future__ import annotations

import numpy as np

import oracle
import synth

# End-to-end tolerance on the layer output: max |gpu - oracle| <= TOL * RMS(oracle), over the
# tokens whose fp64 router margin l_(k) - l_(k+1) is at least MARGIN_MIN.
TOL_BF16 = 2e-2
TOL_FP4 = 6e-2
MARGIN_MIN = 1e-3
# Router logits (fp32 accumulation of exact bf16 x fp32 products) against fp64.
TOL_LOGITS = 1e-5
# Gates: softmax of k <= 32 fp32 logits with expf (<= 2 ulp) and one division; relative.
TOL_GATES = 2e-6


def torch_mod():
    import torch
    return torch


def to_dev(a: np.ndarray, kind: str = "raw"):
    """numpy -> CUDA tensor.  kind='bf16' reinterprets uint16 bits as torch.bfloat16."""
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    if kind == "bf16":
        t = t.view(torch.bfloat16)
    return t


def bf16_tensor_to_f64(t) -> np.ndarray:
    torch = torch_mod()
    return oracle.bf16_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))


def make_plan(w: synth.Workload, path: str = "auto", T_max: int | None = None):
    from decode_batches_gb300 import MoePlan

    s = w.spec
    plan = MoePlan(s.E, s.k, s.d, s.f, s.n_shared, s.wdtype)
    ex = w.experts()
    b = w.router_bias()
    bt = to_dev(b) if b is not None else None
    if s.wdtype == "bf16":
        plan.set_weights(to_dev(w.router_weight()), bt, to_dev(ex.gate, "bf16"), to_dev(ex.up, "bf16"),
                         to_dev(ex.down, "bf16"))
    else:
        plan.set_weights(to_dev(w.router_weight()), bt, to_dev(ex.gate), to_dev(ex.up), to_dev(ex.down),
                         to_dev(ex.gate_scale), to_dev(ex.up_scale), to_dev(ex.down_scale))
    sh = w.shared()
    if sh is not None:
        plan.set_shared(s.f_s, to_dev(sh[0], "bf16"), to_dev(sh[1], "bf16"), to_dev(sh[2], "bf16"))
    plan.allocate_workspace(T_max or w.T)
    if path != "auto":
        plan.set_path(path)
    return plan


def decoded_experts(w: synth.Workload) -> oracle.DecodedExperts:
    ex = w.experts()
    return oracle.DecodedExperts(ex.gate, ex.up, ex.down, ex.gate_scale, ex.up_scale, ex.down_scale)


def oracle_layer(w: synth.Workload, rows=None) -> dict:
    """The oracle on all tokens, or on the token rows `rows` (the layer is per token)."""
    x = w.x() if rows is None else w.x()[rows]
    return oracle.moe_layer(x, w.router_weight(), w.router_bias(), w.spec.k, decoded_experts(w), w.shared())


def sample_rows(w: synth.Workload, n: int, seed: int = 1) -> np.ndarray:
    """A seeded sample of n token rows plus every decode row (rows >= n_prefill)."""
    if w.T <= n:
        return np.arange(w.T)
    rng = np.random.default_rng(seed)
    pre = np.sort(rng.choice(max(w.n_prefill, 1), size=min(n, max(w.n_prefill, 1)), replace=False))
    dec = np.arange(w.n_prefill, w.T)
    return np.unique(np.concatenate([pre, dec]))


def compare_layer(out_gpu: np.ndarray, ref: dict, k: int, tol: float, gpu_ids: np.ndarray | None = None):
    """Returns (max_err / rms, n_excluded).  Asserts routing agreement on included tokens."""
    margin = oracle.topk_margin(ref["logits"], k)
    keep = margin >= MARGIN_MIN
    if gpu_ids is not None:
        bad = np.where(keep & np.any(np.sort(gpu_ids, 1) != np.sort(ref["ids"], 1), axis=1))[0]
        assert bad.size == 0, f"routing differs from the oracle on tokens {bad[:10]} (margins {margin[bad[:10]]})"
    o = ref["out"]
    rms = float(np.sqrt(np.mean(o ** 2)))
    err = np.abs(out_gpu[keep] - o[keep]).max() if keep.any() else 0.0
    rel = float(err / rms)
    assert rel <= tol, f"max|gpu-oracle| = {err:.4g} = {rel:.4g} x RMS > {tol}"
    return rel, int((~keep).sum())
