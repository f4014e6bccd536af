"""GPU parity of the expert FFN, the combine and the whole layer against the fp64 oracle.

Small workloads are compared on every token; the large ones on a seeded sample of tokens plus
every decode row (exact for those tokens: the layer is per token).  Tokens whose fp64 router
margin is below 1e-3 are excluded from the output comparison and counted; routing must agree
with the oracle on every other token."""
import functools

import numpy as np
import pytest

import oracle
import synth
from moe_helpers import (TOL_BF16, TOL_FP4, bf16_tensor_to_f64, compare_layer, make_plan, oracle_layer,
                         sample_rows, to_dev)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

FULL = [("tiny", 0), ("decode", 0), ("mixed", 128), ("verify", 0)]
# every quantum of the mixed-step sweep goes through the whole layer against the oracle
SAMPLED = [("mixed", 512), ("mixed", 1024), ("mixed", 2048), ("mixed", 4096), ("mixed", 8192), ("fp4_zipf", 0)]


@functools.lru_cache(maxsize=None)
def workload(name, q):
    return synth.workload(name, quantum=q or 2048)


@functools.lru_cache(maxsize=None)
def plan_for(spec):
    T_max = {synth.TINY: 64, synth.QWEN_A3B_LIKE: 8195, synth.FP4_ZIPF: 2051}[spec]
    w = {synth.TINY: workload("tiny", 0), synth.QWEN_A3B_LIKE: workload("mixed", 8192),
         synth.FP4_ZIPF: workload("fp4_zipf", 0)}[spec]
    return make_plan(w, T_max=T_max)


@functools.lru_cache(maxsize=None)
def fused_plan_for(spec):
    """A plan whose steps of at most 8 tokens run the one-launch layer (MOE_SMALL_STEP=fused)."""
    import os
    old = os.environ.get("MOE_SMALL_STEP")
    os.environ["MOE_SMALL_STEP"] = "fused"
    try:
        T_max = {synth.TINY: 64, synth.QWEN_A3B_LIKE: 64}[spec]
        w = {synth.TINY: workload("tiny", 0), synth.QWEN_A3B_LIKE: workload("decode", 0)}[spec]
        return make_plan(w, T_max=T_max)
    finally:
        if old is None:
            del os.environ["MOE_SMALL_STEP"]
        else:
            os.environ["MOE_SMALL_STEP"] = old


def paths_for(spec):
    return ["simt", "tc"]


def _cases(lst):
    return [(n, q, p) for n, q in lst for p in paths_for(workload(n, q).spec)]


def _tol(w):
    return TOL_FP4 if w.spec.wdtype == "mxfp4" else TOL_BF16


@pytest.mark.parametrize("name,q,path", _cases(FULL))
def test_forward_full_vs_oracle(name, q, path):
    w = workload(name, q)
    plan = plan_for(w.spec)
    plan.set_path(path)
    assert plan.resolved_path()[0] == path
    x = to_dev(w.x(), "bf16")
    out = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    _, ids, _ = plan.route(x, want_logits=False)
    ref = oracle_layer(w)
    rel, excluded = compare_layer(out, ref, w.spec.k, _tol(w), ids.cpu().numpy())
    assert plan.device_error() == 0
    print(f"{name} q={q} {path}: max err {rel:.3e} x RMS, {excluded} tokens excluded")


@pytest.mark.parametrize("name,q,path", _cases(SAMPLED))
def test_forward_sampled_vs_oracle(name, q, path):
    w = workload(name, q)
    plan = plan_for(w.spec)
    plan.set_path(path)
    x = to_dev(w.x(), "bf16")
    out = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    _, ids, _ = plan.route(x, want_logits=False)
    rows = sample_rows(w, 96)
    ref = oracle_layer(w, rows)
    rel, excluded = compare_layer(out[rows], ref, w.spec.k, _tol(w), ids.cpu().numpy()[rows])
    assert plan.device_error() == 0
    print(f"{name} q={q} {path}: {len(rows)} rows, max err {rel:.3e} x RMS, {excluded} excluded")


@pytest.mark.parametrize("name,q,path", _cases([("tiny", 0), ("decode", 0), ("mixed", 512), ("verify", 0)]))
def test_experts_vs_oracle(name, q, path):
    """The grouped FFN alone, on the oracle's own grouping."""
    w = workload(name, q)
    plan = plan_for(w.spec)
    plan.set_path(path)
    ref = oracle_layer(w)
    y, ys = plan.experts(to_dev(w.x(), "bf16"), to_dev(ref["offsets"]), to_dev(ref["perm"]))
    yg = y.double().cpu().numpy()
    rms = np.sqrt(np.mean(ref["y_perm"] ** 2))
    assert np.abs(yg - ref["y_perm"]).max() <= _tol(w) * rms
    if ref["shared_y"] is not None:
        sg = ys.double().cpu().numpy()
        assert np.abs(sg - ref["shared_y"]).max() <= _tol(w) * np.sqrt(np.mean(ref["shared_y"] ** 2))


def _bf16_ulp(v):
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


@pytest.mark.parametrize("T,k,d,shared", [(1, 2, 256, False), (33, 8, 2048, True), (257, 8, 4096, True)])
def test_combine_vs_oracle(T, k, d, shared):
    from decode_batches_gb300 import MoePlan
    plan = MoePlan(16, k, d, 64, 0, "bf16")
    rng = np.random.default_rng(T)
    y = rng.normal(size=(T * k, d)).astype(np.float32)
    ys = rng.normal(size=(T, d)).astype(np.float32) if shared else None
    g = rng.random((T, k)).astype(np.float32)
    g /= g.sum(1, keepdims=True)
    inv = rng.permutation(T * k).astype(np.int32)
    out = plan.combine(to_dev(y), to_dev(g), to_dev(inv), to_dev(ys) if shared else None)
    y64 = y.astype(np.float64)
    ys64 = ys.astype(np.float64) if shared else None
    ref = oracle.combine(y64, g.astype(np.float64), inv, ys64)
    got = bf16_tensor_to_f64(out)
    # fp32 accumulation of k + 1 terms (relative rounding 2^-24 each on the running sum), then
    # one rounding to bf16: within one bf16 ulp of the exact sum plus the fp32 accumulation bound
    mag = oracle.combine(np.abs(y64), g.astype(np.float64), inv, np.abs(ys64) if shared else None)
    bound = _bf16_ulp(ref) + (k + 2) * 2.0 ** -24 * mag
    assert np.all(np.abs(got - ref) <= bound)


def test_forward_deterministic_and_prefill_independent():
    w = workload("mixed", 512)
    plan = plan_for(w.spec)
    plan.set_path("auto")
    x = to_dev(w.x(), "bf16")
    a = plan.forward(x, n_prefill=w.n_prefill).clone()
    b = plan.forward(x, n_prefill=0).clone()
    c = plan.forward(x, n_prefill=w.T).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_paths_agree():
    w = workload("mixed", 128)
    plan = plan_for(w.spec)
    x = to_dev(w.x(), "bf16")
    plan.set_path("simt")
    a = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    plan.set_path("tc")
    b = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    plan.set_path("auto")
    rms = np.sqrt(np.mean(a ** 2))
    # same arithmetic, different fp32 summation order: at most a couple of output ulps apart
    assert np.all(np.abs(a - b) <= 2 * _bf16_ulp(np.maximum(np.abs(a), np.abs(b))) + 1e-3 * rms)


@pytest.mark.parametrize("T", [1, 8, 9, 15, 16, 17, 64, 65, 255, 256, 257, 1000])
def test_forward_ragged_sizes(T):
    """T around the 16-column MMA step, the 32-token chunk, the 256-row segment limit and the
    routing front ends' switch points (one launch up to 8 tokens, tensor-core router above 16,
    one grouping block up to 64)."""
    w = synth.custom(synth.QWEN_A3B_LIKE, T, n_prefill=T // 2, name=f"ragged{T}")
    plan = plan_for(w.spec)
    plan.set_path("auto")
    x = to_dev(w.x(), "bf16")
    out = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    _, ids, _ = plan.route(x, want_logits=False)
    rows = sample_rows(w, 48)
    ref = oracle_layer(w, rows)
    compare_layer(out[rows], ref, w.spec.k, TOL_BF16, ids.cpu().numpy()[rows])
    assert plan.device_error() == 0


# odd tile counts everywhere (gate/up 3, down 3, shared gate/up 5): with T = 4000 the 16-bit
# kernels run two tiles per unit, and the last unit of each matrix holds one
ODD_TILES = synth.LayerSpec(E=8, k=2, d=384, f=192, n_shared=1, f_s=320, wdtype="bf16")


@pytest.mark.parametrize("T", [3, 4000])
def test_odd_tile_counts(T):
    w = synth.custom(ODD_TILES, T, n_prefill=T, name=f"oddtiles{T}")
    plan = make_plan(w)
    plan.set_path("tc")
    x = to_dev(w.x(), "bf16")
    out = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    _, ids, _ = plan.route(x, want_logits=False)
    rows = sample_rows(w, 64)
    ref = oracle_layer(w, rows)
    compare_layer(out[rows], ref, w.spec.k, TOL_BF16, ids.cpu().numpy()[rows])
    assert plan.device_error() == 0


def test_forward_edge_arguments_and_canaries():
    from decode_batches_gb300 import MoeError
    w = workload("tiny", 0)
    plan = plan_for(w.spec)
    x = to_dev(w.x(), "bf16")
    empty = torch.empty((0, w.spec.d), dtype=torch.bfloat16, device="cuda")
    plan.forward(empty)                                   # T = 0: no-op
    with pytest.raises(MoeError):
        plan.forward(x, n_prefill=w.T + 1)
    big = synth.custom(w.spec, 65).x()
    with pytest.raises(MoeError):
        plan.forward(to_dev(big, "bf16"))                 # T > T_max of the workspace
    # x 2 bytes past a 16-byte boundary: refused on the host, before any launch
    flat = torch.zeros(w.T * w.spec.d + 8, dtype=torch.bfloat16, device="cuda")
    x_mis = flat[1:1 + w.T * w.spec.d].view(w.T, w.spec.d)
    x_mis.copy_(x)
    assert x_mis.data_ptr() % 16 == 2
    with pytest.raises(MoeError):
        plan.forward(x_mis)
    # output written into the middle of a guarded buffer: guards untouched
    guard = 1024
    buf = torch.full((guard * 2 + w.T * w.spec.d,), 12345, dtype=torch.int16, device="cuda")
    out_view = buf[guard:guard + w.T * w.spec.d].view(torch.bfloat16).view(w.T, w.spec.d)
    plan.forward(x, out=out_view)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == 12345) and torch.all(buf[-guard:] == 12345)
    ref = oracle_layer(w)
    compare_layer(bf16_tensor_to_f64(out_view), ref, w.spec.k, TOL_BF16)


@pytest.mark.parametrize("T", [200, 400, 700])
def test_multi_part_experts_against_the_oracle(T):
    """Experts with ~100 rows (one segment, T = 200), ~200 rows (two parts, T = 400) and ~350
    rows (three parts, T = 700) on the tensor-core path, and several shared-expert segments;
    every output against the oracle, through the layer and through the experts entry point."""
    spec = synth.LayerSpec(E=4, k=2, d=256, f=512, n_shared=1, f_s=256, wdtype="bf16")
    w = synth.custom(spec, T, n_prefill=T - 3, name=f"parts{T}")
    plan = make_plan(w)
    plan.set_path("tc")
    x = to_dev(w.x(), "bf16")
    out = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    _, ids, _ = plan.route(x, want_logits=False)
    ref = oracle_layer(w)
    compare_layer(out, ref, spec.k, TOL_BF16, ids.cpu().numpy())
    # the experts entry point builds its own segments from the oracle's offsets
    y, _ = plan.experts(x, to_dev(ref["offsets"]), to_dev(ref["perm"]))
    rms = np.sqrt(np.mean(ref["y_perm"] ** 2))
    assert np.abs(y.double().cpu().numpy() - ref["y_perm"]).max() <= TOL_BF16 * rms
    assert plan.device_error() == 0


@pytest.mark.parametrize("E,k,T", [(16, 1, 37), (16, 1, 300), (8, 8, 300), (40, 3, 37), (40, 3, 300)])
def test_unusual_top_k_against_the_oracle(E, k, T):
    """k = 1 (no mixing), k = E (every expert, dense mixture) and E = 40 (not a multiple of 32 or
    of the router's 128-expert tile: the CUDA-core router) through the tensor-core layer, on the
    one-block routing front end (T = 37) and the general one (T = 300)."""
    spec = synth.LayerSpec(E=E, k=k, d=256, f=256, n_shared=1, f_s=128, wdtype="bf16")
    w = synth.custom(spec, T, n_prefill=T // 2, name=f"topk{E}_{k}_{T}")
    plan = make_plan(w)
    plan.set_path("tc")
    x = to_dev(w.x(), "bf16")
    out = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    _, ids, _ = plan.route(x, want_logits=False)
    compare_layer(out, oracle_layer(w), spec.k, TOL_BF16, ids.cpu().numpy())
    assert plan.device_error() == 0


def test_two_plans_on_two_streams():
    """Two plans (bf16 mixed step, 4-bit verify step) used at the same time on two streams: each
    has its own workspace and plan words (routing counter, unit hand-out words, error word), so
    the interleaved steps do not disturb each other; both results match their oracles."""
    wa, wb = workload("mixed", 512), workload("verify", 0)
    pa, pb = plan_for(wa.spec), plan_for(wb.spec)
    pa.set_path("auto")
    pb.set_path("auto")
    xa, xb = to_dev(wa.x(), "bf16"), to_dev(wb.x(), "bf16")
    oa = torch.empty((wa.T, wa.spec.d), dtype=torch.bfloat16, device="cuda")
    ob = torch.empty((wb.T, wb.spec.d), dtype=torch.bfloat16, device="cuda")
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(4):
        pa.forward(xa, n_prefill=wa.n_prefill, out=oa, stream=sa)
        pb.forward(xb, n_prefill=wb.n_prefill, out=ob, stream=sb)
    torch.cuda.synchronize()
    rows = sample_rows(wa, 48)
    _, ids_a, _ = pa.route(xa, want_logits=False)
    compare_layer(bf16_tensor_to_f64(oa)[rows], oracle_layer(wa, rows), wa.spec.k, TOL_BF16, ids_a.cpu().numpy()[rows])
    _, ids_b, _ = pb.route(xb, want_logits=False)
    compare_layer(bf16_tensor_to_f64(ob), oracle_layer(wb), wb.spec.k, TOL_FP4, ids_b.cpu().numpy())
    assert pa.device_error() == 0 and pb.device_error() == 0


def test_untiled_shape_runs_the_reference_path():
    """d and d_ff that the tensor-core tiles do not divide: the plan keeps the row-interleaved
    layout and the CUDA-core path computes the layer (with shared experts)."""
    spec = synth.LayerSpec(E=5, k=2, d=96, f=40, n_shared=2, f_s=24, wdtype="bf16")
    w = synth.custom(spec, 37, n_prefill=30, name="odd")
    plan = make_plan(w)
    from decode_batches_gb300 import MoeError
    with pytest.raises(MoeError):
        plan.set_path("tc")
    path, why = plan.resolved_path()
    assert path == "simt" and "tensor-core tiles" in why
    x = to_dev(w.x(), "bf16")
    out = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    _, ids, _ = plan.route(x, want_logits=False)
    compare_layer(out, oracle_layer(w), spec.k, TOL_BF16, ids.cpu().numpy())
    assert plan.device_error() == 0


FP4_SMALL = synth.LayerSpec(E=16, k=4, d=256, f=128, n_shared=1, f_s=128, wdtype="mxfp4")


@pytest.mark.parametrize("path", ["simt", "tc", "tc-mx"])
@pytest.mark.parametrize("T", [1, 77, 300])
def test_fp4_small_layer_both_paths(T, path, monkeypatch):
    """4-bit routed weights with a bf16 shared expert, every token: the CUDA-core path, the
    tensor-core path with the dequantising GEMMs and with the block-scaled ones (e2m1 weights x
    two e4m3 terms of x or h)."""
    if path == "tc-mx":
        monkeypatch.setenv("MOE_FP4_GATEUP", "mx")
        monkeypatch.setenv("MOE_FP4_DOWN", "mx")
        path = "tc"
    w = synth.custom(FP4_SMALL, T, n_prefill=T - 1, name=f"fp4small{T}")
    plan = make_plan(w)
    plan.set_path(path)
    x = to_dev(w.x(), "bf16")
    out = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    _, ids, _ = plan.route(x, want_logits=False)
    ref = oracle_layer(w)
    compare_layer(out, ref, FP4_SMALL.k, TOL_FP4, ids.cpu().numpy())
    y, ys = plan.experts(x, to_dev(ref["offsets"]), to_dev(ref["perm"]))
    rms = np.sqrt(np.mean(ref["y_perm"] ** 2))
    assert np.abs(y.double().cpu().numpy() - ref["y_perm"]).max() <= TOL_FP4 * rms
    assert plan.device_error() == 0


# d_ff / 64 odd: the down GEMM's last 128-deep K stage holds a single 64-wide block; a hot
# expert (Zipf routing) spans several 128-row segments
FP4_ODD = synth.LayerSpec(E=12, k=3, d=384, f=192, n_shared=0, f_s=0, wdtype="mxfp4", zipf_s=1.2)


@pytest.mark.parametrize("variant", ["mx", "dequant"])
@pytest.mark.parametrize("T", [5, 390])
def test_fp4_odd_k_blocks_tc(T, variant, monkeypatch):
    """d_ff / 64 odd: the down projection's last 128-deep stage holds one 64-wide block (the
    block-scaled kernels issue two MMAs there, the dequantising ones one slice)."""
    if variant == "mx":
        monkeypatch.setenv("MOE_FP4_GATEUP", "mx")
        monkeypatch.setenv("MOE_FP4_DOWN", "mx")
    w = synth.custom(FP4_ODD, T, n_prefill=T, name=f"fp4odd{T}")
    plan = make_plan(w)
    plan.set_path("tc")
    x = to_dev(w.x(), "bf16")
    out = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    _, ids, _ = plan.route(x, want_logits=False)
    ref = oracle_layer(w)
    compare_layer(out, ref, FP4_ODD.k, TOL_FP4, ids.cpu().numpy())
    assert plan.device_error() == 0


def test_fp4_scales_outside_fp16_range_use_the_reference_path():
    """A scale whose e2m1 multiples are not exact in fp16 keeps the tensor-core path off; the
    CUDA-core path reads the same tiled layout and still matches the oracle."""
    from decode_batches_gb300 import MoeError, MoePlan
    w = synth.custom(FP4_SMALL, 40, n_prefill=40, name="fp4oor")
    ex = w.experts()
    gs = ex.gate_scale.copy()
    gs[3, 5, 2] = 100            # 2^-27: below the fp16-exact range
    ex.gate_scale = gs
    s = w.spec
    plan = MoePlan(s.E, s.k, s.d, s.f, s.n_shared, s.wdtype)
    plan.set_weights(to_dev(w.router_weight()), None, to_dev(ex.gate), to_dev(ex.up), to_dev(ex.down),
                     to_dev(gs), to_dev(ex.up_scale), to_dev(ex.down_scale))
    sh = w.shared()
    plan.set_shared(s.f_s, to_dev(sh[0], "bf16"), to_dev(sh[1], "bf16"), to_dev(sh[2], "bf16"))
    plan.allocate_workspace(w.T)
    with pytest.raises(MoeError):
        plan.set_path("tc")
    path, why = plan.resolved_path()
    assert path == "simt" and "scale byte" in why
    x = to_dev(w.x(), "bf16")
    out = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    ref = oracle.moe_layer(w.x(), w.router_weight(), None, s.k,
                           oracle.DecodedExperts(ex.gate, ex.up, ex.down, gs, ex.up_scale, ex.down_scale), sh)
    compare_layer(out, ref, s.k, TOL_FP4)


def test_composed_prefill_calls_vs_oracle():
    """A prompt prefilled through the step composer: each composed call (its prompt rows plus two
    decode rows) goes through moe_layer_forward with its own T, and every row matches the oracle
    (the layer is per token, so the calls reassemble the whole prompt's output)."""
    from decode_batches_gb300 import compose_prefill
    n_prompt, n_dec = 700, 2
    w = synth.custom(synth.TINY, n_prompt + n_dec, n_prefill=n_prompt, name="composed")
    plan = make_plan(w, T_max=300)
    plan.set_path("tc")
    xs = w.x()
    calls = compose_prefill(1539, n_prompt, 128, True, prefill_cap=256)
    assert sum(c for _, c, _ in calls) == n_prompt and max(c for _, c, _ in calls) <= 128
    ref = oracle_layer(w)
    got = np.zeros_like(ref["out"])
    done = 0
    for _, c, _ in calls:
        rows = np.concatenate([np.arange(done, done + c), np.arange(n_prompt, n_prompt + n_dec)])
        out = bf16_tensor_to_f64(plan.forward(to_dev(xs[rows], "bf16"), n_prefill=c))
        got[done:done + c] = out[:c]
        got[n_prompt:] = out[c:]
        done += c
    compare_layer(got, ref, synth.TINY.k, TOL_BF16)
    assert plan.device_error() == 0


@pytest.mark.parametrize("T", [8, 9, 16, 17, 64, 65])
def test_fp4_front_end_switch_points(T):
    """The 384-expert 4-bit layer at the T where the routing front end, the 64-row geometry and
    the fused fp16 conversion of x switch; every token against the oracle."""
    base = workload("fp4_zipf", 0)
    w = synth.custom(base.spec, T, n_prefill=T // 2, name=f"fp4switch{T}")
    plan = plan_for(base.spec)
    plan.set_path("tc")
    x = to_dev(w.x(), "bf16")
    out = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    _, ids, _ = plan.route(x, want_logits=False)
    compare_layer(out, oracle_layer(w), base.spec.k, TOL_FP4, ids.cpu().numpy())
    assert plan.device_error() == 0


@pytest.mark.parametrize("spec_name,T", [("decode", 1), ("decode", 2), ("decode", 4), ("decode", 7), ("decode", 8),
                                         ("tiny", 1), ("tiny", 5), ("tiny", 8)])
def test_small_step_one_launch_vs_oracle(spec_name, T):
    """Steps of at most 8 tokens on bf16 weights run the whole layer in one launch (router, top-k,
    grouping, weight-streaming gate/up + SwiGLU and down, combine).  Every token against the
    oracle, the same answer twice (bit for bit), and close to the tensor-core path's."""
    spec = workload(spec_name, 0).spec
    w = synth.custom(spec, T, n_prefill=T // 2, name=f"small{spec_name}{T}")
    plan = fused_plan_for(spec)
    plan.set_path("auto")
    x = to_dev(w.x(), "bf16")
    a = plan.forward(x, n_prefill=w.n_prefill).clone()
    assert plan.last_launch_count() == 1
    b = plan.forward(x, n_prefill=w.n_prefill).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    _, ids, _ = plan.route(x, want_logits=False)
    got = bf16_tensor_to_f64(a)
    compare_layer(got, oracle_layer(w), spec.k, TOL_BF16, ids.cpu().numpy())
    plan.set_path("tc")
    c = bf16_tensor_to_f64(plan.forward(x, n_prefill=w.n_prefill))
    plan.set_path("auto")
    rms = np.sqrt(np.mean(got ** 2))
    # same arithmetic except that the tensor-core path rounds y to fp16 (relative 2^-11) and sums
    # in another order: at most a couple of output ulps apart
    assert np.all(np.abs(got - c) <= 2 * _bf16_ulp(np.maximum(np.abs(got), np.abs(c))) + 4e-3 * rms)
    assert plan.device_error() == 0
