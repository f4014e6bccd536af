"""moe_layer_forward captured in a CUDA graph: replays give the eager call's bits.

The 4-bit layer with a narrow shared expert runs the shared gate/up on the plan's second stream
(forked from and joined into the caller's stream), so its capture holds a fork and a join; the
16-bit layer is one stream.  Each replay gets a new input copied into the captured buffer."""
import numpy as np
import pytest

import synth
from moe_helpers import make_plan, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

FP4_FORK = synth.LayerSpec(E=16, k=4, d=256, f=128, n_shared=1, f_s=128, wdtype="mxfp4")


def _inputs(spec, T, n, seed):
    return [to_dev(synth.custom(spec, T, n_prefill=T, name=f"graph{seed}_{i}", seed=seed + i).x(), "bf16")
            for i in range(n)]


@pytest.mark.parametrize("which,T", [("bf16", 5), ("bf16", 300), ("fp4", 7), ("fp4", 300)])
def test_graph_replay_matches_eager(which, T):
    spec = synth.TINY if which == "bf16" else FP4_FORK
    w = synth.custom(spec, T, n_prefill=T, name=f"graph_{which}{T}")
    plan = make_plan(w, path="tc")
    xs = _inputs(spec, T, 3, 11)
    eager = [plan.forward(x, n_prefill=T).clone() for x in xs]
    torch.cuda.synchronize()

    x_static = xs[0].clone()
    out_static = torch.empty_like(x_static)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # one call outside the capture on the capturing stream
        plan.forward(x_static, n_prefill=T, out=out_static)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.forward(x_static, n_prefill=T, out=out_static)
    for x, ref in zip(xs, eager):
        x_static.copy_(x)
        out_static.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_static.view(torch.int16), ref.view(torch.int16))
    assert plan.device_error() == 0


def test_forked_shared_expert_sees_its_own_step():
    """Alternating inputs through the forked order: a shared down projection that read the
    previous step's h_s (a missing join) would make the results differ between repeats."""
    T = 9
    plan = make_plan(synth.custom(FP4_FORK, T, n_prefill=T, name="fork9"), path="tc")
    xs = _inputs(FP4_FORK, T, 2, 23)
    first = [plan.forward(x, n_prefill=T).clone() for x in xs]
    assert not torch.equal(first[0], first[1])
    for i in range(12):
        out = plan.forward(xs[i % 2], n_prefill=T)
        assert torch.equal(out.view(torch.int16), first[i % 2].view(torch.int16))
    assert np.isfinite(first[0].float().cpu().numpy()).all()
    assert plan.device_error() == 0
