"""GPU parity of the whole forward layer (moe_forward) against the oracle, plus
bitwise run-to-run determinism."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import TIE_TAU, TOL, check_routing, need_cuda, row_rel_err, to_np
from token_dispatch_expert_top_gb300 import synth

pytestmark = pytest.mark.gpu

LAYER_CASES = [
    (synth.WORKLOADS["tiny_f32"], None),
    (synth.Workload("mid_bf16", N=512, H=512, I=256, E=16, k=4, S=4, dtype="bf16"), None),
    (synth.Workload("mid_mxfp8", N=512, H=512, I=256, E=16, k=4, S=4, dtype="mxfp8"), None),
    (synth.Workload("mid_mxfp8_skew", N=768, H=1024, I=384, E=32, k=6, S=8, dtype="mxfp8",
                    skew=3.0), None),
    (synth.WORKLOADS["small_bf16"], None),      # every token
]


def check_layer(w, sample=None, fused=False, params=None, seed=0):
    need_cuda()
    from token_dispatch_expert_top_gb300.layer import MoeLayer
    inp = synth.make_inputs(w, device="cpu")
    layer = MoeLayer(w, inp, params=params)
    out = layer.forward(fused=fused)
    assert layer.device_status() == 0
    toks = None
    if sample is not None:
        toks = np.sort(np.random.default_rng(seed).choice(w.N, size=sample, replace=False))
    ref = O.forward(inp, w.E, w.k, w.S, w.dtype, tokens=toks)
    sel = ref["tokens"]
    assert check_routing(to_np(layer.idx), ref["idx"], ref["logits"], ref["gap"]) > 0.97
    ok = ref["gap"][sel] >= TIE_TAU
    err = row_rel_err(to_np(out)[sel][ok], ref["out"][ok])
    assert err.max() < TOL[w.dtype], (w.name, err.max())
    return layer, out


@pytest.mark.parametrize("w,sample", LAYER_CASES, ids=[c[0].name for c in LAYER_CASES])
def test_forward_matches_oracle(w, sample):
    check_layer(w, sample)


@pytest.mark.parametrize("w", [LAYER_CASES[1][0], LAYER_CASES[3][0]], ids=lambda w: w.name)
def test_forward_is_bitwise_deterministic(w):
    need_cuda()
    from token_dispatch_expert_top_gb300.layer import MoeLayer
    layer = MoeLayer(w, synth.make_inputs(w, device="cpu"))
    first = layer.forward().clone()
    for _ in range(3):
        assert torch.equal(layer.forward(), first)
    assert layer.device_status() == 0


def test_forward_empty_batch():
    need_cuda()
    from token_dispatch_expert_top_gb300 import moe as M
    w = synth.Workload("empty", N=0, H=256, I=128, E=4, k=2, S=1, dtype="bf16")
    shape = M.Shape.of(w)
    ws = torch.empty(max(M.moe_workspace_bytes(shape, None), 256), dtype=torch.uint8, device="cuda")
    M.moe_workspace_init(ws)
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    M.moe_forward(dummy, dummy, None, dummy, None, dummy, None, shape, None, dummy, None, None, ws)
    assert M.moe_last_device_status(ws) == 0


# Degenerate shapes: top-1 with a ragged token count, every token on every
# expert (k = E), a single expert (a dense SwiGLU FFN), a bias so steep that
# every token picks the same two experts (fourteen experts without slots), 512
# experts, k = 32, and the largest expert count the library takes (1024).
DEGENERATE = [
    synth.Workload("top1_ragged", N=300, H=512, I=256, E=16, k=1, S=3, dtype="mxfp8"),
    synth.Workload("k_eq_E", N=256, H=512, I=256, E=4, k=4, S=2, dtype="mxfp8"),
    synth.Workload("one_expert", N=200, H=256, I=128, E=1, k=1, S=2, dtype="bf16"),
    synth.Workload("two_hot", N=384, H=512, I=256, E=16, k=2, S=4, dtype="mxfp8", skew=50.0),
    # more experts than the tensor-core router takes (the SIMT router), and the largest k
    synth.Workload("many_experts", N=512, H=512, I=256, E=512, k=8, S=4, dtype="mxfp8"),
    synth.Workload("top32", N=256, H=512, I=256, E=64, k=32, S=2, dtype="mxfp8"),
    synth.Workload("max_experts", N=1024, H=256, I=128, E=1024, k=8, S=8, dtype="mxfp8"),
]


@pytest.mark.parametrize("w", DEGENERATE, ids=lambda w: w.name)
def test_forward_degenerate_shapes(w):
    layer, out = check_layer(w)
    if w.k == w.E:
        assert np.all(np.sort(to_np(layer.idx), axis=1) == np.arange(w.E))
    if w.skew >= 50.0:
        idx = to_np(layer.idx)
        assert len(np.unique(idx)) == w.k        # all tokens on the same k experts
    staged = out.clone()
    fused = layer.forward(fused=True)
    assert layer.device_status() == 0
    assert torch.equal(fused, staged)


@pytest.mark.parametrize("w,macro", [(LAYER_CASES[2][0], 2), (LAYER_CASES[2][0], 4), (LAYER_CASES[1][0], 2),
                                     (LAYER_CASES[3][0], 3)],
                         ids=["mid_mxfp8-2", "mid_mxfp8-4", "mid_bf16-2", "mid_mxfp8_skew-3"])
def test_macrobatched_forward_is_bitwise_equal(w, macro):
    """Macrobatches (each combine on the library's second stream, overlapping the next
    macrobatch's routing, layout and dispatch) give moe_forward's output bit for bit."""
    need_cuda()
    from token_dispatch_expert_top_gb300.layer import MoeLayer
    layer = MoeLayer(w, synth.make_inputs(w, device="cpu"))
    ref = layer.forward().clone()
    for _ in range(3):
        got = layer.forward_macrobatched(macro)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
    assert layer.device_status() == 0


@pytest.mark.parametrize("w,macro", [(LAYER_CASES[3][0], 3), (LAYER_CASES[2][0], 4)],
                         ids=["mid_mxfp8_skew-3", "mid_mxfp8-4"])
def test_macrobatched_forward_matches_oracle(w, macro):
    """The macrobatched forward against the oracle directly (every token)."""
    need_cuda()
    from token_dispatch_expert_top_gb300.layer import MoeLayer
    inp = synth.make_inputs(w, device="cpu")
    layer = MoeLayer(w, inp)
    out = layer.forward_macrobatched(macro)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    ref = O.forward(inp, w.E, w.k, w.S, w.dtype)
    ok = ref["gap"] >= TIE_TAU
    err = row_rel_err(to_np(out)[ok], ref["out"][ok])
    assert err.max() < TOL[w.dtype], (w.name, macro, err.max())


def test_macrobatched_forward_rejects_uneven_split():
    need_cuda()
    from token_dispatch_expert_top_gb300 import moe as M
    w = LAYER_CASES[2][0]          # N = 512, S = 4
    assert M.moe_macro_workspace_bytes(M.Shape.of(w), None, 3) == 0     # 512 % (3 * 4) != 0
    assert M.moe_macro_workspace_bytes(M.Shape.of(w), None, 4) > 0
