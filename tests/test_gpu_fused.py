"""The persistent fused forward (moe_forward_fused): bitwise equal to the staged
forward for every ring size, minibatch and SM split (so it inherits the staged
path's parity with the oracle), no dropped tokens with rings far smaller than the
batch, and bounded waits that report MOE_ERR_TIMEOUT instead of hanging."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import TIE_TAU, TOL, need_cuda, row_rel_err, to_np
from token_dispatch_expert_top_gb300 import synth

pytestmark = pytest.mark.gpu

MID_MX = synth.Workload("mid_mxfp8", N=512, H=512, I=256, E=16, k=4, S=4, dtype="mxfp8")
MID_BF16 = synth.Workload("mid_bf16", N=512, H=512, I=256, E=16, k=4, S=4, dtype="bf16")
SKEW_MX = synth.Workload("skew_mxfp8", N=768, H=1024, I=512, E=32, k=6, S=8, dtype="mxfp8",
                         skew=3.0)


def _layers(w, params_list):
    need_cuda()
    from token_dispatch_expert_top_gb300 import moe as M
    from token_dispatch_expert_top_gb300.layer import MoeLayer
    inp = synth.make_inputs(w, device="cpu")
    return M, MoeLayer, inp


def _params(M, ring=0, mb=0, g=0, c=0, timeout_ns=0, skip=0, reverse=0):
    return M.Params(ring, mb, g, c, timeout_ns, skip, reverse)


@pytest.mark.parametrize("w", [MID_MX, MID_BF16, SKEW_MX], ids=lambda w: w.name)
def test_fused_equals_staged_default_params(w):
    M, MoeLayer, inp = _layers(w, None)
    layer = MoeLayer(w, inp)
    staged = layer.forward().clone()
    idx_staged = layer.idx.clone()
    fused = layer.forward(fused=True)
    assert layer.device_status() == 0
    assert torch.equal(layer.idx, idx_staged)
    assert torch.equal(fused, staged)


@pytest.mark.parametrize("ring,mb,g", [(64, 32, 1), (256, 128, 4), (1024, 512, 16), (96, 32, 2),
                                       (3072, 0, 0), (64, 64, 3)])
def test_fused_ring_and_split_sweep_bitwise(ring, mb, g):
    w = SKEW_MX
    M, MoeLayer, inp = _layers(w, None)
    p = _params(M, ring=ring, mb=mb, g=g)
    layer = MoeLayer(w, inp, params=p)
    staged = layer.forward().clone()
    fused = layer.forward(fused=True)
    assert layer.device_status() == 0
    assert torch.equal(fused, staged), (ring, mb, g)


def test_fused_matches_oracle_small_ring():
    w = MID_MX
    M, MoeLayer, inp = _layers(w, None)
    layer = MoeLayer(w, inp, params=_params(M, ring=128, mb=64, g=2))
    out = to_np(layer.forward(fused=True))
    assert layer.device_status() == 0
    ref = O.forward(inp, w.E, w.k, w.S, w.dtype)
    ok = ref["gap"] >= TIE_TAU
    assert row_rel_err(out[ok], ref["out"][ok]).max() < TOL[w.dtype]


def test_fused_is_bitwise_deterministic():
    w = SKEW_MX
    M, MoeLayer, inp = _layers(w, None)
    layer = MoeLayer(w, inp, params=_params(M, ring=256, mb=128, g=4))
    first = layer.forward(fused=True).clone()
    for _ in range(3):
        assert torch.equal(layer.forward(fused=True), first)
    assert layer.device_status() == 0


def test_fused_wait_runs_out_and_reports_timeout():
    """The gather role never publishes minibatch 1 (a counter nothing sets): every
    wait gives up after timeout_ns, the call reports MOE_ERR_TIMEOUT, and the
    context stays usable for the next call."""
    w = MID_MX
    M, MoeLayer, inp = _layers(w, None)
    p_bad = _params(M, ring=256, mb=128, g=2, timeout_ns=200_000_000, skip=2)
    layer = MoeLayer(w, inp, params=p_bad)
    layer.forward(fused=True)
    assert layer.device_status() == M.MOE_ERR_TIMEOUT
    # the same workspace and context still work
    good = _params(M, ring=256, mb=128, g=2)
    out = layer.forward(fused=True, params=good).clone()
    assert layer.device_status() == 0
    assert torch.equal(out, layer.forward())


def test_fused_rejects_bad_ring():
    w = MID_MX
    M, MoeLayer, inp = _layers(w, None)
    layer = MoeLayer(w, inp)
    with pytest.raises(M.MoeError):
        layer.forward(fused=True, params=_params(M, ring=100, mb=64))     # ring not a multiple
    with pytest.raises(M.MoeError):
        layer.forward(fused=True, params=_params(M, g=100000))            # more CTAs than fit


@pytest.mark.parametrize("w,ring,mb,g", [(SKEW_MX, 0, 0, 0), (SKEW_MX, 256, 128, 4), (SKEW_MX, 1024, 512, 16),
                                         (SKEW_MX, 96, 32, 2), (MID_MX, 0, 0, 0), (MID_BF16, 128, 64, 2)],
                         ids=["skew-default", "skew-256", "skew-1024", "skew-96", "mid-default", "bf16-128"])
def test_fused_reverse_ring_traversal_bitwise(w, ring, mb, g):
    """Minibatches cut from the last slot down (reverse ring traversal) give the
    same output bit for bit."""
    M, MoeLayer, inp = _layers(w, None)
    layer = MoeLayer(w, inp, params=_params(M, ring=ring, mb=mb, g=g))
    staged = layer.forward().clone()
    fused = layer.forward(fused=True, params=_params(M, ring=ring, mb=mb, g=g, reverse=1))
    assert layer.device_status() == 0
    assert torch.equal(fused, staged), (ring, mb, g)


@pytest.mark.parametrize("ring,mb,g", [(256, 128, 4), (0, 0, 0)], ids=["ring256", "default"])
def test_fused_reverse_ring_matches_oracle(ring, mb, g):
    """Reverse ring traversal against the oracle directly (every token)."""
    w = SKEW_MX
    M, MoeLayer, inp = _layers(w, None)
    layer = MoeLayer(w, inp, params=_params(M, ring=ring, mb=mb, g=g))
    out = to_np(layer.forward(fused=True, params=_params(M, ring=ring, mb=mb, g=g, reverse=1)))
    assert layer.device_status() == 0
    ref = O.forward(inp, w.E, w.k, w.S, w.dtype)
    ok = ref["gap"] >= TIE_TAU
    assert row_rel_err(out[ok], ref["out"][ok]).max() < TOL[w.dtype]


@pytest.mark.parametrize("H", [256, 768], ids=["H256", "H768"])
def test_fused_first_call_scale_rows_not_16_byte_multiples(H):
    """MXFP8 scale rows of H/32 = 8 or 24 bytes: the fused kernel's own gather must
    copy them whole.  The fused forward runs first on a fresh workspace, so no
    earlier call has filled the ring, and is checked against the oracle, then
    against the staged forward bit for bit."""
    w = synth.Workload(f"fused_h{H}", N=256, H=H, I=256, E=16, k=4, S=4, dtype="mxfp8")
    M, MoeLayer, inp = _layers(w, None)
    layer = MoeLayer(w, inp)
    fused = layer.forward(fused=True).clone()
    assert layer.device_status() == 0
    ref = O.forward(inp, w.E, w.k, w.S, w.dtype)
    ok = ref["gap"] >= TIE_TAU
    assert row_rel_err(to_np(fused)[ok], ref["out"][ok]).max() < TOL[w.dtype]
    assert torch.equal(layer.forward(), fused)
