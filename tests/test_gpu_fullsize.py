"""Full-size parity for the DeepSeek-V3-shaped layers (N=8192 or 16384, H=7168,
I=2048, E=256, top-8, MXFP8): routing of every token and the outputs of a seeded
sample of 1024 tokens against the oracle, every slot row of the hottest expert in
the skewed layers, and the persistent fused forward equal to the staged one bit for
bit -- with the default ring and with rings of 64, 256 and 1024 slots."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import TIE_TAU, TOL, check_routing, need_cuda, row_rel_err, to_np
from token_dispatch_expert_top_gb300 import synth

pytestmark = pytest.mark.gpu


def _setup(name, params=None):
    need_cuda()
    from token_dispatch_expert_top_gb300.layer import MoeLayer
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w)            # drawn on the device
    layer = MoeLayer(w, inp, params=params)
    return w, inp, layer


def _oracle_weights(inp, dtype):
    return lambda e: O.expert_operands(inp["w_gate_up"][e].cpu(), inp["w_down"][e].cpu(), dtype)


@pytest.mark.parametrize("name,sample", [("dsv3_mxfp8", 1024), ("dsv3_mxfp8_skew", 1024),
                                         ("dsv3_mxfp8_skew05", 1024), ("dsv3_mxfp8_skew_16k", 1024)])
def test_fullsize_sampled_parity_and_fused_equality(name, sample):
    w, inp, layer = _setup(name)
    staged = layer.forward().clone()
    idx = to_np(layer.idx)
    fused = layer.forward(fused=True)
    assert layer.device_status() == 0
    assert torch.equal(fused, staged)
    toks = np.sort(np.random.default_rng(0).choice(w.N, size=sample, replace=False))
    ref = O.forward(inp, w.E, w.k, w.S, w.dtype, tokens=toks, weights=_oracle_weights(inp, w.dtype))
    assert check_routing(idx, ref["idx"], ref["logits"], ref["gap"]) > 0.97   # every token
    ok = (ref["gap"] >= TIE_TAU)[toks]
    err = row_rel_err(to_np(staged)[toks][ok], ref["out"][ok])
    assert err.max() < TOL[w.dtype], err.max()
    if w.skew:
        counts = np.bincount(ref["idx"].ravel(), minlength=w.E)
        print(f"{name}: max/mean expert load {counts.max() / counts.mean():.1f}, "
              f"{(counts == 0).sum()} empty experts")


@pytest.mark.parametrize("name", ["dsv3_mxfp8_skew", "dsv3_mxfp8_skew05"])
def test_fullsize_hottest_expert_rows(name):
    """The hottest expert of a skewed layer (every token, or about 18x the mean):
    all of its slot rows through the expert FFN entry point against the oracle's
    FFN of those rows."""
    from token_dispatch_expert_top_gb300 import moe as M
    w, inp, layer = _setup(name)
    layer.forward()
    shape = layer.shape
    counts = torch.empty(w.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(w.E + 1, dtype=torch.int32, device="cuda")
    sched = torch.empty((w.T, 2), dtype=torch.int32, device="cuda")
    inv = torch.empty((w.N, w.k), dtype=torch.int32, device="cuda")
    M.moe_layout(layer.idx, shape, counts, offsets, sched, inv, layer.ws)
    from token_dispatch_expert_top_gb300.layer import quantize_mxfp8
    xq, xs = quantize_mxfp8(layer.x)
    rows = (sched[:, 0].long() * w.rows_per_shard + sched[:, 1].long())
    a, a_s = xq[rows].contiguous(), xs[rows].contiguous()
    y = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    M.moe_expert_ffn(a, a_s, offsets, layer.wgu, layer.wgu_sf, layer.wd, layer.wd_sf, shape, y, layer.ws)
    assert M.moe_last_device_status(layer.ws) == 0
    cnt = to_np(counts)
    e = int(cnt.argmax())
    off = to_np(offsets)
    pick = np.arange(off[e], off[e + 1])
    tok = to_np(rows)[pick]
    a64 = O.mxfp8_values(O._f64(inp["x"][torch.from_numpy(tok).cuda()]))
    wg, wu, wd = _oracle_weights(inp, w.dtype)(e)
    ref = O.expert_ffn(a64, wg, wu, wd, w.dtype)
    err = row_rel_err(to_np(y)[pick], ref)
    assert err.max() < TOL[w.dtype], (e, cnt[e], err.max())


@pytest.mark.parametrize("name", ["dsv3_mxfp8_skew", "dsv3_mxfp8_skew05"])
@pytest.mark.parametrize("ring", [64, 256, 1024])
def test_fullsize_skew_ring_sweep_bitwise(ring, name):
    from token_dispatch_expert_top_gb300 import moe as M
    need_cuda()
    p = M.Params(ring, ring // 2, 0, 0, 0, 0)
    w, inp, layer = _setup(name, params=p)
    staged = layer.forward().clone()
    fused = layer.forward(fused=True)
    assert layer.device_status() == 0
    assert torch.equal(fused, staged)


def test_fullsize_backward_sampled_parity():
    """The 16384-token skewed layer, forward + backward: dx of 64 sampled tokens,
    and the weight gradients of one expert from each load band -- a light one
    (<= 64 slots) and a medium one (100-600 slots), with their router rows and bias
    entries, and a heavy one (the most loaded expert with at most N/2 slots, else
    the hottest; dW_gate_up and dW_down only, since its router row needs every
    token's FFN) -- against the oracle's backward restricted to those tokens and
    experts.  Tokens and the light and medium experts are drawn among those whose
    routing is away from top-k near-ties."""
    need_cuda()
    from token_dispatch_expert_top_gb300.layer import MoeLayer
    w = synth.WORKLOADS["dsv3_mxfp8_skew_16k"]
    inp = synth.make_inputs(w)
    layer = MoeLayer(w, inp, train=True)
    gen = torch.Generator(device="cuda").manual_seed(3)
    dout = torch.randn((w.N, w.H), generator=gen, device="cuda").to(torch.bfloat16)
    layer.forward_train()
    dx, dwr, db, dwgu, dwd = layer.backward(dout)
    assert layer.device_status() == 0 and layer.backward_status() == 0
    lg = O.router_logits(inp["x"], inp["w_router"], inp["bias"])
    gap = O.topk_gap(lg, w.k)
    ridx, _ = O.route_topk(lg, w.k)
    assert check_routing(to_np(layer.saved["idx"]), ridx, lg, gap) > 0.97
    rng = np.random.default_rng(0)
    toks = np.sort(rng.choice(np.nonzero(gap >= TIE_TAU)[0], 64, replace=False))
    counts = np.bincount(ridx.ravel(), minlength=w.E)
    clean = lambda e: np.all(gap[(ridx == e).any(axis=1)] >= TIE_TAU)
    light = [int(e) for e in np.argsort(counts, kind="stable") if 0 < counts[e] <= 64 and clean(e)]
    mid = [int(e) for e in np.argsort(counts, kind="stable") if 100 <= counts[e] <= 600 and clean(e)]
    under = [int(e) for e in np.argsort(-counts, kind="stable") if counts[e] <= w.N // 2]
    heavy = under[0] if under and counts[under[0]] > 600 else int(np.argmax(counts))
    rexps = np.array(sorted(light[:1] + mid[:1]))
    assert len(rexps) >= 1
    exps = np.array(sorted(set(rexps.tolist()) | {heavy}))
    ref = O.backward(inp, w.E, w.k, w.S, w.dtype, dout, tokens=toks, experts=exps,
                     weights=_oracle_weights(inp, w.dtype), router_experts=rexps)
    tol = TOL[w.dtype]
    err = row_rel_err(to_np(dx)[toks], ref["dx"])
    assert err.max() < tol, ("dx", err.max())
    g_gu, g_d, g_r, g_b = to_np(dwgu), to_np(dwd), to_np(dwr), to_np(db)
    for i, e in enumerate(exps):
        e_gu = row_rel_err(g_gu[e], ref["dw_gate_up"][i]).max()
        e_d = row_rel_err(g_d[e], ref["dw_down"][i]).max()
        assert max(e_gu, e_d) < tol, (int(e), int(counts[e]), e_gu, e_d)
    for i, e in enumerate(rexps):
        e_r = row_rel_err(g_r[e:e + 1], ref["dw_router"][i:i + 1]).max()
        assert e_r < tol, (int(e), int(counts[e]), e_r)
        scale = np.abs(ref["dlogit"][:, e]).sum()
        assert abs(g_b[e] - ref["dbias"][i]) <= tol * scale, (int(e), g_b[e], ref["dbias"][i])
    print(f"backward 16k: dx err {err.max():.4f}, experts {exps.tolist()} with "
          f"{counts[exps].tolist()} slots (router rows of {rexps.tolist()})")


def test_small_bf16_backward_sampled_parity():
    """The BF16 layer (N=4096, H=2048, I=1408, E=64, top-6): I is not a multiple of
    256, so the dgrad and wgrad GEMMs run their padded column tiles.  dx of sampled
    tokens and the full weight gradients of two experts (≈340 slots each) against the
    oracle's backward, away from top-k near-ties."""
    need_cuda()
    from token_dispatch_expert_top_gb300.layer import MoeLayer
    w = synth.WORKLOADS["small_bf16"]
    inp = synth.make_inputs(w)
    layer = MoeLayer(w, inp, train=True)
    dout = torch.randn((w.N, w.H), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    layer.forward_train()
    dx, dwr, db, dwgu, dwd = layer.backward(dout.cuda())
    assert layer.device_status() == 0 and layer.backward_status() == 0
    lg = O.router_logits(inp["x"], inp["w_router"], inp["bias"])
    gap = O.topk_gap(lg, w.k)
    ridx, _ = O.route_topk(lg, w.k)
    assert check_routing(to_np(layer.saved["idx"]), ridx, lg, gap) > 0.99
    rng = np.random.default_rng(0)
    toks = np.sort(rng.choice(np.nonzero(gap >= TIE_TAU)[0], 16, replace=False))
    counts = np.bincount(ridx.ravel(), minlength=w.E)
    cand = [int(e) for e in np.argsort(counts, kind="stable")
            if np.all(gap[(ridx == e).any(axis=1)] >= TIE_TAU)]
    exps = np.array(sorted(cand[:2]))
    ref = O.backward(inp, w.E, w.k, w.S, w.dtype, dout, tokens=toks, experts=exps)
    tol = TOL[w.dtype]
    assert row_rel_err(to_np(dx)[toks], ref["dx"]).max() < tol
    g_gu, g_d, g_r = to_np(dwgu), to_np(dwd), to_np(dwr)
    for i, e in enumerate(exps):
        err = max(row_rel_err(g_gu[e], ref["dw_gate_up"][i]).max(),
                  row_rel_err(g_d[e], ref["dw_down"][i]).max(),
                  row_rel_err(g_r[e:e + 1], ref["dw_router"][i:i + 1]).max())
        assert err < tol, (int(e), int(counts[e]), err)
