"""GPU parity of the backward pass through the C ABI against the oracle: the
dgrad weight packing (bit-exact), the reverse combine (bit-exact dy codes, FP32
gate and logit gradients), the expert dgrad GEMMs, the reverse dispatch, the
router weight gradient, and the whole backward of small layers."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import TIE_TAU, TOL, need_cuda, row_rel_err, to_np
from test_gpu_steps import _expected_pack, _expected_pack_sf
from token_dispatch_expert_top_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    need_cuda()
    from token_dispatch_expert_top_gb300 import moe
    return moe


def _bws(M, shape):
    ws = torch.empty(M.moe_backward_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    M.moe_workspace_init(ws)
    return ws


def _random_routing(rng, N, E, k, hot=None):
    idx = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
    if hot is not None:                      # make expert `hot` take every token
        for n in range(N):
            if hot not in idx[n]:
                idx[n, -1] = hot
    return idx


# ------------------------------------------------------------------ dgrad packing
@pytest.mark.parametrize("dtype,H,I", [("mxfp8", 512, 256), ("mxfp8", 256, 384), ("bf16", 512, 384)])
def test_pack_dgrad_weights_layout(M, dtype, H, I):
    from token_dispatch_expert_top_gb300.layer import pack_expert_weights_dgrad
    E = 2
    w = synth.Workload("packt", N=8, H=H, I=I, E=E, k=1, S=1, dtype=dtype)
    shape = M.Shape.of(w)
    g = torch.Generator().manual_seed(11)
    wgu = (torch.randn((E, 2 * I, H), generator=g) * 3).to(torch.bfloat16)
    wd = (torch.randn((E, H, I), generator=g) * 0.01).to(torch.bfloat16)
    wd[0, 5:37, 7] = 0.0                                 # a zero block in a column
    p_gu, p_gu_sf, p_d, p_d_sf = pack_expert_weights_dgrad(shape, wgu.cuda(), wd.cuda())
    Ip = (I + 255) // 256 * 256
    mx = dtype == "mxfp8"
    # W^T by definition, padded with zero rows to Ip
    gu_t = wgu.transpose(1, 2).float().numpy().astype(np.float64)            # [E][H][2I]
    d_t = np.zeros((E, Ip, H))
    d_t[:, :I] = wd.transpose(1, 2).float().numpy()                           # [E][I][H]
    rows = lambda n, r: n * 256 + r
    if mx:
        c_gu, s_gu = O.quantize_mxfp8(gu_t.reshape(-1, 2 * I))
        c_d, s_d = O.quantize_mxfp8(d_t.reshape(-1, H))
        exp_gu = _expected_pack(c_gu.reshape(E, H, 2 * I), rows, H // 256, 2 * I // 128)
        exp_d = _expected_pack(c_d.reshape(E, Ip, H), rows, Ip // 256, H // 128)
        np.testing.assert_array_equal(to_np(p_gu), exp_gu)
        np.testing.assert_array_equal(to_np(p_d), exp_d)
        np.testing.assert_array_equal(
            to_np(p_gu_sf), _expected_pack_sf(s_gu.reshape(E, H, -1), rows, H // 256, 2 * I // 128))
        np.testing.assert_array_equal(
            to_np(p_d_sf), _expected_pack_sf(s_d.reshape(E, Ip, -1), rows, Ip // 256, H // 128))
    else:
        b_gu = wgu.transpose(1, 2).contiguous().view(torch.uint8).numpy()      # [E][H][4I] bytes
        b_d = np.zeros((E, Ip, 2 * H), dtype=np.uint8)
        b_d[:, :I] = wd.transpose(1, 2).contiguous().view(torch.uint8).numpy()
        np.testing.assert_array_equal(to_np(p_gu), _expected_pack(b_gu, rows, H // 256, 4 * I // 128))
        np.testing.assert_array_equal(to_np(p_d), _expected_pack(b_d, rows, Ip // 256, 2 * H // 128))


# ------------------------------------------------------------------ reverse combine
@pytest.mark.parametrize("dtype,N,H,E,k", [("mxfp8", 300, 1024, 16, 6), ("bf16", 257, 512, 8, 2),
                                           ("mxfp8", 64, 256, 32, 16)])
def test_reverse_combine(M, dtype, N, H, E, k):
    rng = np.random.default_rng(21)
    w = synth.Workload("rc", N=N, H=H, I=128, E=E, k=k, S=1, dtype=dtype)
    shape = M.Shape.of(w)
    ws = _bws(M, shape)
    T = N * k
    mx = dtype == "mxfp8"
    dout = torch.randn((N, H), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    dout[3] *= 1e-30                                       # a token with tiny gradients
    y = torch.randn((T, H), generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    _, _, _, inv_np = O.layout(_random_routing(rng, N, E, k), E, 1)
    g = rng.random((N, k)).astype(np.float32) + 0.05
    g /= g.sum(1, keepdims=True)
    dy = torch.empty((T, H), dtype=torch.uint8 if mx else torch.bfloat16, device="cuda")
    dy_sf = torch.empty((T, H // 32), dtype=torch.uint8, device="cuda") if mx else None
    f = lambda *s: torch.empty(s, dtype=torch.float32, device="cuda")
    dgate, dlogit, sgate, sdl = f(N, k), f(N, k), f(T), f(T)
    M.moe_reverse_combine(dout.cuda(), y.cuda(), torch.from_numpy(inv_np).cuda(),
                          torch.from_numpy(g).cuda(), shape, dy, dy_sf, dgate, dlogit, sgate, sdl, ws)
    assert M.moe_last_device_status(ws) == 0
    # dy: the FP32 product g * dout, then the oracle's quantiser / BF16 rounding
    prod = (g.reshape(N, k, 1) * to_np(dout).reshape(N, 1, H)).astype(np.float32)   # IEEE FP32 products
    exp = np.empty((T, H))
    exp[inv_np.ravel()] = prod.reshape(T, H)
    if mx:
        oc, os_ = O.quantize_mxfp8(exp)
        np.testing.assert_array_equal(to_np(dy), oc)
        np.testing.assert_array_equal(to_np(dy_sf), os_)
    else:
        np.testing.assert_array_equal(to_np(dy), O.round_bf16(exp))
    # dgate = <dout, y[slot]> (FP32 sums), dlogit through the oracle's gate Jacobian
    d64, y64 = O._f64(dout), O._f64(y)
    ref_dg = np.einsum("nh,njh->nj", d64, y64[inv_np])
    scale = np.einsum("nh,njh->nj", np.abs(d64), np.abs(y64[inv_np]))
    assert np.all(np.abs(to_np(dgate) - ref_dg) <= 1e-5 * scale + 1e-30)
    ref_dl = O.gate_backward(g.astype(np.float64), ref_dg)
    dl_scale = g * scale.max(axis=1, keepdims=True)
    assert np.all(np.abs(to_np(dlogit) - ref_dl) <= 4e-5 * dl_scale + 1e-30)
    # per-slot copies
    np.testing.assert_array_equal(to_np(sgate)[inv_np], g)
    np.testing.assert_array_equal(to_np(sdl)[inv_np], to_np(dlogit))


# ------------------------------------------------------------------ expert dgrad
DGRAD_CASES = [
    ("mxfp8", 512, 256, [0, 1, 130, 255, 300]),
    ("mxfp8", 1024, 384, [129, 0, 256, 40]),
    ("bf16", 512, 384, [0, 1, 130, 255, 300]),
    ("mxfp8", 7168, 2048, [37, 0, 256, 129]),
]


@pytest.mark.parametrize("dtype,H,I,counts", DGRAD_CASES,
                         ids=[f"{c[0]}-H{c[1]}-I{c[2]}-E{len(c[3])}" for c in DGRAD_CASES])
def test_expert_dgrad_matches_oracle(M, dtype, H, I, counts):
    from token_dispatch_expert_top_gb300.layer import (pack_expert_weights, pack_expert_weights_dgrad,
                                                       quantize_mxfp8)
    E, T = len(counts), sum(counts)
    w = synth.Workload("dgrad", N=T, H=H, I=I, E=E, k=1, S=1, dtype=dtype)
    shape = M.Shape.of(w)
    ws = torch.empty(M.moe_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    M.moe_workspace_init(ws)
    bws = _bws(M, shape)
    g = torch.Generator().manual_seed(8)
    a = torch.randn((T, H), generator=g).to(torch.bfloat16)
    wgu = (torch.randn((E, 2 * I, H), generator=g) / H ** 0.5).to(torch.bfloat16)
    wd = (torch.randn((E, H, I), generator=g) / I ** 0.5).to(torch.bfloat16)
    dyv = torch.randn((T, H), generator=g).to(torch.bfloat16)
    offsets_np = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    offsets = torch.from_numpy(offsets_np).cuda()
    mx = dtype == "mxfp8"
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    uv = torch.empty((T, 2 * I), dtype=torch.bfloat16, device="cuda")
    if mx:
        a_c, a_s = quantize_mxfp8(a.cuda())
        packed = pack_expert_weights(shape, *quantize_mxfp8(wgu.cuda()), *quantize_mxfp8(wd.cuda()))
        M.moe_expert_ffn_train(a_c, a_s, offsets, *packed, shape, y, uv, ws)
        dy, dy_s = quantize_mxfp8(dyv.cuda())
    else:
        packed = pack_expert_weights(shape, wgu.cuda(), None, wd.cuda(), None)
        M.moe_expert_ffn_train(a.cuda(), None, offsets, *packed, shape, y, uv, ws)
        dy, dy_s = dyv.cuda(), None
    pt = pack_expert_weights_dgrad(shape, wgu.cuda(), wd.cuda())
    duv = torch.empty((T, 2 * I), dtype=torch.bfloat16, device="cuda")
    duv_c = torch.empty((T, 2 * I), dtype=torch.uint8, device="cuda") if mx else None
    duv_s = torch.empty((T, 2 * I // 32), dtype=torch.uint8, device="cuda") if mx else None
    da = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    M.moe_expert_ffn_dgrad(dy, dy_s, uv, offsets, *pt, shape, duv, duv_c, duv_s, da, bws)
    assert M.moe_last_device_status(ws) == 0 and M.moe_last_device_status(bws) == 0
    a64 = O._f64(a)
    if mx:
        a64 = O.mxfp8_values(a64)
    g_uv, g_duv, g_da, g_y = to_np(uv), to_np(duv), to_np(da), to_np(y)
    for e in range(E):
        lo, hi = offsets_np[e], offsets_np[e + 1]
        if lo == hi:
            continue
        wg, wu, wdd = O.expert_operands(wgu[e], wd[e], dtype)
        r = O.expert_ffn_backward(a64[lo:hi], wg, wu, wdd, O._f64(dyv[lo:hi]), dtype,
                                  O.expert_operands_dgrad(wgu[e], wd[e], dtype))
        # the saved pre-activations: BF16 of the FP32 sums
        assert row_rel_err(g_uv[lo:hi], np.hstack([r["u"], r["v"]])).max() < 8e-3
        assert row_rel_err(g_y[lo:hi], r["y"]).max() < TOL[dtype]
        err_duv = row_rel_err(g_duv[lo:hi], np.hstack([r["du"], r["dv"]])).max()
        err_da = row_rel_err(g_da[lo:hi], r["da"]).max()
        assert err_duv < TOL[dtype] and err_da < TOL[dtype], (e, err_duv, err_da)
    if mx:
        # The MXFP8 operand copy and the BF16 copy round the same FP32 values, so each
        # MXFP8 value lies within the MX rule's error of the BF16 one: half an E4M3
        # step (2^-4 relative; 2^-10 of the block scale below the normal range),
        # or the saturation at 448 x scale, plus the BF16 half step.
        v = to_np(duv).astype(np.float64)
        sc = np.exp2(to_np(duv_s).astype(np.float64) - 127).repeat(32, axis=1)
        q = O.dequantize_mxfp8(to_np(duv_c), to_np(duv_s))
        bound = np.maximum(2.0 ** -4 * np.abs(v), np.abs(v) - 448 * sc) + 2.0 ** -10 * sc
        assert np.all(np.abs(q - v) <= bound + 2.0 ** -8 * np.abs(v))
        # and the scale is the MX rule's for the block's amax (up to the BF16 step)
        amax = np.abs(v).reshape(T, -1, 32).max(axis=2)
        want = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8
        got = to_np(duv_s).astype(np.float64) - 127
        assert np.all((np.abs(got - want) <= 1) | (amax == 0))


# ------------------------------------------------------------------ reverse dispatch
@pytest.mark.parametrize("N,H,E,k", [(300, 1024, 16, 6), (77, 256, 40, 16)])
def test_reverse_dispatch(M, N, H, E, k):
    rng = np.random.default_rng(31)
    w = synth.Workload("rd", N=N, H=H, I=128, E=E, k=k, S=1, dtype="mxfp8")
    shape = M.Shape.of(w)
    ws = _bws(M, shape)
    T = N * k
    idx = _random_routing(rng, N, E, k)
    _, _, _, inv_np = O.layout(idx, E, 1)
    da = torch.randn((T, H), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    wr = (torch.randn((E, H), generator=torch.Generator().manual_seed(4)) / H ** 0.5).to(torch.bfloat16)
    dl = rng.standard_normal((N, k)).astype(np.float32)
    dx = torch.empty((N, H), dtype=torch.bfloat16, device="cuda")
    M.moe_reverse_dispatch(da.cuda(), torch.from_numpy(inv_np).cuda(), torch.from_numpy(idx).cuda(),
                           torch.from_numpy(dl).cuda(), wr.cuda(), shape, dx, ws)
    assert M.moe_last_device_status(ws) == 0
    ref = O.combine(O._f64(da), inv_np, np.ones((N, k))) + np.einsum(
        "nj,njh->nh", dl.astype(np.float64), O._f64(wr)[idx])
    assert row_rel_err(to_np(dx), O.round_bf16(ref)).max() < 8e-3


# ------------------------------------------------------------------ router wgrad
@pytest.mark.parametrize("N,H,E,k,S,hot", [(600, 1024, 16, 4, 3, None), (1000, 512, 64, 8, 10, 5),
                                           (64, 256, 256, 2, 1, None)])
def test_router_wgrad(M, N, H, E, k, S, hot):
    rng = np.random.default_rng(41)
    w = synth.Workload("rw", N=N, H=H, I=128, E=E, k=k, S=S, dtype="bf16")
    shape = M.Shape.of(w)
    ws = _bws(M, shape)
    T = N * k
    idx = _random_routing(rng, N, E, k, hot)
    counts, offsets_np, sched_np, inv_np = O.layout(idx, E, S)
    x = torch.randn((N, H), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    sdl = rng.standard_normal(T).astype(np.float32)
    dw = torch.full((E, H), float("nan"), dtype=torch.float32, device="cuda")
    db = torch.full((E,), float("nan"), dtype=torch.float32, device="cuda")
    M.moe_router_wgrad(x.cuda(), torch.from_numpy(sched_np).cuda(),
                       torch.from_numpy(offsets_np).cuda(), torch.from_numpy(sdl).cuda(), shape, dw,
                       db, ws)
    assert M.moe_last_device_status(ws) == 0
    tok = sched_np[:, 0] * (N // S) + sched_np[:, 1]
    x64 = O._f64(x)
    ref = np.zeros((E, H))
    ref_b = np.zeros(E)
    for e in range(E):
        s = slice(offsets_np[e], offsets_np[e + 1])
        ref[e] = sdl[s].astype(np.float64) @ x64[tok[s]]
        ref_b[e] = sdl[s].astype(np.float64).sum()
    absref = np.zeros((E, H))
    for e in range(E):
        s = slice(offsets_np[e], offsets_np[e + 1])
        absref[e] = np.abs(sdl[s]).astype(np.float64) @ np.abs(x64[tok[s]])
    got = to_np(dw)
    assert np.all(np.abs(got - ref) <= 1e-5 * absref + 1e-30)
    assert np.all(got[counts == 0] == 0.0)
    np.testing.assert_allclose(to_np(db), ref_b, rtol=1e-5, atol=1e-4)


# ------------------------------------------------------------------ whole backward
BWD_LAYERS = [
    synth.Workload("bwd_mx", N=512, H=512, I=256, E=16, k=4, S=4, dtype="mxfp8"),
    synth.Workload("bwd_bf16", N=256, H=512, I=384, E=8, k=2, S=2, dtype="bf16"),
    synth.Workload("bwd_mx_skew", N=512, H=1024, I=256, E=32, k=8, S=4, dtype="mxfp8", skew=3.0),
    # top-1: the renormalised gate is exactly 1, so the router gets no gradient
    synth.Workload("bwd_top1", N=256, H=512, I=256, E=16, k=1, S=2, dtype="mxfp8"),
    # the largest expert count the library takes; many experts have no slots
    synth.Workload("bwd_max_experts", N=512, H=256, I=128, E=1024, k=4, S=4, dtype="bf16"),
]


@pytest.mark.parametrize("w", BWD_LAYERS, ids=lambda w: w.name)
def test_backward_layer_matches_oracle(M, w):
    """moe_forward_train then moe_backward against the oracle's backward: every
    token's input gradient, every router row and bias entry.  The seeds have no
    top-k near-ties (smallest FP64 gap > 4e-4), so both sides route alike."""
    from token_dispatch_expert_top_gb300.layer import MoeLayer
    inp = synth.make_inputs(w, device="cpu")
    layer = MoeLayer(w, inp, train=True)
    dout = torch.randn((w.N, w.H), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    layer.forward_train()
    dx, dwr, db, dwgu, dwd = layer.backward(dout.cuda())
    assert layer.device_status() == 0 and layer.backward_status() == 0
    ref = O.backward(inp, w.E, w.k, w.S, w.dtype, dout)
    np.testing.assert_array_equal(to_np(layer.saved["idx"]), ref["idx"])
    np.testing.assert_array_equal(to_np(layer.saved["inv"]), ref["inv"])
    tol = TOL[w.dtype]
    err_dx = row_rel_err(to_np(dx), ref["dx"])
    assert err_dx.max() < tol, err_dx.max()
    live = to_np(layer.saved["offsets"])
    used = np.diff(live) > 0
    err_wr = row_rel_err(to_np(dwr)[used], ref["dw_router"][used])
    assert err_wr.max() < tol, err_wr.max()
    assert np.all(to_np(dwr)[~used] == 0.0)
    assert np.abs(to_np(db) - ref["dbias"]).max() <= tol * np.abs(ref["dbias"]).max()
    if w.k == 1:
        assert not to_np(dwr).any() and not to_np(db).any()
    # expert weight gradients: every row of every expert with at least 4 slots; an
    # expert with fewer has a gradient of rank < 4 whose row i scales with one du_i
    # (itself an FP32 sum rounded to BF16 that cancellation can leave a few BF16 ulps
    # off), so it is measured against its whole matrix's largest entry; zeros otherwise
    g_gu, g_d = to_np(dwgu), to_np(dwd)
    cnt = np.diff(live)
    many, few = cnt >= 4, (cnt > 0) & (cnt < 4)
    err_w = max(row_rel_err(g_gu[many].reshape(-1, w.H), ref["dw_gate_up"][many].reshape(-1, w.H)).max(initial=0),
                row_rel_err(g_d[many].reshape(-1, w.I), ref["dw_down"][many].reshape(-1, w.I)).max(initial=0))
    for e in np.flatnonzero(few):
        for got, want in ((g_gu[e], ref["dw_gate_up"][e]), (g_d[e], ref["dw_down"][e])):
            err_w = max(err_w, np.abs(got - want).max() / max(np.abs(want).max(), 1e-30))
    assert err_w < tol, err_w
    assert np.all(g_gu[~used] == 0.0) and np.all(g_d[~used] == 0.0)
    # deterministic: a second backward is bitwise identical
    dx1, dwr1, db1, gu1, d1 = dx.clone(), dwr.clone(), db.clone(), dwgu.clone(), dwd.clone()
    layer.backward(dout.cuda())
    assert torch.equal(dx1, layer.dx) and torch.equal(dwr1, layer.dw_router)
    assert torch.equal(db1, layer.dbias)
    assert torch.equal(gu1, layer.dw_gate_up) and torch.equal(d1, layer.dw_down)


# ------------------------------------------------------------------ expert wgrad
WGRAD_CASES = [
    # dtype, N, H, I, E, k, hot (an expert every token picks), empty expert
    ("mxfp8", 300, 512, 256, 6, 2, 1, 4),
    ("bf16", 200, 512, 384, 4, 2, None, 2),
    ("mxfp8", 64, 7168, 2048, 4, 2, None, None),
]


@pytest.mark.parametrize("dtype,N,H,I,E,k,hot,empty", WGRAD_CASES,
                         ids=[f"{c[0]}-H{c[2]}-I{c[3]}-E{c[4]}" for c in WGRAD_CASES])
def test_expert_wgrad_matches_oracle(M, dtype, N, H, I, E, k, hot, empty):
    rng = np.random.default_rng(51)
    S = 2
    w = synth.Workload("wg", N=N, H=H, I=I, E=E, k=k, S=S, dtype=dtype)
    shape = M.Shape.of(w)
    ws = _bws(M, shape)
    T = N * k
    idx = np.empty((N, k), dtype=np.int32)
    pool = [e for e in range(E) if e != empty]
    for n in range(N):
        idx[n] = rng.choice(pool, size=k, replace=False)
        if hot is not None and hot not in idx[n]:
            idx[n, -1] = hot
    counts, offsets_np, sched_np, _ = O.layout(idx, E, S)
    gen = torch.Generator().manual_seed(6)
    x = torch.randn((N, H), generator=gen).to(torch.bfloat16)
    dout = torch.randn((N, H), generator=gen).to(torch.bfloat16)
    uv = (torch.randn((T, 2 * I), generator=gen) * 2).to(torch.bfloat16)
    duv = (torch.randn((T, 2 * I), generator=gen) * 0.1).to(torch.bfloat16)
    sg = (rng.random(T) * 0.9 + 0.1).astype(np.float32)
    dwgu = torch.full((E, 2 * I, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    dwd = torch.full((E, H, I), float("nan"), dtype=torch.bfloat16, device="cuda")
    M.moe_expert_wgrad(duv.cuda(), x.cuda(), dout.cuda(), uv.cuda(), torch.from_numpy(sched_np).cuda(),
                       torch.from_numpy(sg).cuda(), torch.from_numpy(offsets_np).cuda(), shape, dwgu, dwd,
                       ws)
    assert M.moe_last_device_status(ws) == 0
    tok = sched_np[:, 0] * (N // S) + sched_np[:, 1]
    x64, d64, uv64, duv64 = O._f64(x), O._f64(dout), O._f64(uv), O._f64(duv)
    g_gu, g_d = to_np(dwgu), to_np(dwd)
    for e in range(E):
        s = slice(offsets_np[e], offsets_np[e + 1])
        if counts[e] == 0:
            assert np.all(g_gu[e] == 0.0) and np.all(g_d[e] == 0.0)
            continue
        dy = sg[s].astype(np.float64)[:, None] * d64[tok[s]]
        dwg, dwu, dwdn = O.expert_wgrad(x64[tok[s]], duv64[s, :I], duv64[s, I:], dy, uv64[s, :I],
                                        uv64[s, I:], dtype)
        err = max(row_rel_err(g_gu[e, :I], dwg).max(), row_rel_err(g_gu[e, I:], dwu).max(),
                  row_rel_err(g_d[e], dwdn).max())
        assert err < 2e-2, (e, counts[e], err)


def test_backward_empty_batch_zeroes_weight_gradients(M):
    """N = 0: no expert has slots, so every weight gradient is zero."""
    w = synth.Workload("bwd_empty", N=0, H=512, I=256, E=8, k=2, S=1, dtype="mxfp8")
    shape = M.Shape.of(w)
    ws = torch.empty(max(M.moe_backward_workspace_bytes(shape), 256), dtype=torch.uint8, device="cuda")
    M.moe_workspace_init(ws)
    dummy = torch.empty(64, dtype=torch.bfloat16, device="cuda")
    dwr = torch.full((w.E, w.H), float("nan"), device="cuda")
    db = torch.full((w.E,), float("nan"), device="cuda")
    dwgu = torch.full((w.E, 2 * w.I, w.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    dwd = torch.full((w.E, w.H, w.I), float("nan"), dtype=torch.bfloat16, device="cuda")
    M.moe_backward(dummy, dummy, dummy, M.Saved(), dummy, None, dummy, None, shape, None, dummy, dwr, db,
                   dwgu, dwd, ws)
    assert M.moe_last_device_status(ws) == 0
    for t in (dwr, db, dwgu, dwd):
        assert not t.float().isnan().any() and not t.float().any()
