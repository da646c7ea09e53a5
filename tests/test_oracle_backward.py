"""Pins of the oracle's backward pass.

The backward is pinned against things other than itself:
  * central finite differences of the oracle's own (already pinned) FP64 forward,
    on tiny unrounded layers whose top-k choices are far from ties;
  * torch autograd through a float64 torch statement of the layer (the derivative
    is taken by autograd, not by hand);
  * closed forms and invariants the mathematics fixes: the layer output is linear in
    W_down and in W_up (Euler's identity gives sum <dW, W> = L), adding one vector to
    every router row or one constant to every bias leaves the output unchanged (their
    gradients sum to zero), top-1 routing has no router gradient, and identical
    experts make the gates irrelevant.
"""
import numpy as np
import pytest
import torch

import oracle as O


def _layer(N=8, H=32, I=16, E=6, k=2, seed=0, bias=True, spread=3.0):
    rng = np.random.default_rng(seed)
    inp = {
        "x": rng.standard_normal((N, H)),
        "w_router": rng.standard_normal((E, H)) * spread / np.sqrt(H),
        "bias": rng.standard_normal(E) if bias else None,
        "w_gate_up": rng.standard_normal((E, 2 * I, H)) / np.sqrt(H),
        "w_down": rng.standard_normal((E, H, I)) / np.sqrt(I),
    }
    dout = rng.standard_normal((N, H))
    return inp, dout


def _loss(inp, E, k, S, dout, dtype="f64"):
    return float(np.sum(O.forward(inp, E, k, S, dtype)["out"] * dout))


def _grads(b):
    return {"x": b["dx"], "w_router": b["dw_router"], "bias": b["dbias"],
            "w_gate_up": b["dw_gate_up"], "w_down": b["dw_down"]}


def _min_gap(inp, k):
    lg = O.router_logits(inp["x"], inp["w_router"], inp["bias"])
    return O.topk_gap(lg, k).min()


# ------------------------------------------------------------------ finite differences
@pytest.mark.parametrize("N,H,I,E,k", [(8, 32, 16, 6, 2), (5, 16, 8, 4, 3), (6, 8, 4, 3, 3),
                                       (7, 16, 8, 5, 1)])
def test_directional_derivatives_match_central_differences(N, H, I, E, k):
    inp, dout = _layer(N, H, I, E, k, seed=N * 100 + E)
    S = 1
    eps = 1e-6
    assert _min_gap(inp, k) > 1e-3          # no choice flips under the perturbation
    b = O.backward(inp, E, k, S, "f64", dout)
    g = _grads(b)
    rng = np.random.default_rng(1)
    for name in ("x", "w_router", "bias", "w_gate_up", "w_down"):
        for _ in range(3):
            d = rng.standard_normal(inp[name].shape)
            plus = dict(inp, **{name: inp[name] + eps * d})
            minus = dict(inp, **{name: inp[name] - eps * d})
            fd = (_loss(plus, E, k, S, dout) - _loss(minus, E, k, S, dout)) / (2 * eps)
            an = float(np.sum(g[name] * d))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_single_entries_match_central_differences():
    N, H, I, E, k = 6, 16, 8, 4, 2
    inp, dout = _layer(N, H, I, E, k, seed=5)
    assert _min_gap(inp, k) > 1e-3
    b = O.backward(inp, E, k, 1, "f64", dout)
    g = _grads(b)
    rng = np.random.default_rng(2)
    eps = 1e-6
    for name in ("x", "w_router", "bias", "w_gate_up", "w_down"):
        shape = inp[name].shape
        for _ in range(6):
            at = tuple(int(rng.integers(0, s)) for s in shape)
            plus = {kk: (v.copy() if kk == name else v) for kk, v in inp.items()}
            minus = {kk: (v.copy() if kk == name else v) for kk, v in inp.items()}
            plus[name][at] += eps
            minus[name][at] -= eps
            fd = (_loss(plus, E, k, 1, dout) - _loss(minus, E, k, 1, dout)) / (2 * eps)
            assert abs(fd - g[name][at]) <= 1e-7 * max(1.0, abs(fd)), (name, at, fd, g[name][at])


# ------------------------------------------------------------------ torch autograd
def _torch_layer_grads(inp, E, k, dout):
    """The layer written with torch float64 ops; autograd takes the derivative."""
    t = {kk: torch.tensor(v, dtype=torch.float64, requires_grad=True) for kk, v in inp.items()
         if v is not None}
    x, wr, wgu, wd = t["x"], t["w_router"], t["w_gate_up"], t["w_down"]
    I = wd.shape[2]
    logits = x @ wr.T + (t["bias"] if "bias" in t else 0.0)
    sel = torch.topk(logits.detach(), k, dim=1).indices
    gates = torch.softmax(torch.gather(logits, 1, sel), dim=1)
    out = torch.zeros_like(x)
    for j in range(k):
        wg_j = wgu[sel[:, j], :I]                       # [N, I, H]
        wu_j = wgu[sel[:, j], I:]
        wd_j = wd[sel[:, j]]                            # [N, H, I]
        u = torch.einsum("nh,nih->ni", x, wg_j)
        v = torch.einsum("nh,nih->ni", x, wu_j)
        h = torch.nn.functional.silu(u) * v
        y = torch.einsum("ni,nhi->nh", h, wd_j)
        out = out + gates[:, j:j + 1] * y
    (out * torch.tensor(dout)).sum().backward()
    return {kk: v.grad.numpy() for kk, v in t.items()}


@pytest.mark.parametrize("N,H,I,E,k,bias", [(16, 32, 24, 8, 2, True), (12, 16, 8, 4, 4, False),
                                            (10, 8, 16, 1, 1, False), (9, 24, 8, 6, 3, True)])
def test_matches_torch_autograd(N, H, I, E, k, bias):
    inp, dout = _layer(N, H, I, E, k, seed=17 + N, bias=bias)
    b = O.backward(inp, E, k, 1, "f64", dout)
    ref = _torch_layer_grads(inp, E, k, dout)
    g = _grads(b)
    for name, r in ref.items():
        np.testing.assert_allclose(g[name], r, rtol=1e-10, atol=1e-12, err_msg=name)


def test_intermediates_match_torch_autograd():
    """dh, du, dv and da of every pair against autograd of one expert's FFN."""
    inp, dout = _layer(10, 16, 8, 4, 2, seed=3)
    E, k = 4, 2
    b = O.backward(inp, E, k, 1, "f64", dout)
    I = 8
    for p_i, p in enumerate(b["pairs"]):
        n, j = divmod(int(p), k)
        e = int(b["idx"][n, j])
        a = torch.tensor(inp["x"][n], requires_grad=True)
        wg = torch.tensor(inp["w_gate_up"][e, :I])
        wu = torch.tensor(inp["w_gate_up"][e, I:])
        wd = torch.tensor(inp["w_down"][e])
        u = (wg @ a).detach().requires_grad_(True)
        v = (wu @ a).detach().requires_grad_(True)
        h = (torch.nn.functional.silu(u) * v)
        hh = h.detach().requires_grad_(True)
        y = wd @ hh
        dy = torch.tensor(b["dy"][p_i])
        y.backward(dy)
        h.backward(hh.grad)
        np.testing.assert_allclose(b["dh"][p_i], hh.grad.numpy(), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(b["du"][p_i], u.grad.numpy(), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(b["dv"][p_i], v.grad.numpy(), rtol=1e-12, atol=1e-14)
        da = (wg.T @ u.grad + wu.T @ v.grad).numpy()
        np.testing.assert_allclose(b["da"][p_i], da, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(b["dy"][p_i], b["gate"][n, j] * dout[n], rtol=0, atol=0)


# ------------------------------------------------------------------ closed forms
@pytest.mark.parametrize("dtype", ["f64", "f32", "bf16", "mxfp8"])
def test_euler_identity_for_the_linear_weights(dtype):
    """out is linear in W_down and in W_up, so sum_e <dW, W> = L for each (for the
    rounded dtypes, with the values the forward used and L before the output's own
    rounding, up to the rounding of h and y)."""
    inp, dout = _layer(12, 64, 32, 4, 2, seed=11)
    E, k = 4, 2
    if dtype != "f64":
        inp = {kk: (None if v is None else O.round_to(v, "bf16" if dtype == "mxfp8" else dtype))
               for kk, v in inp.items()}
    b = O.backward(inp, E, k, 1, dtype, dout)
    # L through the unrounded combine of the forward's y
    f = O.forward(inp, E, k, 1, dtype)
    L = float(np.sum(O.combine(f["y"], np.arange(12 * k, dtype=np.int32).reshape(12, k),
                               f["gate"]) * dout))
    I = 32
    wd_vals = np.stack([O.expert_operands(inp["w_gate_up"][e], inp["w_down"][e], dtype)[2]
                        for e in range(E)])
    wu_vals = np.stack([O.expert_operands(inp["w_gate_up"][e], inp["w_down"][e], dtype)[1]
                        for e in range(E)])
    s_d = float(np.sum(b["dw_down"] * wd_vals))
    s_u = float(np.sum(b["dw_gate_up"][:, I:] * wu_vals))
    # the wgrad GEMMs round dy and h along the slots (MXFP8 blocks of 32 slots)
    tol = {"f64": 1e-10, "f32": 1e-5, "bf16": 2e-2, "mxfp8": 6e-2}[dtype]
    assert abs(s_d - L) <= tol * max(1.0, abs(L)), (s_d, L)
    # W_up feeds h, which is rounded before the down GEMM: exact only without rounding
    tol_u = 1e-10 if dtype == "f64" else (1e-5 if dtype == "f32" else 6e-2)
    assert abs(s_u - L) <= tol_u * max(1.0, abs(L)), (s_u, L)


@pytest.mark.parametrize("dtype", ["f64", "bf16", "mxfp8"])
def test_router_shift_invariances(dtype):
    """Adding one vector to every router row, or one constant to every bias, moves
    every logit of a token by the same amount: gates and output do not change, so
    the router gradients sum to zero over experts, and so does each token's dlogit."""
    inp, dout = _layer(32, 64, 32, 8, 3, seed=12)
    b = O.backward(inp, 8, 3, 2, dtype, dout)
    scale = np.abs(b["dw_router"]).max()
    assert scale > 0
    np.testing.assert_allclose(b["dw_router"].sum(axis=0), 0.0, atol=1e-12 * max(1, scale) * 8)
    np.testing.assert_allclose(b["dbias"].sum(), 0.0, atol=1e-13 * 8)
    np.testing.assert_allclose(b["dlogit"].sum(axis=1), 0.0, atol=1e-14)
    # only the selected experts of a token have a logit gradient
    mask = np.zeros_like(b["dlogit"], dtype=bool)
    np.put_along_axis(mask, b["idx"].astype(np.int64), True, axis=1)
    assert np.all(b["dlogit"][~mask] == 0.0)


def test_top1_routing_has_no_router_gradient():
    inp, dout = _layer(16, 32, 16, 6, 1, seed=13)
    b = O.backward(inp, 6, 1, 1, "f64", dout)
    assert np.all(b["dlogit"] == 0.0) and np.all(b["dw_router"] == 0.0)
    assert np.all(b["dbias"] == 0.0) and np.all(b["dx_router"] == 0.0)


def test_identical_experts_make_the_gates_irrelevant():
    """With every expert equal, out = FFN(x) whatever the gates (they sum to one):
    no router gradient, each token's input gradient is the dense FFN's, and the
    expert weight gradients add up to the dense FFN's."""
    N, H, I, E, k = 20, 32, 16, 5, 3
    inp, dout = _layer(N, H, I, E, k, seed=14)
    inp["w_gate_up"][:] = inp["w_gate_up"][0]
    inp["w_down"][:] = inp["w_down"][0]
    b = O.backward(inp, E, k, 1, "f64", dout)
    np.testing.assert_allclose(b["dlogit"], 0.0, atol=1e-13)
    dense = {"x": inp["x"], "w_router": inp["w_router"][:1], "bias": None,
             "w_gate_up": inp["w_gate_up"][:1], "w_down": inp["w_down"][:1]}
    d1 = O.backward(dense, 1, 1, 1, "f64", dout)
    np.testing.assert_allclose(b["dx"], d1["dx"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["dw_gate_up"].sum(0), d1["dw_gate_up"][0], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(b["dw_down"].sum(0), d1["dw_down"][0], rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("dtype,c", [("f64", -2.5), ("mxfp8", -4.0), ("bf16", 0.5)])
def test_linear_in_dout_and_zero_for_zero_dout(dtype, c):
    """Linear in dout; with rounding points, for power-of-two factors (which every
    rounding commutes with)."""
    inp, dout = _layer(12, 32, 32, 4, 2, seed=15)
    b1 = _grads(O.backward(inp, 4, 2, 1, dtype, dout))
    b2 = _grads(O.backward(inp, 4, 2, 1, dtype, c * dout))
    b0 = _grads(O.backward(inp, 4, 2, 1, dtype, np.zeros_like(dout)))
    for name in b1:
        np.testing.assert_allclose(b2[name], c * b1[name], rtol=1e-12, atol=1e-14)
        assert np.all(b0[name] == 0.0)


def test_rounded_backward_is_near_the_exact_one():
    """The rounding points move each gradient by about the formats' precision."""
    inp, dout = _layer(16, 64, 64, 4, 2, seed=18)
    b64 = O.backward(inp, 4, 2, 1, "f64", dout)
    for dtype, tol in (("bf16", 2e-2), ("mxfp8", 0.15)):
        b = O.backward(inp, 4, 2, 1, dtype, dout)
        for name in ("dx", "dw_router", "da", "du", "dv"):
            ref = b64[name]
            err = np.abs(b[name] - ref).max() / np.abs(ref).max()
            assert err < tol, (dtype, name, err)


def test_subsets_agree_with_the_full_backward():
    inp, dout = _layer(24, 32, 16, 6, 2, seed=16)
    full = O.backward(inp, 6, 2, 3, "bf16", dout)
    part = O.backward(inp, 6, 2, 3, "bf16", dout, tokens=[0, 7, 23], experts=[2, 5])
    np.testing.assert_allclose(part["dx"], full["dx"][[0, 7, 23]], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(part["dw_gate_up"], full["dw_gate_up"][[2, 5]], rtol=1e-13,
                               atol=1e-14)
    np.testing.assert_allclose(part["dw_down"], full["dw_down"][[2, 5]], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(part["dw_router"], full["dw_router"][[2, 5]], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(part["dbias"], full["dbias"][[2, 5]], rtol=1e-13, atol=1e-14)
    assert part["full"].any() and not part["full"].all()
    for i, p in enumerate(part["pairs"]):
        j = int(np.nonzero(full["pairs"] == p)[0][0])
        np.testing.assert_allclose(part["dgate"].ravel()[p], full["dgate"].ravel()[p], rtol=1e-13,
                                   atol=1e-14)
        if part["full"][i]:
            np.testing.assert_allclose(part["da"][i], full["da"][j], rtol=1e-13, atol=1e-14)
    # the router rows of one set of experts and the weight gradients of another
    r = O.backward(inp, 6, 2, 3, "bf16", dout, tokens=[4], experts=[1], router_experts=[0, 3])
    np.testing.assert_allclose(r["dw_router"], full["dw_router"][[0, 3]], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(r["dbias"], full["dbias"][[0, 3]], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(r["dw_gate_up"], full["dw_gate_up"][[1]], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(r["dx"], full["dx"][[4]], rtol=1e-13, atol=1e-14)


def test_round_along_slots_blocks_start_at_the_segment():
    """MXFP8 wgrad operands: blocks of 32 slots from the segment's first slot; the
    last, partial block is scaled by its own rows only; other formats round
    element-wise."""
    rng = np.random.default_rng(19)
    m = rng.standard_normal((40, 6)) * np.exp2(rng.integers(-8, 8, size=(40, 1)))
    q = O.round_along_slots(m, "mxfp8")
    np.testing.assert_array_equal(q[:32], O.mxfp8_values(m[:32].T).T)
    tail = np.vstack([m[32:], np.zeros((24, 6))])
    np.testing.assert_array_equal(q[32:], O.mxfp8_values(tail.T).T[:8])
    # a power-of-two column is exact; a block's scale follows its own amax
    m2 = np.zeros((32, 1))
    m2[5, 0] = 2.0 ** -20
    np.testing.assert_array_equal(O.round_along_slots(m2, "mxfp8"), m2)
    np.testing.assert_array_equal(O.round_along_slots(m, "bf16"), O.round_bf16(m))
