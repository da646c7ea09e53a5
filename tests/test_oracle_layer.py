"""Pins of the oracle's router, layout, expert FFN and combine: brute force on tiny
inputs, library routines (numpy stable argsort, cumsum, scipy softmax, torch matmul
and silu), invariants and closed forms."""
import itertools
import math

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle as O
from token_dispatch_expert_top_gb300 import synth


# ----------------------------------------------------------------------------- top-k
@pytest.mark.parametrize("E,k", [(2, 1), (4, 2), (6, 3), (8, 2), (8, 3), (5, 5)])
def test_topk_matches_brute_force_subsets(E, k):
    rng = np.random.default_rng(E * 10 + k)
    # integer-valued logits make ties common
    logits = rng.integers(-3, 4, size=(300, E)).astype(np.float64)
    idx, gate = O.route_topk(logits, k)
    for n in range(logits.shape[0]):
        l = logits[n]
        # the best subset: largest logit sum; among equal sums the one whose sorted
        # (logit desc, index asc) list is smallest -- i.e. lower indices win ties
        best = max(itertools.combinations(range(E), k),
                   key=lambda c: (sum(l[list(c)]), [-i for i in sorted(c)]))
        assert sorted(idx[n].tolist()) == sorted(best), (n, l, idx[n], best)
        # listed by descending logit, ties by ascending index
        ordered = sorted(best, key=lambda e: (-l[e], e))
        assert idx[n].tolist() == ordered


def test_topk_matches_numpy_stable_argsort():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((2000, 64)).astype(np.float32).astype(np.float64)
    logits[::7, 3] = logits[::7, 11]          # plant exact ties
    idx, _ = O.route_topk(logits, 6)
    ref = np.argsort(-logits, axis=1, kind="stable")[:, :6]
    np.testing.assert_array_equal(idx, ref)


def test_gates_renormalised_softmax():
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((500, 16)) * 3
    idx, gate, probs = O.route_topk(logits, 4, want_probs=True)
    np.testing.assert_allclose(gate.sum(1), 1.0, rtol=0, atol=4e-16)
    np.testing.assert_allclose(probs, softmax(logits, axis=1), rtol=1e-14, atol=0)
    # closed form: renormalised top-k softmax == softmax over the selected logits
    sel = np.take_along_axis(logits, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(gate, softmax(sel, axis=1), rtol=1e-14, atol=0)
    # gates come out in descending order (same order as the logits)
    assert np.all(np.diff(gate, axis=1) <= 0)


def test_gates_k_equals_E_is_plain_softmax():
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((100, 8))
    idx, gate = O.route_topk(logits, 8)
    p = softmax(logits, axis=1)
    np.testing.assert_allclose(gate, np.take_along_axis(p, idx.astype(np.int64), 1),
                               rtol=1e-14, atol=0)


# ---------------------------------------------------------------------------- layout
def _check_layout(idx, E, S):
    N, k = idx.shape
    counts, offsets, sched, inv = O.layout(idx, E, S)
    flat = idx.ravel()
    assert counts.sum() == N * k
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    # slot order == stable sort of the flat choices by expert (library routine)
    order = np.argsort(flat, kind="stable")           # order[slot] = flat index n*k+j
    np.testing.assert_array_equal(inv.ravel()[order], np.arange(N * k))
    # bijection onto [0, T)
    assert np.array_equal(np.sort(inv.ravel()), np.arange(N * k))
    # same-expert slots are contiguous: slot s of expert e lies in [off[e], off[e+1])
    slot_expert = np.empty(N * k, dtype=np.int64)
    slot_expert[inv.ravel()] = flat
    for e in range(E):
        assert np.all(slot_expert[offsets[e]:offsets[e + 1]] == e)
    # sched rows decode to the token: shard * (N/S) + row, ascending inside an expert
    tok = sched[:, 0].astype(np.int64) * (N // S) + sched[:, 1]
    np.testing.assert_array_equal(tok[inv.ravel()], np.repeat(np.arange(N), k))
    for e in range(E):
        assert np.all(np.diff(tok[offsets[e]:offsets[e + 1]]) > 0)
    assert np.all((sched[:, 0] >= 0) & (sched[:, 0] < S))
    assert np.all((sched[:, 1] >= 0) & (sched[:, 1] < N // S))
    return counts, offsets, sched, inv


def _random_choices(rng, N, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)


@pytest.mark.parametrize("N,E,k,S", [(64, 8, 2, 2), (256, 16, 4, 8), (1000, 64, 6, 10),
                                     (48, 3, 3, 48), (32, 1, 1, 1), (96, 8, 8, 4)])
def test_layout_invariants(N, E, k, S):
    rng = np.random.default_rng(N + E + k)
    _check_layout(_random_choices(rng, N, E, k), E, S)


def test_layout_empty_and_hot_experts():
    rng = np.random.default_rng(11)
    N, E, k = 512, 32, 2
    idx = np.empty((N, k), dtype=np.int32)
    idx[:, 0] = 5                                   # every token picks expert 5 ...
    idx[:, 1] = rng.choice([7, 30], size=N)        # ... and one of two others
    counts, offsets, _, _ = _check_layout(idx, E, 4)
    assert counts[5] == N and counts[:5].sum() == 0 and counts[31] == 0


def test_layout_no_tokens():
    idx = np.zeros((0, 2), dtype=np.int32)
    counts, offsets, sched, inv = O.layout(idx, 4, 1)
    assert counts.sum() == 0 and np.all(offsets == 0) and sched.shape == (0, 2)


# ------------------------------------------------------------------------ expert FFN
def test_silu_closed_forms():
    u = np.array([0.0, 1.0, -1.0, 40.0, -40.0, 2.5])
    h = O.swiglu(u, np.ones_like(u))
    assert h[0] == 0.0
    assert abs(h[1] - math.e / (1 + math.e)) < 1e-15
    assert abs(h[2] - (-1 / (1 + math.e))) < 1e-15
    assert abs(h[3] - 40.0) < 1e-15 and abs(h[4]) < 1e-15
    np.testing.assert_allclose(h, torch.nn.functional.silu(torch.from_numpy(u)).numpy(),
                               rtol=1e-15, atol=1e-300)
    # the up projection multiplies element-wise
    v = np.array([2.0, -3.0, 0.5, 1.0, 7.0, 0.0])
    np.testing.assert_allclose(O.swiglu(u, v), h * v, rtol=1e-15, atol=0)


def _dense_ffn_torch(x, wgu, wd, cast):
    """Independent dense SwiGLU FFN with torch FP64 ops and the same rounding points."""
    x = torch.from_numpy(x)
    I = wgu.shape[0] // 2
    wg = torch.from_numpy(wgu[:I])
    wu = torch.from_numpy(wgu[I:])
    h = torch.nn.functional.silu(x @ wg.T) * (x @ wu.T)
    h = cast(h)
    return cast(h @ torch.from_numpy(wd).T).numpy()


@pytest.mark.parametrize("dtype,cast,tol", [
    ("f32", lambda t: t.float().double(), 1e-6),
    ("bf16", lambda t: t.bfloat16().double(), 1e-2),
])
def test_single_expert_top1_is_a_dense_ffn(dtype, cast, tol):
    w = synth.Workload("dense", N=48, H=64, I=96, E=1, k=1, S=4, dtype=dtype)
    inp = synth.make_inputs(w, device="cpu")
    res = O.forward(inp, w.E, w.k, w.S, w.dtype)
    assert np.all(res["idx"] == 0) and np.all(res["gate"] == 1.0)
    x = O._f64(inp["x"])
    wgu = O._f64(inp["w_gate_up"][0])
    wd = O._f64(inp["w_down"][0])
    ref = _dense_ffn_torch(x, wgu, wd, cast)
    # equal up to a last-place rounding flip where FP64 sums differ in order
    np.testing.assert_allclose(res["out"], ref, rtol=tol, atol=tol * np.abs(ref).max())
    frac_exact = np.mean(res["out"] == ref)
    assert frac_exact > 0.95


def test_single_expert_top1_mxfp8_is_dense_ffn_on_quantised_operands():
    w = synth.Workload("dense8", N=40, H=128, I=64, E=1, k=1, S=5, dtype="mxfp8")
    inp = synth.make_inputs(w, device="cpu")
    res = O.forward(inp, w.E, w.k, w.S, w.dtype)
    x = O.mxfp8_values(O._f64(inp["x"]))
    wgu = O.mxfp8_values(O._f64(inp["w_gate_up"][0]))
    wd = O.mxfp8_values(O._f64(inp["w_down"][0]))
    xt, wg, wu, wdt = (torch.from_numpy(a) for a in (x, wgu[:64], wgu[64:], wd))
    h = torch.nn.functional.silu(xt @ wg.T) * (xt @ wu.T)
    h = torch.from_numpy(O.mxfp8_values(h.numpy()))
    ref = (h @ wdt.T).bfloat16().double().numpy()
    np.testing.assert_allclose(res["out"], ref, rtol=1e-2, atol=1e-2 * np.abs(ref).max())


def test_identity_experts_closed_form():
    # expert e returns c_e * a: out[n] = (sum_j g[n,j] c_{e_j}) x[n]
    w = synth.Workload("ident", N=64, H=128, I=32, E=8, k=3, S=2, dtype="f32")
    inp = synth.make_inputs(w, device="cpu")
    c = np.linspace(0.5, 2.0, w.E)
    res = O.forward(inp, w.E, w.k, w.S, w.dtype, expert_fn=lambda e, a: c[e] * a)
    x = O._f64(inp["x"])
    coef = (res["gate"] * c[res["idx"]]).sum(1)
    np.testing.assert_allclose(res["out"], coef[:, None] * x, rtol=2e-7, atol=0)
    # all c_e = 1: the gates sum to one, so the layer returns x (after FP32 rounding)
    res1 = O.forward(inp, w.E, w.k, w.S, w.dtype, expert_fn=lambda e, a: a)
    np.testing.assert_array_equal(res1["out"], x)


def test_combine_constant_rows_closed_form():
    rng = np.random.default_rng(12)
    n, k, H = 20, 4, 8
    gate = rng.random((n, k))
    consts = rng.standard_normal(n * k)
    y = np.repeat(consts[:, None], H, axis=1)
    inv = rng.permutation(n * k).reshape(n, k).astype(np.int32)
    out = O.combine(y, inv, gate)
    expect = (gate * consts[inv]).sum(1)
    np.testing.assert_allclose(out, np.repeat(expect[:, None], H, 1), rtol=1e-15, atol=1e-15)
    # one-hot rows pick out single gates
    y = np.zeros((n * k, H))
    y[inv[:, 2], 0] = 1.0
    np.testing.assert_array_equal(O.combine(y, inv, gate)[:, 0], gate[:, 2])


def test_token_subset_equals_full_layer():
    w = synth.Workload("subset", N=64, H=64, I=64, E=8, k=2, S=2, dtype="bf16")
    inp = synth.make_inputs(w, device="cpu")
    full = O.forward(inp, w.E, w.k, w.S, w.dtype)
    toks = [0, 5, 17, 63]
    part = O.forward(inp, w.E, w.k, w.S, w.dtype, tokens=toks)
    np.testing.assert_array_equal(part["out"], full["out"][toks])


def test_skew_bias_concentrates_load():
    w = synth.Workload("skew", N=2048, H=64, I=32, E=64, k=4, S=4, dtype="bf16", skew=3.0)
    inp = synth.make_inputs(w, device="cpu", with_weights=False)
    lg = O.router_logits(inp["x"], inp["w_router"], inp["bias"])
    idx, _ = O.route_topk(lg, w.k)
    counts = np.bincount(idx.ravel(), minlength=w.E)
    assert counts.max() / counts.mean() > 8
    # the hottest expert is the rank-1 expert (bias 0, all others negative)
    assert inp["bias"].argmax().item() == counts.argmax()
