"""The pins catch plausible oracle mistakes.

Each case plants one mistake in the oracle (on the CPU, by swapping one oracle
function for a wrong variant) and checks that at least one pin test then fails.
"""
import numpy as np
import pytest

import oracle as O
import test_oracle_backward as B
import test_oracle_backward_axes as X
import test_oracle_formats as F
import test_oracle_layer as L
import test_oracle_nvfp4 as N


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def _topk_ties_to_higher_index(orig):
    def f(logits, k, want_probs=False):
        rev = np.ascontiguousarray(logits[:, ::-1])
        res = orig(rev, k, want_probs)
        idx = (logits.shape[1] - 1 - res[0]).astype(np.int32)
        return (idx,) + tuple(res[1:])
    return f


def _gates_not_renormalised(orig):
    def f(logits, k, want_probs=False):
        idx, gate, probs = orig(logits, k, True)
        gate = np.take_along_axis(probs, idx.astype(np.int64), 1)
        return (idx, gate, probs) if want_probs else (idx, gate)
    return f


def _layout_descending_tokens(orig):
    def f(idx, E, S):
        counts, offsets, sched, inv = orig(idx, E, S)
        T = inv.size
        slot_expert = np.empty(T, dtype=np.int64)
        slot_expert[inv.ravel()] = idx.ravel()
        new = inv.copy().ravel()
        for e in range(E):       # reverse the order inside each expert segment
            a, b = offsets[e], offsets[e + 1]
            new = np.where((inv.ravel() >= a) & (inv.ravel() < b), a + b - 1 - inv.ravel(), new)
        sched2 = np.empty_like(sched)
        sched2[new] = sched[inv.ravel()]
        return counts, offsets, sched2, new.reshape(inv.shape).astype(np.int32)
    return f


def _swiglu_swapped(orig):
    return lambda u, v: orig(v, u)


def _combine_drops_last_choice(orig):
    def f(y, inv, gate):
        g = gate.copy()
        g[:, -1] = 0.0
        return orig(y, inv, g)
    return f


def _quantize_wrong_emax(orig):
    def f(a):
        codes, scales = orig(a)          # scale one binade too large (emax 7 for 8)
        return codes, scales + 1
    return f


def _round_bf16_truncates(orig):
    def f(a):
        a = np.ascontiguousarray(a, dtype=np.float64)
        bits = a.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
        return bits.view(np.float32).astype(np.float64)
    return f


def _ffn_transposed_down(orig):
    def f(a, wg, wu, wd, dtype):
        return orig(a, wg, wu, wd.T.copy() if wd.shape[0] == wd.shape[1] else wd[::-1].copy(), dtype)
    return f


def _swiglu_backward_swapped(orig):
    def f(u, v, dh):
        du, dv = orig(u, v, dh)
        return dv, du
    return f


def _silu_derivative_drops_second_term(orig):
    def f(u, v, dh):
        du, dv = orig(u, v, dh)
        s = 1.0 / (1.0 + np.exp(-u))
        return dh * v * s, dv
    return f


def _gate_backward_drops_mean(orig):
    return lambda gate, dgate: np.asarray(gate) * np.asarray(dgate)


def _nvfp4_nibbles_swapped(orig):
    def f(a):
        q, s, st = orig(a)
        return ((q >> 4) | (q << 4)).astype(np.uint8), s, st
    return f


def _nvfp4_scale_without_tensor_scale(orig):
    def f(a):
        q, s, st = orig(a)              # block scales taken on amax/6 alone, st dropped
        e4 = O.lib().orc_e4m3_encode
        amax = np.abs(np.asarray(a, dtype=np.float64)).reshape(a.shape[0], -1, 16).max(axis=2)
        s2 = np.vectorize(lambda t: e4(float(np.float32(t))))(amax / 6.0).astype(np.uint8)
        return q, s2, 1.0
    return f


def _e2m1_ties_away(orig):
    def f(v):
        v = np.asarray(v, dtype=np.float64)
        a = np.minimum(np.abs(v), 6.0)
        mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
        d = np.abs(a[..., None] - mags)
        code = (d.shape[-1] - 1 - np.argmin(d[..., ::-1], axis=-1)).astype(np.uint8)
        return code | np.where(np.signbit(v), 8, 0).astype(np.uint8)
    return f


def _dgrad_weights_along_forward_axis(orig):
    def f(w_gate_up_e, w_down_e, dtype):
        if dtype != "mxfp8":
            return orig(w_gate_up_e, w_down_e, dtype)
        return O.expert_operands(w_gate_up_e, w_down_e, dtype)     # along H and I
    return f


def _dgrad_operand_along_slots_for(K):
    """Quantise the dgrad operand whose reduction length is K down the slots
    instead of along K (the pins use K = 64 for dy and K = 32 for du, dv)."""
    def mutant(orig):
        def f(m, fmt):
            if fmt == "mxfp8" and m.shape[1] == K:
                return O.round_along_slots(m, fmt)
            return orig(m, fmt)
        return f
    return mutant


def _bwd_format(pos, fmt):
    """Keep one dgrad operand of the MXFP8 layer in BF16 instead of MXFP8."""
    def mutant(orig):
        row = list(orig["mxfp8"])
        row[pos] = fmt
        return {**orig, "mxfp8": tuple(row)}
    return mutant


def _wgrad_operands_along_rows(orig):
    return lambda m, fmt: O.round_to(m, fmt)


def _wgrad_blocks_end_at_the_segment(orig):
    def f(m, fmt):
        if fmt != "mxfp8":
            return orig(m, fmt)
        pad = (-m.shape[0]) % 32          # the partial block first instead of last
        mp = np.vstack([np.zeros((pad, m.shape[1])), m]) if pad else m
        return np.ascontiguousarray(O.mxfp8_values(np.ascontiguousarray(mp.T)).T[pad:])
    return f


def _autograd_pin():
    B.test_matches_torch_autograd(16, 32, 24, 8, 2, True)


def _fd_pin():
    B.test_directional_derivatives_match_central_differences(8, 32, 16, 6, 2)


CASES = [
    ("route_topk", _topk_ties_to_higher_index, [L.test_topk_matches_numpy_stable_argsort]),
    ("route_topk", _gates_not_renormalised, [L.test_gates_renormalised_softmax]),
    ("layout", _layout_descending_tokens, [lambda: L.test_layout_invariants(64, 8, 2, 2)]),
    ("swiglu", _swiglu_swapped, [L.test_silu_closed_forms]),
    ("combine", _combine_drops_last_choice, [L.test_combine_constant_rows_closed_form]),
    ("quantize_mxfp8", _quantize_wrong_emax, [F.test_mxfp8_scale_for_power_of_two_amax]),
    ("round_bf16", _round_bf16_truncates, [F.test_bf16_rounding_matches_torch_on_ties_and_near_ties]),
    ("expert_ffn", _ffn_transposed_down,
     [lambda: L.test_single_expert_top1_is_a_dense_ffn("bf16", lambda t: t.bfloat16().double(), 1e-2)]),
    ("swiglu_backward", _swiglu_backward_swapped, [_fd_pin]),
    ("swiglu_backward", _silu_derivative_drops_second_term, [_autograd_pin]),
    ("gate_backward", _gate_backward_drops_mean, [_fd_pin]),
    ("gate_backward", _gate_backward_drops_mean, [lambda: B.test_router_shift_invariances("f64")]),
    ("quantize_nvfp4", _nvfp4_nibbles_swapped, [lambda: N.test_nvfp4_reproduces_exactly_representable_blocks(0)]),
    ("quantize_nvfp4", _nvfp4_scale_without_tensor_scale,
     [lambda: N.test_nvfp4_reproduces_exactly_representable_blocks(5)]),
    ("e2m1_encode", _e2m1_ties_away, [N.test_e2m1_encode_is_round_to_nearest_even_with_saturation]),
    ("expert_operands_dgrad", _dgrad_weights_along_forward_axis,
     [X.test_dgrad_weights_are_quantised_down_their_reduction_axis]),
    ("round_dgrad_operand", _dgrad_operand_along_slots_for(64),
     [lambda: X.test_dgrad_dy_is_quantised_along_H_per_slot("random")]),
    ("round_dgrad_operand", _dgrad_operand_along_slots_for(64),
     [lambda: X.test_dgrad_dy_is_quantised_along_H_per_slot("hand")]),
    ("round_dgrad_operand", _dgrad_operand_along_slots_for(32),
     [lambda: X.test_dgrad_du_dv_are_quantised_along_I_per_slot("random")]),
    ("round_dgrad_operand", _dgrad_operand_along_slots_for(32),
     [lambda: X.test_dgrad_du_dv_are_quantised_along_I_per_slot("hand")]),
    ("BWD_FORMATS", _bwd_format(0, "bf16"), [lambda: X.test_dgrad_dy_is_quantised_along_H_per_slot("hand")]),
    ("BWD_FORMATS", _bwd_format(2, "bf16"),
     [lambda: X.test_dgrad_du_dv_are_quantised_along_I_per_slot("hand")]),
    ("round_along_slots", _wgrad_operands_along_rows,
     [lambda: X.test_wgrad_operands_are_quantised_along_the_slots(64, "random")]),
    ("round_along_slots", _wgrad_operands_along_rows,
     [lambda: X.test_wgrad_operands_are_quantised_along_the_slots(64, "hand")]),
    ("round_along_slots", _wgrad_blocks_end_at_the_segment,
     [lambda: X.test_wgrad_operands_are_quantised_along_the_slots(40, "random"),
      B.test_round_along_slots_blocks_start_at_the_segment]),
]


@pytest.mark.parametrize("name,mutant,pins", CASES,
                         ids=[f"{i}-{c[0]}-{c[1].__name__.strip('_')}" for i, c in enumerate(CASES)])
def test_planted_mistake_is_caught(monkeypatch, name, mutant, pins):
    monkeypatch.setattr(O, name, mutant(getattr(O, name)))
    assert any(_fails(p) for p in pins), f"no pin caught the planted mistake in {name}"
