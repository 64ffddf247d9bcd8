"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Each mutant is a one-line source edit of the oracle (a dropped term, a wrong
sign, a wrong index or operand, a wrong comparison).  The mutated copy is
loaded as a separate module; the pins of test_oracle_pins run against it and at
least one must fail.  Nothing here touches the GPU or the product library.
"""
import importlib.util
import os
import sys
import types

import numpy as np
import pytest

import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "ttt_oracle.py")

MUTANTS = {
    "forward drops the residual": (
        'return h + a @ Wb["W2"].T, {"h": h', 'return a @ Wb["W2"].T, {"h": h'),
    "forward uses W1 transposed (square shapes hide it)": (
        'z = h @ Wb["W1"].T', 'z = h @ Wb["W1"][:, :h.shape[1]]'),
    "backward drops the residual path": (
        'dh = dout + dz @ Wb["W1"] if need_dh', 'dh = dz @ Wb["W1"] if need_dh'),
    "GELU derivative drops z*phi": (
        "return 0.5 * (1.0 + erf(z / SQRT2)) + z * INV_SQRT_2PI", "return 0.5 * (1.0 + erf(z / SQRT2)) + 0 * INV_SQRT_2PI"),
    "RMSNorm backward sign": (
        "(dy - xh * np.mean(xh * dy", "(dy + xh * np.mean(xh * dy"),
    "RMSNorm eps outside the sqrt": (
        "r = 1.0 / np.sqrt(np.mean(x * x, axis=-1) + eps)", "r = 1.0 / (np.sqrt(np.mean(x * x, axis=-1)) + eps)"),
    "chunk gradient is a sum, not a mean": (
        "    dlogits /= b\n", "    dlogits /= 1\n"),
    "CE picks the wrong target column": (
        "losses = lse - logits[np.arange(len(targets)), targets]",
        "losses = lse - logits[np.arange(len(targets)), (targets + 1) % logits.shape[1]]"),
    "losses scored after the update": (
        "    losses, grads = chunk_loss_and_grads(net, st.W, h_in, tgt, w)\n    s, norm = clip_scale(grads, clip)\n    st.W = sgd_step(st.W, grads, eta, s)\n",
        "    losses, grads = chunk_loss_and_grads(net, st.W, h_in, tgt, w)\n    s, norm = clip_scale(grads, clip)\n    st.W = sgd_step(st.W, grads, eta, s)\n    losses = token_losses(net, st.W, x_in, tgt)\n"),
    "targets not shifted by one": (
        "tokens[lo:lo + b], tokens[lo + 1:lo + b + 1],", "tokens[lo:lo + b], tokens[lo:lo + b],"),
    "clip scale inverted": (
        "return min(1.0, clip / (norm + CLIP_EPS)), norm", "return min(1.0, (norm + CLIP_EPS) / clip), norm"),
    "update sign": ("nb[k] = Wb[k] - (eta * s) * v", "nb[k] = Wb[k] + (eta * s) * v"),
    "Settlement tie rejects": ("accept = bool(A >= 0.0)", "accept = bool(A > 0.0)"),
    "Settlement A sign": (
        "A = heldout_loss(net, st.Wc, q) - heldout_loss(net, st.W, q)",
        "A = heldout_loss(net, st.W, q) - heldout_loss(net, st.Wc, q)"),
    "SwiGLU up-gradient uses g": ("du = da * silu(cache[\"g\"])", "du = da * cache[\"g\"]"),
    "SwiGLU gate gradient drops silu'": (
        'dg = da * cache["u"] * silu_grad(cache["g"])', 'dg = da * cache["u"] * silu(cache["g"])'),
    "masked chunk mean divides by the chunk length": (
        "return m / max(1.0, float(m.sum()))", "return m / len(m)"),
    "mask ignored in the update": (
        "w = None if mask is None else mask_weights(mask)", "w = None"),
    "reset one chunk late": (
        "if st.reset_every and st.chunks_done % st.reset_every == 0:",
        "if st.reset_every and (st.chunks_done - 1) % st.reset_every == 0 and st.chunks_done > 1:"),
    "reset keeps the current weights": (
        "st.W = copy.deepcopy(net.fast0)       # R9", "st.W = copy.deepcopy(st.W)       # R9"),
    "static MLP skipped in the backward": (
        "if net.static is not None and l > 0:", "if False:"),
    "static MLP after the fast one": (
        "            h, _ = block_forward(net.kind, net.static[l], h)      # R10\n        h, _ = block_forward(net.kind, Wb, h)\n",
        "            pass\n        h, _ = block_forward(net.kind, Wb, h)\n"
        "        if net.static is not None:\n            h, _ = block_forward(net.kind, net.static[l], h)\n"),
    "attention window one too wide": ("return (s <= t) & (s > t - k)", "return (s <= t) & (s >= t - k)"),
    "attention anti-causal": ("return (s <= t) & (s > t - k)", "return (s >= t) & (s > t - k)"),
    "attention without 1/sqrt(d_h)": ("Q[:, c] @ K[:, c].T / np.sqrt(dh)", "Q[:, c] @ K[:, c].T"),
    "attention drops its residual": (
        "h = h + attention(net.attn[p], h, net.heads, net.window)", "h = attention(net.attn[p], h, net.heads, net.window)"),
    "attention heads read the first head's columns": ("c = slice(i * dh, (i + 1) * dh)", "c = slice(0, dh)"),
    "decoded input attends to itself only": (
        "st.h_last = frozen_prefix(net, np.array(st.hist[-reach:]))[-1]",
        "st.h_last = frozen_prefix(net, np.array(st.hist[-1:]))[-1]"),
    "decoded chunk recomputes its prefix rows without context": (
        "h_in=np.array(st.pend_h) if attn else None)", "h_in=None)"),
    "weight error without its square root": ("return np.sqrt(num / den)", "return num / den"),
    "weight error normalised by the first argument": (
        "den += float(np.sum(np.asarray(b[k], np.float64) ** 2))",
        "den += float(np.sum(np.asarray(a[k], np.float64) ** 2))"),
    "p_next with the initial weights": (
        "p_next = softmax_next(net, st.W, st.x_last, rows(T, T + 1))",
        "p_next = softmax_next(net, net.fast0, st.x_last, rows(T, T + 1))"),
}

PINS = [
    ("test_fast_weight_gradients_match_central_differences", ("gelu", 3)),
    ("test_fast_weight_gradients_match_central_differences", ("swiglu", 3)),
    ("test_gelu_closed_form_values", ()),
    ("test_rmsnorm_unit_rms_and_scale_invariance", ()),
    ("test_rmsnorm_backward_finite_differences", ()),
    ("test_cross_entropy_identities", ()),
    ("test_b1_is_the_per_token_update_of_eq2", ()),
    ("test_eta0_gives_the_static_ttt_naive_loss_of_eq4", ()),
    ("test_single_chunk_b_equals_T", ()),
    ("test_prequential_losses_use_the_previous_chunks_weights_eq3_eq6", ()),
    ("test_clip_bounds_the_step", ()),
    ("test_p_next_is_f_of_last_token_with_final_weights", ()),
    ("test_settlement_commits_a_descent_step", ()),
    ("test_settlement_rejects_an_ascent_step_and_reverts_exactly", ()),
    ("test_settlement_tie_commits", ()),
    ("test_settlement_two_token_case_by_hand", ()),
    ("test_forward_by_hand_nonsquare", ()),
    ("test_decoding_a_full_chunk_equals_a_longer_prefill", ()),
    ("test_reset_every_chunk_scores_like_eq4_and_ends_at_w0", ()),
    ("test_static_mlp_gradients_match_central_differences", ()),
    ("test_attention_by_hand_one_and_two_heads", ()),
    ("test_attention_with_zero_queries_is_the_window_mean", ()),
    ("test_attention_sees_exactly_its_receptive_field", ()),
    ("test_decoding_with_attention_equals_a_longer_prefill", (8,)),
    ("test_decoding_with_attention_equals_a_longer_prefill", (7,)),
    ("test_static_mlp_runs_before_the_fast_one", ()),
    ("test_reset_splits_the_stream_into_independent_runs", ()),
    ("test_reset_counts_decoded_chunks_too", ()),
    ("test_all_ones_mask_is_the_unmasked_method", ()),
    ("test_all_zeros_mask_never_updates_and_scores_like_eq4", ()),
    ("test_single_unmasked_target_is_that_tokens_own_gradient", ()),
    ("test_masked_chunk_gradient_matches_central_differences", ()),
    ("test_weights_rel_frobenius_on_a_hand_computed_pair", ()),
]


def _load_mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("ttt_oracle_mutant")
    mod.__dict__["__name__"] = "ttt_oracle_mutant"
    sys.modules["ttt_oracle_mutant"] = mod
    exec(compile(src.replace(old, new), "ttt_oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name", list(MUTANTS))
def test_every_planted_mistake_fails_a_pin(name, monkeypatch):
    mod = _load_mutant(*MUTANTS[name])
    monkeypatch.setattr(P, "O", mod)
    caught = []
    for pin, args in PINS:
        try:
            with np.errstate(all="ignore"):
                getattr(P, pin)(*args)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught.append(pin)
    assert caught, f"no pin caught mutant '{name}'"
