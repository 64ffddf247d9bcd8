"""Pins of the float64 oracle against facts the pages and the mathematics fix.

None of these re-types the oracle's formulas: each checks a closed form, a
special case that reduces to another equation on the pages, finite
differences, or an invariant, chosen so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them.
"""
import copy
import math

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import ttt_oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def rand_net(kind="gelu", d=8, f=16, V=16, n_prefix=1, n_fast=2, fast_mats=None,
             std=0.5, seed=0, eps=1e-6):
    rng = np.random.default_rng(seed)
    mats = {"gelu": {"W1": (f, d), "W2": (d, f)},
            "swiglu": {"Wg": (f, d), "Wu": (f, d), "Wd": (d, f)}}[kind]
    blk = lambda: {k: rng.normal(0, std, s) for k, s in mats.items()}
    w = {"E": rng.normal(0, 1.0, (V, d)), "U": rng.normal(0, std, (V, d)),
         "prefix": [blk() for _ in range(n_prefix)], "fast": [blk() for _ in range(n_fast)]}
    if fast_mats is None:
        fast_mats = tuple(mats)
    return O.Net.from_weights(w, kind, fast_mats, eps)


def rand_tokens(V, B, T, seed=1):
    rng = np.random.default_rng(seed)
    t = rng.integers(0, V, size=(B, T + 1))
    t[:, 0] = 0
    return t


# ------------------------------------------------------------------ pointwise
def test_gelu_closed_form_values():
    # Phi(1) and Phi(-1) from the standard normal table
    assert O.gelu(np.array(0.0)) == 0.0
    assert abs(O.gelu(np.array(1.0)) - 0.8413447460685429) < 1e-15
    assert abs(O.gelu(np.array(-1.0)) + 0.15865525393145707) < 1e-15
    x = np.linspace(-6, 6, 101)
    np.testing.assert_allclose(O.gelu(x), x * stats.norm.cdf(x), rtol=1e-13, atol=1e-15)
    assert abs(O.gelu_grad(np.array(0.0)) - 0.5) < 1e-15
    h = 1e-6
    np.testing.assert_allclose(O.gelu_grad(x), (O.gelu(x + h) - O.gelu(x - h)) / (2 * h),
                               rtol=1e-8, atol=1e-9)


def test_silu_closed_form_values():
    assert O.silu(np.array(0.0)) == 0.0
    x = np.linspace(-8, 8, 81)
    np.testing.assert_allclose(O.silu(x), x * stats.logistic.cdf(x), rtol=1e-13, atol=1e-15)
    h = 1e-6
    np.testing.assert_allclose(O.silu_grad(x), (O.silu(x + h) - O.silu(x - h)) / (2 * h),
                               rtol=1e-8, atol=1e-9)


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 2.0, (5, 7))
    y, r = O.rmsnorm(x, 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-14)
    y2, _ = O.rmsnorm(3.5 * x, 0.0)
    np.testing.assert_allclose(y2, y, rtol=1e-14)
    # with eps the mean square is ms / (ms + eps)
    eps = 0.3
    ye, _ = O.rmsnorm(x, eps)
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.mean(ye * ye, axis=-1), ms / (ms + eps), rtol=1e-14)


def test_rmsnorm_backward_finite_differences():
    rng = np.random.default_rng(4)
    x = rng.normal(0, 1.0, (3, 6))
    dy = rng.normal(0, 1.0, (3, 6))
    eps = 0.01
    y, r = O.rmsnorm(x, eps)
    dx = O.rmsnorm_backward(x, r, dy)
    fd = np.zeros_like(x)
    h = 1e-6
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            fd[i, j] = (np.sum(O.rmsnorm(xp, eps)[0] * dy) - np.sum(O.rmsnorm(xm, eps)[0] * dy)) / (2 * h)
    np.testing.assert_allclose(dx, fd, rtol=1e-7, atol=1e-9)


def test_cross_entropy_identities():
    rng = np.random.default_rng(5)
    V = 11
    logits = rng.normal(0, 3.0, (6, V))
    tgt = rng.integers(0, V, 6)
    losses, p = O.cross_entropy(logits, tgt)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(losses, -np.log(p[np.arange(6), tgt]), rtol=1e-12)
    # a shift of all logits leaves the loss unchanged; uniform logits give ln V
    np.testing.assert_allclose(O.cross_entropy(logits + 100.0, tgt)[0], losses, rtol=1e-12)
    np.testing.assert_allclose(O.cross_entropy(np.zeros((2, V)), np.array([0, 3]))[0],
                               np.log(V), rtol=1e-15)
    # the loss gradient (softmax - onehot) sums to zero on every row
    dl = p.copy()
    dl[np.arange(6), tgt] -= 1
    np.testing.assert_allclose(dl.sum(-1), 0.0, atol=1e-15)
    # and matches finite differences of the loss
    h = 1e-6
    for j in range(V):
        lp, lm = logits.copy(), logits.copy()
        lp[:, j] += h
        lm[:, j] -= h
        fd = (O.cross_entropy(lp, tgt)[0] - O.cross_entropy(lm, tgt)[0]) / (2 * h)
        np.testing.assert_allclose(dl[:, j], fd, rtol=1e-6, atol=1e-9)


# ------------------------------------------------------------------ gradients
def _chunk_mean_loss(net, fast, x_in, tgt):
    return float(np.mean(O.token_losses(net, fast, x_in, tgt)))


@pytest.mark.parametrize("kind", ["gelu", "swiglu"])
@pytest.mark.parametrize("b", [1, 3])
def test_fast_weight_gradients_match_central_differences(kind, b):
    """eq. (5)'s gradient of the chunk mean, every fast matrix, rel <= 1e-6."""
    net = rand_net(kind, d=8, f=16, V=16, n_prefix=1, n_fast=2, seed=10 + b)
    tok = rand_tokens(16, 1, b, seed=20 + b)[0]
    x_in, tgt = tok[:-1], tok[1:]
    fast = copy.deepcopy(net.fast0)
    _, grads = O.chunk_loss_and_grads(net, fast, O.frozen_prefix(net, x_in), tgt)
    h = 1e-5
    for l, Wb in enumerate(fast):
        for k in net.fast_mats:
            fd = np.zeros_like(Wb[k])
            for idx in np.ndindex(Wb[k].shape):
                orig = Wb[k][idx]
                Wb[k][idx] = orig + h
                lp = _chunk_mean_loss(net, fast, x_in, tgt)
                Wb[k][idx] = orig - h
                lm = _chunk_mean_loss(net, fast, x_in, tgt)
                Wb[k][idx] = orig
                fd[idx] = (lp - lm) / (2 * h)
            an = grads[l][k]
            rel = np.linalg.norm(fd - an) / np.linalg.norm(an)
            assert rel <= 1e-6, (kind, b, l, k, rel)
            assert np.max(np.abs(fd - an)) <= 1e-6 * np.max(np.abs(an)) + 1e-12


def test_partial_fast_set_in_place_down_projection():
    """In-Place TTT: only the down projection is fast; gate/up never move."""
    net = rand_net("swiglu", n_fast=1, fast_mats=("Wd",), std=0.3, seed=7)
    tok = rand_tokens(16, 1, 12, seed=8)
    out = O.prefill(net, 0.1, 0.0, 4, tok)
    W = out["W"][0][0]
    np.testing.assert_array_equal(W["Wg"], net.fast0[0]["Wg"])
    np.testing.assert_array_equal(W["Wu"], net.fast0[0]["Wu"])
    assert np.max(np.abs(W["Wd"] - net.fast0[0]["Wd"])) > 1e-6


# ------------------------------------------------------------------ the loop
def test_b1_is_the_per_token_update_of_eq2():
    """With b = 1 the chunked loop is W_t = W_{t-1} - eta grad l_t(W_{t-1})."""
    net = rand_net("gelu", n_prefix=0, n_fast=1, std=0.3, seed=30)
    T, eta = 9, 0.2
    tok = rand_tokens(16, 1, T, seed=31)[0]
    out = O.prefill(net, eta, 0.0, 1, tok[None])
    W = copy.deepcopy(net.fast0)
    ref = np.zeros(T)
    for t in range(1, T + 1):
        x_prev, x_t = tok[t - 1:t], tok[t:t + 1]
        l, g = O.chunk_loss_and_grads(net, W, O.frozen_prefix(net, x_prev), x_t)
        ref[t - 1] = l[0]
        W = [{k: Wb[k] - eta * g[i].get(k, 0.0) for k in Wb} for i, Wb in enumerate(W)]
    np.testing.assert_allclose(out["losses"][0], ref, rtol=0, atol=1e-13)
    assert O.weights_rel_frobenius(out["W"][0], W, net.fast_mats) < 1e-14


def test_eta0_gives_the_static_ttt_naive_loss_of_eq4():
    net = rand_net("gelu", seed=40)
    tok = rand_tokens(16, 2, 12, seed=41)
    out = O.prefill(net, 0.0, 1.0, 4, tok)
    for s in range(2):
        np.testing.assert_allclose(out["losses"][s], O.static_losses(net, tok[s]),
                                   rtol=0, atol=1e-13)
        assert O.weights_rel_frobenius(out["W"][s], net.fast0, net.fast_mats) == 0.0


def test_single_chunk_b_equals_T():
    """b = T: every loss uses W_0 and W_T = W_0 - eta s mean-gradient (eq. (6))."""
    net = rand_net("gelu", seed=50)
    T, eta, c = 8, 0.3, 0.05
    tok = rand_tokens(16, 1, T, seed=51)
    out = O.prefill(net, eta, c, T, tok)
    np.testing.assert_allclose(out["losses"][0], O.static_losses(net, tok[0]), atol=1e-13)
    _, g = O.chunk_loss_and_grads(net, net.fast0, O.frozen_prefix(net, tok[0, :-1]), tok[0, 1:])
    norm = math.sqrt(sum(float(np.sum(v * v)) for gb in g for v in gb.values()))
    s = min(1.0, c / (norm + 1e-6))
    for l, Wb in enumerate(out["W"][0]):
        for k in net.fast_mats:
            np.testing.assert_allclose(Wb[k], net.fast0[l][k] - eta * s * g[l][k], atol=1e-14)


def test_prequential_losses_use_the_previous_chunks_weights_eq3_eq6():
    net = rand_net("gelu", seed=60)
    b, T, eta = 3, 12, 0.5
    tok = rand_tokens(16, 1, T, seed=61)
    out = O.prefill(net, eta, 0.0, b, tok, snapshots=True)
    snaps = out["snapshots"][0]
    assert len(snaps) == T // b + 1
    L_ref = 0.0
    for i in range(1, T // b + 1):
        sl = slice((i - 1) * b, i * b)
        l_prev = O.token_losses(net, snaps[i - 1], tok[0, (i - 1) * b:i * b], tok[0, (i - 1) * b + 1:i * b + 1])
        l_next = O.token_losses(net, snaps[i], tok[0, (i - 1) * b:i * b], tok[0, (i - 1) * b + 1:i * b + 1])
        np.testing.assert_allclose(out["losses"][0, sl], l_prev, atol=1e-13)
        assert np.max(np.abs(out["losses"][0, sl] - l_next)) > 1e-6
        L_ref += l_prev.sum()
    assert abs(out["losses"][0].mean() - L_ref / T) < 1e-13


def test_zero_head_gives_ln_V_and_no_update():
    net = rand_net("gelu", seed=70)
    net.U[:] = 0.0
    tok = rand_tokens(16, 1, 8, seed=71)
    out = O.prefill(net, 1.0, 0.0, 4, tok)
    np.testing.assert_allclose(out["losses"][0], np.log(16), rtol=1e-15)
    assert O.weights_rel_frobenius(out["W"][0], net.fast0, net.fast_mats) == 0.0
    np.testing.assert_allclose(out["p_next"][0], 1.0 / 16, rtol=1e-15)


def test_clip_bounds_the_step():
    net = rand_net("gelu", seed=80)
    tok = rand_tokens(16, 1, 4, seed=81)
    _, g = O.chunk_loss_and_grads(net, net.fast0, O.frozen_prefix(net, tok[0, :-1]), tok[0, 1:])
    s, norm = O.clip_scale(g, 1e-3)
    assert norm > 1e-3 and abs(s * norm - 1e-3) < 1e-9 and s * norm <= 1e-3
    s2, _ = O.clip_scale(g, 10 * norm)
    assert s2 == 1.0
    s3, _ = O.clip_scale(g, 0.0)
    assert s3 == 1.0
    out = O.prefill(net, 1.0, 1e-3, 4, tok)
    step = math.sqrt(sum(float(np.sum((out["W"][0][l][k] - net.fast0[l][k]) ** 2))
                         for l in range(2) for k in net.fast_mats))
    assert abs(step - 1e-3) < 1e-9


def test_batch_sequences_are_independent():
    net = rand_net("gelu", seed=90)
    tok = rand_tokens(16, 3, 12, seed=91)
    out = O.prefill(net, 0.4, 0.5, 4, tok)
    for s in range(3):
        one = O.prefill(net, 0.4, 0.5, 4, tok[s:s + 1])
        np.testing.assert_array_equal(one["losses"][0], out["losses"][s])
        np.testing.assert_array_equal(one["p_next"][0], out["p_next"][s])


def test_p_next_is_f_of_last_token_with_final_weights():
    net = rand_net("gelu", seed=95)
    tok = rand_tokens(16, 1, 8, seed=96)
    out = O.prefill(net, 0.4, 0.0, 4, tok)
    logits = O.forward_logits(net, out["W"][0], O.frozen_prefix(net, tok[0, -1:]))
    p = np.exp(logits[0] - logits[0].max())
    np.testing.assert_allclose(out["p_next"][0], p / p.sum(), rtol=1e-13)


# ------------------------------------------------------------------ decoding
def test_decoding_a_full_chunk_equals_a_longer_prefill():
    net = rand_net("gelu", seed=100)
    b, T, extra, eta, c = 4, 8, 8, 0.3, 0.7
    tok = rand_tokens(16, 1, T + extra, seed=101)
    long = O.prefill(net, eta, c, b, tok)
    short = O.prefill(net, eta, c, b, tok[:, :T + 1])
    st = short["states"][0]
    dec_losses = []
    for t in range(T + 1, T + extra + 1):
        l, p = O.decode_step(net, st, tok[0, t], eta, c, b)
        dec_losses.append(l)
    np.testing.assert_allclose(dec_losses, long["losses"][0, T:], atol=1e-13)
    np.testing.assert_allclose(p, long["p_next"][0], atol=1e-14)
    assert O.weights_rel_frobenius(st.W, long["W"][0], net.fast_mats) < 1e-14


def test_ragged_prefill_is_completed_by_decoding():
    """T mod b != 0: the tail waits in the pending buffer (3.2 Decoding)."""
    net = rand_net("gelu", seed=110)
    b, eta = 4, 0.3
    tok = rand_tokens(16, 1, 8, seed=111)
    full = O.prefill(net, eta, 0.0, b, tok)
    part = O.prefill(net, eta, 0.0, b, tok[:, :7])          # T = 6: one chunk + 2 pending
    np.testing.assert_allclose(part["losses"][0], full["losses"][0, :6], atol=1e-13)
    st = part["states"][0]
    assert len(st.pend_in) == 2
    for t in (7, 8):
        O.decode_step(net, st, tok[0, t], eta, 0.0, b)
    assert O.weights_rel_frobenius(st.W, full["W"][0], net.fast_mats) < 1e-14


# ------------------------------------------------------------------ Settlement
def _settle_case(eta, seed=120):
    net = rand_net("gelu", seed=seed)
    b = 6
    tok = rand_tokens(16, 1, b, seed=seed + 1)
    q = tok[:, None, :].transpose(1, 0, 2)       # held-out chunk = the chunk itself
    out = O.prefill(net, eta, 0.0, b, tok, settle_every=1, settle_q=q)
    return net, out


def test_settlement_commits_a_descent_step():
    net, out = _settle_case(1e-3)
    assert out["A"][0, 0] > 0 and out["accept"][0, 0]
    assert O.weights_rel_frobenius(out["W"][0], net.fast0, net.fast_mats) > 0


def test_settlement_rejects_an_ascent_step_and_reverts_exactly():
    net, out = _settle_case(-1e-3)
    assert out["A"][0, 0] < 0 and not out["accept"][0, 0]
    for l in range(2):
        for k in net.fast_mats:
            np.testing.assert_array_equal(out["W"][0][l][k], net.fast0[l][k])


def test_settlement_tie_commits():
    # delta = 0 (eta = 0) gives A = 0 exactly, and A >= 0 commits
    net = rand_net("gelu", seed=130)
    tok = rand_tokens(16, 2, 8, seed=131)
    q = rand_tokens(16, 4, 5, seed=132).reshape(2, 2, 6)
    out = O.prefill(net, 0.0, 1.0, 2, tok, settle_every=2, settle_q=q)
    assert np.all(out["A"] == 0.0) and np.all(out["accept"])


def test_settlement_two_token_case_by_hand():
    """V = 2, d = 2, one GELU fast block with f = 1, U = I, eps = 0.

    Committed W1 = 0 gives a = GELU(0) = 0, so h = E[q0] = (1, 0), y = (sqrt2, 0)
    and L(q, W_c) = ln(e^sqrt2 + 1) - 0 for target q1 = 1.  The candidate sets
    W1 = (c, 0): z = c, h = (1, GELU(c)) with W2 = (0, 1)^T, y = h / rms(h).
    """
    c = 1.3
    gel = c * 0.5 * (1 + math.erf(c / math.sqrt(2)))
    rms = math.sqrt((1 + gel * gel) / 2)
    y = (1 / rms, gel / rms)
    L_cand = math.log(math.exp(y[0]) + math.exp(y[1])) - y[1]
    L_comm = math.log(math.exp(math.sqrt(2)) + 1.0)
    w = {"E": np.array([[1.0, 0.0], [0.0, 1.0]]), "U": np.eye(2), "prefix": [],
         "fast": [{"W1": np.zeros((1, 2)), "W2": np.array([[0.0], [1.0]])}]}
    net = O.Net.from_weights(w, "gelu", ("W1", "W2"), 0.0)
    st = O.SeqState(W=copy.deepcopy(net.fast0), Wc=copy.deepcopy(net.fast0), x_last=0)
    st.W[0]["W1"] = np.array([[c, 0.0]])
    A, acc = O.settle(net, st, np.array([0, 1]))
    assert abs(A - (L_comm - L_cand)) < 1e-14
    assert A > 0 and acc
    # the reverse candidate (back to W1 = 0 from committed W1 = (c, 0)) is rejected
    st2 = O.SeqState(W=copy.deepcopy(net.fast0), Wc=copy.deepcopy(net.fast0), x_last=0)
    st2.Wc[0]["W1"] = np.array([[c, 0.0]])
    A2, acc2 = O.settle(net, st2, np.array([0, 1]))
    assert abs(A2 + (L_comm - L_cand)) < 1e-14 and not acc2
    np.testing.assert_array_equal(st2.W[0]["W1"], np.array([[c, 0.0]]))


# ------------------------------------------------------------------ a hand-built forward
def test_forward_by_hand_nonsquare():
    """d = 2, f = 3, V = 3; W1 picks h_0 into every hidden unit (so a transposed
    W1 or W2 changes the answer), W2 sums the hidden units into h_1."""
    E = np.array([[2.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    W1 = np.array([[1.0, 0.0], [0.5, 0.0], [-1.0, 0.0]])
    W2 = np.array([[0.0, 0.0, 0.0], [1.0, 1.0, 1.0]])
    U = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, -1.0]])
    net = O.Net.from_weights({"E": E, "U": U, "prefix": [], "fast": [{"W1": W1, "W2": W2}]},
                             "gelu", ("W1", "W2"), 0.0)
    G = lambda z: z * 0.5 * (1 + math.erf(z / math.sqrt(2)))
    # token 0: h = (2, 0); z = (2, 1, -2); h1 = 0 + G(2) + G(1) + G(-2)
    h = np.array([2.0, G(2.0) + G(1.0) + G(-2.0)])
    y = h / math.sqrt(np.mean(h * h))
    logits = np.array([y[0], y[1], y[0] - y[1]])
    lse = math.log(np.sum(np.exp(logits)))
    got = O.token_losses(net, net.fast0, np.array([0, 0, 0]), np.array([0, 1, 2]))
    np.testing.assert_allclose(got, lse - logits, rtol=1e-14)


# ------------------------------------------------------------------ Source Masking (reading R8)
def test_all_ones_mask_is_the_unmasked_method():
    net = rand_net("gelu", seed=80)
    tok = rand_tokens(16, 2, 13, seed=81)
    a = O.prefill(net, 0.2, 0.5, 4, tok)
    b = O.prefill(net, 0.2, 0.5, 4, tok, loss_mask=np.ones((2, 13), dtype=np.uint8))
    np.testing.assert_array_equal(a["losses"], b["losses"])
    for s in range(2):
        assert O.weights_rel_frobenius(b["W"][s], a["W"][s], net.fast_mats) == 0.0


def test_all_zeros_mask_never_updates_and_scores_like_eq4():
    """No target enters any update: W stays W_0 and every loss is the static
    (eq. (4)) loss, although every token is still scored."""
    net = rand_net("swiglu", n_fast=1, fast_mats=("Wd",), seed=82)
    tok = rand_tokens(16, 2, 12, seed=83)
    out = O.prefill(net, 0.3, 0.0, 4, tok, loss_mask=np.zeros((2, 12), dtype=np.uint8))
    for s in range(2):
        np.testing.assert_allclose(out["losses"][s], O.static_losses(net, tok[s]), rtol=0, atol=1e-13)
        assert O.weights_rel_frobenius(out["W"][s], net.fast0, net.fast_mats) == 0.0


def test_single_unmasked_target_is_that_tokens_own_gradient():
    """Only target j of a chunk unmasked: the chunk gradient equals the
    gradient of token j alone (a one-token chunk, eq. (2)); tokens do not mix
    inside the MLP-only network."""
    net = rand_net("gelu", n_fast=2, seed=84)
    tok = rand_tokens(16, 1, 6, seed=85)[0]
    x_in, tgt = tok[:-1], tok[1:]
    j = 3
    mask = np.zeros(6)
    mask[j] = 1
    _, g = O.chunk_loss_and_grads(net, net.fast0, O.frozen_prefix(net, x_in), tgt, O.mask_weights(mask))
    _, g1 = O.chunk_loss_and_grads(net, net.fast0, O.frozen_prefix(net, x_in[j:j + 1]), tgt[j:j + 1])
    for l in range(2):
        for k in net.fast_mats:
            np.testing.assert_allclose(g[l][k], g1[l][k], rtol=1e-12, atol=1e-15)


def test_masked_chunk_gradient_matches_central_differences():
    """The gradient of (1/n) sum_{m_t = 1} l_t, every fast matrix, rel <= 1e-6."""
    net = rand_net("gelu", d=8, f=16, V=16, n_prefix=1, n_fast=1, seed=86)
    tok = rand_tokens(16, 1, 5, seed=87)[0]
    x_in, tgt = tok[:-1], tok[1:]
    mask = np.array([1, 0, 1, 1, 0])
    w = O.mask_weights(mask)
    fast = copy.deepcopy(net.fast0)
    _, grads = O.chunk_loss_and_grads(net, fast, O.frozen_prefix(net, x_in), tgt, w)
    obj = lambda: float(np.sum(w * O.token_losses(net, fast, x_in, tgt)))
    h = 1e-5
    for k in net.fast_mats:
        fd = np.zeros_like(fast[0][k])
        for idx in np.ndindex(fast[0][k].shape):
            orig = fast[0][k][idx]
            fast[0][k][idx] = orig + h
            lp = obj()
            fast[0][k][idx] = orig - h
            lm = obj()
            fast[0][k][idx] = orig
            fd[idx] = (lp - lm) / (2 * h)
        rel = np.linalg.norm(fd - grads[0][k]) / np.linalg.norm(grads[0][k])
        assert rel <= 1e-6, (k, rel)
    assert abs(w.sum() - 1.0) < 1e-15


# ------------------------------------------------------------------ periodic reset (R9)
def test_reset_every_chunk_scores_like_eq4_and_ends_at_w0():
    """A reset after every update: each chunk is scored by W_0, so the losses
    are the static (eq. (4)) losses, and the run ends on W_0."""
    net = rand_net("gelu", seed=90)
    tok = rand_tokens(16, 2, 12, seed=91)
    out = O.prefill(net, 0.4, 0.0, 3, tok, reset_every=1)
    for s in range(2):
        np.testing.assert_allclose(out["losses"][s], O.static_losses(net, tok[s]), rtol=0, atol=1e-13)
        assert O.weights_rel_frobenius(out["W"][s], net.fast0, net.fast_mats) == 0.0


def test_reset_splits_the_stream_into_independent_runs():
    """reset_every = k: every k-chunk segment is a fresh run from W_0 on that
    segment's tokens (the MLP-only network sees no earlier context), so the
    losses and the weights equal those of independent prefills."""
    net = rand_net("swiglu", n_fast=1, fast_mats=("Wd",), seed=92)
    b, k, eta, c = 2, 3, 0.5, 0.8
    T = 2 * k * b + 2 * b + 1                   # two whole segments, a partial one, a ragged tail
    tok = rand_tokens(16, 1, T, seed=93)
    out = O.prefill(net, eta, c, b, tok, reset_every=k)
    seg = k * b
    for m, lo in enumerate(range(0, T, seg)):
        hi = min(lo + seg, T)
        part = O.prefill(net, eta, c, b, tok[:, lo:hi + 1])
        np.testing.assert_allclose(out["losses"][0, lo:hi], part["losses"][0], rtol=0, atol=1e-13)
    # the run ends inside the third segment: its weights are that segment's own run
    assert O.weights_rel_frobenius(out["W"][0], part["W"][0], net.fast_mats) < 1e-14
    assert out["states"][0].chunks_done == T // b


def test_reset_beyond_the_stream_is_no_reset():
    net = rand_net("gelu", seed=94)
    tok = rand_tokens(16, 1, 12, seed=95)
    a = O.prefill(net, 0.3, 0.5, 4, tok)
    r = O.prefill(net, 0.3, 0.5, 4, tok, reset_every=4)
    np.testing.assert_array_equal(a["losses"], r["losses"])
    assert O.weights_rel_frobenius(r["W"][0], a["W"][0], net.fast_mats) == 0.0


def test_reset_counts_decoded_chunks_too():
    """Decoding's steps advance the same counter: a prefill of one chunk and a
    decoded second chunk with reset_every = 2 land back on W_0, and the next
    decoded token is scored like the static model."""
    net = rand_net("gelu", seed=96)
    b = 3
    tok = rand_tokens(16, 1, 3 * b + 1, seed=97)
    out = O.prefill(net, 0.5, 0.0, b, tok[:, :b + 1], reset_every=2)
    st = out["states"][0]
    assert O.weights_rel_frobenius(st.W, net.fast0, net.fast_mats) > 0.0
    for t in range(b + 1, 2 * b + 1):
        O.decode_step(net, st, tok[0, t], 0.5, 0.0, b)
    assert st.chunks_done == 2
    assert O.weights_rel_frobenius(st.W, net.fast0, net.fast_mats) == 0.0
    l, _ = O.decode_step(net, st, tok[0, 2 * b + 1], 0.5, 0.0, b)
    np.testing.assert_allclose(l, O.static_losses(net, tok[0, 2 * b:2 * b + 2])[0], rtol=0, atol=1e-13)


def test_reset_and_settlement_are_exclusive():
    net = rand_net("gelu", seed=98)
    tok = rand_tokens(16, 1, 8, seed=99)
    with pytest.raises(ValueError):
        O.prefill(net, 0.3, 0.0, 2, tok, settle_every=2, settle_q=np.zeros((2, 1, 4), np.int64), reset_every=2)


# ------------------------------------------------------------------ two MLPs per fast block (R10)
def _with_static(net, seed, std=0.5):
    rng = np.random.default_rng(seed)
    net.static = [{k: rng.normal(0, std, v.shape) for k, v in b.items()} for b in net.fast0]
    return net


def test_static_mlp_gradients_match_central_differences():
    """With a frozen MLP before every fast one, the fast gradients (which pass
    through the later static MLPs to the earlier fast blocks) match central
    differences at rel <= 1e-6, and the static MLPs get no gradient."""
    net = _with_static(rand_net("gelu", d=8, f=16, V=16, n_prefix=1, n_fast=3, seed=60), seed=61)
    tok = rand_tokens(16, 1, 3, seed=62)[0]
    x_in, tgt = tok[:-1], tok[1:]
    fast = copy.deepcopy(net.fast0)
    _, grads = O.chunk_loss_and_grads(net, fast, O.frozen_prefix(net, x_in), tgt)
    h = 1e-5
    for l, Wb in enumerate(fast):
        assert set(grads[l]) == set(net.fast_mats)
        for k in net.fast_mats:
            fd = np.zeros_like(Wb[k])
            for idx in np.ndindex(Wb[k].shape):
                orig = Wb[k][idx]
                Wb[k][idx] = orig + h
                lp = _chunk_mean_loss(net, fast, x_in, tgt)
                Wb[k][idx] = orig - h
                lm = _chunk_mean_loss(net, fast, x_in, tgt)
                Wb[k][idx] = orig
                fd[idx] = (lp - lm) / (2 * h)
            rel = np.linalg.norm(fd - grads[l][k]) / np.linalg.norm(grads[l][k])
            assert rel <= 1e-6, (l, k, rel)


def test_static_mlp_runs_before_the_fast_one():
    """Static-first (R10): fast block 0's static MLP acts like one more frozen
    prefix block, so moving it into the prefix (and leaving an identity static
    MLP, W2 = 0, in its place) changes no loss and no weight of a whole run."""
    net = _with_static(rand_net("gelu", n_prefix=1, n_fast=2, seed=63), seed=64)
    moved = copy.deepcopy(net)
    moved.prefix = moved.prefix + [copy.deepcopy(net.static[0])]
    moved.static[0] = {"W1": net.static[0]["W1"], "W2": np.zeros_like(net.static[0]["W2"])}
    tok = rand_tokens(16, 2, 12, seed=65)
    a = O.prefill(net, 0.3, 0.5, 4, tok)
    b = O.prefill(moved, 0.3, 0.5, 4, tok)
    np.testing.assert_allclose(a["losses"], b["losses"], rtol=0, atol=1e-13)
    for s in range(2):
        assert O.weights_rel_frobenius(a["W"][s], b["W"][s], net.fast_mats) < 1e-14


def test_identity_static_mlps_are_the_plain_network():
    """W2 = 0 in every static MLP makes each one the identity: the run equals
    the network without static MLPs, exactly."""
    net = rand_net("gelu", n_prefix=1, n_fast=2, seed=66)
    with_id = copy.deepcopy(net)
    with_id.static = [{"W1": np.ones_like(b["W1"]), "W2": np.zeros_like(b["W2"])} for b in net.fast0]
    tok = rand_tokens(16, 1, 12, seed=67)
    a = O.prefill(net, 0.3, 0.5, 3, tok)
    b = O.prefill(with_id, 0.3, 0.5, 3, tok)
    np.testing.assert_array_equal(a["losses"], b["losses"])
    assert O.weights_rel_frobenius(b["W"][0], a["W"][0], net.fast_mats) == 0.0


def test_static_mlps_change_the_result():
    """Non-trivial static MLPs do change the losses (they are not skipped)."""
    net = rand_net("gelu", n_prefix=0, n_fast=2, seed=68)
    with_s = _with_static(copy.deepcopy(net), seed=69)
    tok = rand_tokens(16, 1, 8, seed=70)
    a = O.prefill(net, 0.3, 0.0, 4, tok)
    b = O.prefill(with_s, 0.3, 0.0, 4, tok)
    assert np.max(np.abs(a["losses"] - b["losses"])) > 1e-3


# ------------------------------------------------------------------ sliding-window attention (R11)
def _attn_net(E, heads, window, Wa, d, f=3, kind="gelu"):
    """One frozen block whose MLP is the identity (W2 = 0) after its attention."""
    V = E.shape[0]
    mlp = {"W1": np.ones((f, d)), "W2": np.zeros((d, f))}
    w = {"E": E, "U": np.eye(V, d), "prefix": [mlp], "fast": [{"W1": np.ones((f, d)), "W2": np.zeros((d, f))}],
         "attn": [Wa]}
    return O.Net.from_weights(w, kind, ("W1", "W2"), 0.0, heads=heads, window=window)


def test_attention_by_hand_one_and_two_heads():
    """d = 2, tokens (0, 1) with e0 = (1, 0), e1 = (0, 2), every projection the
    identity.  Position 1 sees (0, 1): one head scores 0 and 4/sqrt(2); two
    heads (d_h = 1) score (0, 0) and (0, 4); a window of 1 sees itself only."""
    E = np.array([[1.0, 0.0], [0.0, 2.0]])
    I = {k: np.eye(2) for k in ("Wq", "Wk", "Wv", "Wo")}
    e0, e1 = E[0], E[1]
    h = O.frozen_prefix(_attn_net(E, 1, 2, I, 2), np.array([0, 1]))
    p = np.exp([0.0, 4.0 / math.sqrt(2.0)])
    p /= p.sum()
    np.testing.assert_allclose(h[0], 2 * e0, rtol=1e-14)
    np.testing.assert_allclose(h[1], e1 + p[0] * e0 + p[1] * e1, rtol=1e-14)
    h2 = O.frozen_prefix(_attn_net(E, 2, 2, I, 2), np.array([0, 1]))
    q = np.exp([0.0, 4.0])
    q /= q.sum()
    np.testing.assert_allclose(h2[1], e1 + np.array([0.5, 2.0 * q[1]]), rtol=1e-14)
    h1 = O.frozen_prefix(_attn_net(E, 1, 1, I, 2), np.array([0, 1]))
    np.testing.assert_allclose(h1[1], 2 * e1, rtol=1e-14)


def test_attention_with_zero_queries_is_the_window_mean():
    """Wq = 0: every score is 0, so position t gets the mean of V over
    positions max(0, t - k + 1) .. t, then Wo."""
    rng = np.random.default_rng(140)
    d, V, k, n = 6, 9, 3, 8
    E = rng.normal(size=(V, d))
    Wa = {"Wq": np.zeros((d, d)), "Wk": rng.normal(size=(d, d)), "Wv": rng.normal(size=(d, d)),
          "Wo": rng.normal(size=(d, d))}
    x = rng.integers(0, V, size=n)
    h = O.frozen_prefix(_attn_net(E, 2, k, Wa, d), x)
    Vv = E[x] @ Wa["Wv"].T
    for t in range(n):
        lo = max(0, t - k + 1)
        np.testing.assert_allclose(h[t], E[x[t]] + Vv[lo:t + 1].mean(axis=0) @ Wa["Wo"].T, rtol=1e-12, atol=1e-13)


def test_attention_sees_exactly_its_receptive_field():
    """Two attention blocks of window k: position t depends on the 2(k - 1) + 1
    inputs ending at t and on nothing earlier (no positional encoding, so the
    suffix alone reproduces the row)."""
    rng = np.random.default_rng(141)
    d, f, V, k, n = 8, 16, 16, 3, 12
    blk = lambda: {"W1": rng.normal(0, 0.5, (f, d)), "W2": rng.normal(0, 0.5, (d, f))}
    att = lambda: {m: rng.normal(0, 0.5, (d, d)) for m in ("Wq", "Wk", "Wv", "Wo")}
    w = {"E": rng.normal(size=(V, d)), "U": rng.normal(size=(V, d)), "prefix": [blk(), blk()], "fast": [blk()],
         "attn": [att(), att()]}
    net = O.Net.from_weights(w, "gelu", ("W1", "W2"), 1e-6, heads=2, window=k)
    x = rng.integers(0, V, size=n)
    full = O.frozen_prefix(net, x)
    r = 2 * (k - 1) + 1
    np.testing.assert_allclose(O.frozen_prefix(net, x[n - r:])[-1], full[-1], rtol=1e-12, atol=1e-12)
    x2 = x.copy()
    x2[n - r - 1] = (x2[n - r - 1] + 1) % V           # just outside: no change
    np.testing.assert_array_equal(O.frozen_prefix(net, x2)[-1], full[-1])
    x3 = x.copy()
    x3[n - r] = (x3[n - r] + 1) % V                   # just inside: a change
    assert np.max(np.abs(O.frozen_prefix(net, x3)[-1] - full[-1])) > 1e-6


def test_attention_prefill_scores_chunks_with_their_context():
    """With attention the chunk losses depend on the tokens before the chunk
    (the bigram defect's fix), and decoding or Settlement raise."""
    rng = np.random.default_rng(142)
    d, f, V = 8, 16, 16
    blk = lambda: {"W1": rng.normal(0, 0.5, (f, d)), "W2": rng.normal(0, 0.5, (d, f))}
    att = {m: rng.normal(0, 0.5, (d, d)) for m in ("Wq", "Wk", "Wv", "Wo")}
    w = {"E": rng.normal(size=(V, d)), "U": rng.normal(size=(V, d)), "prefix": [blk()], "fast": [blk()],
         "attn": [att]}
    net = O.Net.from_weights(w, "gelu", ("W1", "W2"), 1e-6, heads=2, window=6)
    tok = rand_tokens(V, 1, 12, seed=143)
    a = O.prefill(net, 0.0, 0.0, 4, tok)
    tok2 = tok.copy()
    tok2[0, 2] = (tok2[0, 2] + 1) % V                 # a token of chunk 1 only
    b = O.prefill(net, 0.0, 0.0, 4, tok2)
    assert np.max(np.abs(a["losses"][0, 4:8] - b["losses"][0, 4:8])) > 1e-6    # chunk 2 sees it
    np.testing.assert_array_equal(a["losses"][0, 9:], b["losses"][0, 9:])       # beyond the window: not
    with pytest.raises(ValueError):
        O.settle(net, a["states"][0], tok[0, :6])


@pytest.mark.parametrize("T", [8, 7], ids=["whole_chunks", "ragged"])
def test_decoding_with_attention_equals_a_longer_prefill(T):
    """Decoding continues the positions: a prefill of T tokens then decoding
    to T + extra gives the losses, weights and p_{T+1} of one prefill of
    T + extra, with two attention layers whose window reaches into prefill."""
    rng = np.random.default_rng(144)
    d, f, V = 8, 16, 16
    blk = lambda: {"W1": rng.normal(0, 0.5, (f, d)), "W2": rng.normal(0, 0.5, (d, f))}
    att = lambda: {m: rng.normal(0, 0.5, (d, d)) for m in ("Wq", "Wk", "Wv", "Wo")}
    w = {"E": rng.normal(size=(V, d)), "U": rng.normal(size=(V, d)), "prefix": [blk(), blk()], "fast": [blk()],
         "attn": [att(), att()]}
    net = O.Net.from_weights(w, "gelu", ("W1", "W2"), 1e-6, heads=2, window=3)
    b, extra, eta, c = 4, 9, 0.3, 0.7
    tok = rand_tokens(V, 1, T + extra, seed=145)
    long = O.prefill(net, eta, c, b, tok)
    short = O.prefill(net, eta, c, b, tok[:, :T + 1])
    st = short["states"][0]
    dec = []
    for t in range(T + 1, T + extra + 1):
        l, p = O.decode_step(net, st, tok[0, t], eta, c, b)
        dec.append(l)
    np.testing.assert_allclose(dec, long["losses"][0, T:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(p, long["p_next"][0], rtol=0, atol=1e-12)
    assert O.weights_rel_frobenius(st.W, long["W"][0], net.fast_mats) < 1e-13


def test_weights_rel_frobenius_on_a_hand_computed_pair():
    """The parity tests' weight error ||Wa - Wb||_F / ||Wb||_F over every fast
    matrix of one sequence, on integer matrices worked by hand:
    block 0: W1 differs by one entry of 2, W2 by one entry of 1; block 1: W2
    differs by one entry of 2.  Squared differences 4 + 1 + 0 + 4 = 9; squared
    norms of Wb 26 + 4 + 4 + 4 = 38; so the error is 3 / sqrt(38).  Over W2
    alone: 5 / 8 under the root.  A missing root, Wa's norm as the
    denominator (43) or a block left out all change the value."""
    Wa = [{"W1": np.array([[1.0, 2.0], [3.0, 4.0]]), "W2": np.array([[0.0, 1.0]])},
          {"W1": np.array([[1.0, 1.0], [1.0, 1.0]]), "W2": np.array([[2.0, 2.0]])}]
    Wb = [{"W1": np.array([[1.0, 0.0], [3.0, 4.0]]), "W2": np.array([[0.0, 2.0]])},
          {"W1": np.array([[1.0, 1.0], [1.0, 1.0]]), "W2": np.array([[2.0, 0.0]])}]
    assert abs(O.weights_rel_frobenius(Wa, Wb, ("W1", "W2")) - 3.0 / np.sqrt(38.0)) < 1e-15
    assert abs(O.weights_rel_frobenius(Wa, Wb, ("W2",)) - np.sqrt(5.0 / 8.0)) < 1e-15
    assert O.weights_rel_frobenius(Wb, Wb, ("W1", "W2")) == 0.0
