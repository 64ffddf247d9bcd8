"""Float64 CPU oracle of the chunked next-token test-time-training (TTT) loop.

TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the CPU
baseline leg of the benchmark may import or run anything in this package.  The
product library never calls it and shares no code, header, table or helper with
it: only the seeded input generators in `synth` feed both.

Sources (the pages define the method; nothing here is copied from code):
  [E2E] "End-to-End Test-Time Training for Long Context" (paper review page).
        Method 1: eq. (1) per-token loss l_t(W) = CE(f(x_{t-1}; W), x_t),
        eq. (2) online update, output p_{T+1} = f(x_T; W_T).
        Method 2: eq. (3) prequential loss, eq. (4) TTT-naive loss.
        Method 3: eq. (5) mini-batch update with the (1/b) mean over the chunk,
        eq. (6) generalised loss, output f(x_T; W_{T/b}).
        3.1 Implementation Details: only MLP layers are updated; only the last
        blocks are fast.  3.2 Decoding Multiple Tokens: a step is taken only
        when decoded tokens fill a mini-batch.
  [INP] "In-Place Test-Time Training" (review page), Key Terms: the MLP final
        projection is the fast weight; chunk-wise update.
  [SGF] "Self-Generated Feedback Destabilizes Test-Time Training" (summary
        page), "How it works": one clipped gradient step per 1024-token chunk
        on the last three FFN modules; weights restored after each evaluation.
        Settlement paragraph: candidate W+delta, A(delta; W, q) =
        L(q, W) - L(q, W + delta), commit delta only when A >= 0.

Readings taken where the pages leave a step open:
  R1  Every sequence of a batch owns its fast weights, all starting from the
      shared W_0; gradients never mix across sequences (each sequence is its
      own test sequence in eq. (3)).
  R2  Chunk i (1-based) feeds inputs x_{(i-1)b} .. x_{ib-1} and targets
      x_{(i-1)b+1} .. x_{ib}; losses[s, t-1] holds l_t.  x_0 is BOS (= 0).
  R3  Block = h + GELU(h W1^T) W2^T (GELU) or h + (silu(h Wg^T) * h Wu^T) Wd^T
      (SwiGLU): no per-block norm, no biases.  One final RMSNorm with unit,
      frozen gain: y = x / sqrt(mean(x^2) + eps), eps = 1e-6.  Exact erf GELU.
      logits = y U^T with U stored [V, d].
  R4  Clip: g is the concatenation of all fast-matrix gradients of one
      sequence; s = min(1, c / (||g||_2 + 1e-6)); c = 0 means no clipping.
      Plain SGD: W <- W - eta * s * g (no momentum, no weight decay).
  R5  Settlement: delta is the sum of the updates since the last commit.  The
      stream keeps running on W_c + delta; after every `settle_every`-th chunk
      update, A = L(q, W_c) - L(q, W_c + delta) is scored on that event's
      held-out chunk q, and A >= 0 commits (W_c <- W) else reverts (W <- W_c).
      L(q, W) is the mean of the len(q)-1 next-token CEs of q through the
      whole network with no update.  Weights returned after the last chunk
      are the stream's current weights, committed or not.
  R6  If b does not divide T, the trailing T mod b tokens are scored with the
      last weights and kept pending; decoding completes that chunk.
  R7  Decoding: decode_step(x_new) appends the pair (x_prev, x_new); when b
      pairs are pending, one (clipped) step is taken on them with the weights
      that scored them; p_next = softmax(f(x_new; W)) uses the weights after
      that step.  Settlement is not applied while decoding.
  R8  Source Masking (the [SGF] Settlement paragraph compares Settlement with
      Source Masking, which uses per-token source labels, but gives no
      formula): a per-token mask marks the targets whose loss enters the
      update; every token is still scored (prequential losses are unchanged
      in definition), and a chunk's TTT loss is the mean over its unmasked
      targets, (1/n) sum_{t: m_t = 1} l_t with n = max(1, sum m_t), so a chunk
      without any unmasked target leaves W unchanged.  All-ones masks are the
      unmasked method.
  R9  Periodic reset (the [SGF] limits paragraph reports an 8-chunk reset as a
      mitigation, without a formula): after every `reset_every`-th chunk
      update of a sequence (prefill and decoding counted together) its fast
      weights return to W_0.  Reset and Settlement are alternatives, never
      combined in one run.
  R10 Two MLPs per updated block ([E2E] 3.1, "Two MLP layers per block": a
      static MLP is added to every block that TTT updates, to keep what
      pre-training stored): a fast block is two residual sublayers, the
      frozen MLP first and the fast MLP second, h <- h + MLP_s(h) then
      h <- h + MLP_f(h), both of the block's kind and widths.  The page does
      not give the order; static-first is this reading.  Gradients reach
      earlier fast blocks through the later static MLPs.
  R11 Sliding-window attention in the frozen blocks ([E2E] Method, the
      bigram defect and its fix: a sliding-window attention layer of window
      k, with k >= b so a chunk remembers its own tokens before the update;
      3.1: attention layers stay frozen).  Every frozen prefix block becomes
      h <- h + Attn(h) then h <- h + MLP(h); Attn(h) = concat over heads of
      softmax(Q_h K_h^T / sqrt(d_h) + M) V_h, times Wo^T, with Q = h Wq^T,
      K = h Wk^T, V = h Wv^T (all [d, d], stored [out, in]) and M = 0 where
      the key position s satisfies t - k < s <= t for query position t, -inf
      elsewhere.  Positions count the inputs x_0 (BOS) .. of one sequence from
      0; no positional encoding is added (the pages name none).  The fast
      blocks hold no attention, so the whole prefix of a sequence depends on
      its tokens only and is computed once over x_0 .. x_T.  Decoding goes on
      at the following positions: a decoded input attends to itself and the
      k - 1 inputs before it, prefill's included, and the prefix rows of the
      pending inputs are the ones computed when each input arrived.
      Settlement is not defined here with attention (the held-out chunk's
      attention context is not fixed by the pages).
"""
from __future__ import annotations

import copy
from dataclasses import dataclass, field

import numpy as np
from scipy.special import erf

SQRT2 = np.sqrt(2.0)
INV_SQRT_2PI = 1.0 / np.sqrt(2.0 * np.pi)
CLIP_EPS = 1e-6


# ---------------------------------------------------------------- pointwise
def gelu(z):
    """Exact GELU, z * Phi(z) (reading R3)."""
    return z * 0.5 * (1.0 + erf(z / SQRT2))


def gelu_grad(z):
    """d/dz [z Phi(z)] = Phi(z) + z phi(z)."""
    return 0.5 * (1.0 + erf(z / SQRT2)) + z * INV_SQRT_2PI * np.exp(-0.5 * z * z)


def silu(g):
    return g / (1.0 + np.exp(-g))


def silu_grad(g):
    s = 1.0 / (1.0 + np.exp(-g))
    return s * (1.0 + g * (1.0 - s))


# ---------------------------------------------------------------- layers
def rmsnorm(x, eps):
    """y = x / sqrt(mean(x^2) + eps), unit gain (reading R3).  Returns y, rstd."""
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1) + eps)
    return x * r[:, None], r


def rmsnorm_backward(x, r, dy):
    """dx = r * (dy - xhat * mean(xhat * dy)) with xhat = x * r."""
    xh = x * r[:, None]
    return r[:, None] * (dy - xh * np.mean(xh * dy, axis=-1)[:, None])


def block_forward(kind, Wb, h):
    """One residual MLP block (reading R3).  Returns (h_out, cache)."""
    if kind == "gelu":
        z = h @ Wb["W1"].T
        a = gelu(z)
        return h + a @ Wb["W2"].T, {"h": h, "z": z, "a": a}
    if kind == "swiglu":
        g = h @ Wb["Wg"].T
        u = h @ Wb["Wu"].T
        a = silu(g) * u
        return h + a @ Wb["Wd"].T, {"h": h, "g": g, "u": u, "a": a}
    raise ValueError(kind)


def block_backward(kind, Wb, cache, dout, fast_mats, need_dh):
    """Gradients of the block's fast matrices and (optionally) d h_in.

    Only the MLP matrices named in `fast_mats` get gradients ([E2E] 3.1: the
    embedding, norms and everything else stay frozen).
    """
    grads = {}
    h = cache["h"]
    if kind == "gelu":
        if "W2" in fast_mats:
            grads["W2"] = dout.T @ cache["a"]
        if "W1" in fast_mats or need_dh:
            dz = (dout @ Wb["W2"]) * gelu_grad(cache["z"])
            if "W1" in fast_mats:
                grads["W1"] = dz.T @ h
            dh = dout + dz @ Wb["W1"] if need_dh else None
        else:
            dh = None
        return grads, dh
    if kind == "swiglu":
        if "Wd" in fast_mats:
            grads["Wd"] = dout.T @ cache["a"]
        if "Wg" in fast_mats or "Wu" in fast_mats or need_dh:
            da = dout @ Wb["Wd"]
            dg = da * cache["u"] * silu_grad(cache["g"])
            du = da * silu(cache["g"])
            if "Wg" in fast_mats:
                grads["Wg"] = dg.T @ h
            if "Wu" in fast_mats:
                grads["Wu"] = du.T @ h
            dh = dout + dg @ Wb["Wg"] + du @ Wb["Wu"] if need_dh else None
        else:
            dh = None
        return grads, dh
    raise ValueError(kind)


def cross_entropy(logits, targets):
    """Per-row CE = logsumexp(logits) - logits[target] and softmax (eq. (1))."""
    m = logits.max(axis=-1)
    e = np.exp(logits - m[:, None])
    se = e.sum(axis=-1)
    lse = m + np.log(se)
    losses = lse - logits[np.arange(len(targets)), targets]
    return losses, e / se[:, None]


# ---------------------------------------------------------------- network
@dataclass
class Net:
    """Frozen parameters plus the fast set's initial values W_0 (all float64)."""
    kind: str
    eps: float
    E: np.ndarray
    U: np.ndarray
    prefix: list
    fast0: list               # per fast block: dict of all its matrices
    fast_mats: tuple          # which matrices of a fast block are fast
    static: list | None = None  # per fast block: its frozen MLP (R10), or None
    attn: list | None = None    # per prefix block: its attention (Wq, Wk, Wv, Wo) (R11), or None
    heads: int = 0
    window: int = 0

    @staticmethod
    def from_weights(w: dict, kind: str, fast_mats, eps: float, heads: int = 0, window: int = 0) -> "Net":
        f64 = lambda a: np.asarray(a, dtype=np.float64)
        st = w.get("static")
        at = w.get("attn") if heads else None
        return Net(kind=kind, eps=eps, E=np.asarray(w["E"]), U=f64(w["U"]),
                   prefix=[{k: f64(v) for k, v in b.items()} for b in w["prefix"]],
                   fast0=[{k: f64(v) for k, v in b.items()} for b in w["fast"]],
                   fast_mats=tuple(fast_mats),
                   static=None if st is None else [{k: f64(v) for k, v in b.items()} for b in st],
                   attn=None if at is None else [{k: f64(v) for k, v in b.items()} for b in at],
                   heads=heads if at is not None else 0, window=window if at is not None else 0)

    @property
    def vocab(self):
        return self.U.shape[0]


def window_mask(n, k):
    """R11: allowed[t, s] iff t - k < s <= t."""
    t = np.arange(n)[:, None]
    s = np.arange(n)[None, :]
    return (s <= t) & (s > t - k)


def attention(Wa, h, heads, window):
    """Sliding-window multi-head attention over the rows of h, row t being
    position t of one sequence (R11)."""
    n, d = h.shape
    dh = d // heads
    Q, K, V = h @ Wa["Wq"].T, h @ Wa["Wk"].T, h @ Wa["Wv"].T
    allowed = window_mask(n, window)
    out = np.zeros_like(h)
    for i in range(heads):
        c = slice(i * dh, (i + 1) * dh)
        S = np.where(allowed, Q[:, c] @ K[:, c].T / np.sqrt(dh), -np.inf)
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P /= P.sum(axis=1, keepdims=True)
        out[:, c] = P @ V[:, c]
    return out @ Wa["Wo"].T


def frozen_prefix(net: Net, x):
    """Embedding rows then the frozen blocks ([E2E] 3.1: these never train).
    With attention (R11) x is one whole sequence from position 0."""
    h = np.asarray(net.E[x], dtype=np.float64)
    for p, Wb in enumerate(net.prefix):
        if net.attn is not None:
            h = h + attention(net.attn[p], h, net.heads, net.window)
        h, _ = block_forward(net.kind, Wb, h)
    return h


def forward_logits(net: Net, fast, h_in):
    h = h_in
    for l, Wb in enumerate(fast):
        if net.static is not None:
            h, _ = block_forward(net.kind, net.static[l], h)      # R10
        h, _ = block_forward(net.kind, Wb, h)
    y, _ = rmsnorm(h, net.eps)
    return y @ net.U.T


def token_losses(net: Net, fast, x_in, targets, h_in=None):
    """l_t for each (input, target) pair with fixed weights `fast` (eq. (1));
    h_in: the prefix output of these inputs when already computed."""
    logits = forward_logits(net, fast, frozen_prefix(net, x_in) if h_in is None else h_in)
    return cross_entropy(logits, targets)[0]


def chunk_loss_and_grads(net: Net, fast, h_in, targets, weights=None):
    """Losses of one chunk and the gradient of their mean (eq. (5)'s (1/b) sum);
    with `weights` [b], the gradient of sum_t weights[t] * l_t instead (the
    Source Masking reading R8 passes mask / max(1, sum(mask)))."""
    b = len(targets)
    caches, static_caches = [], []
    h = h_in
    for l, Wb in enumerate(fast):
        if net.static is not None:
            h, c = block_forward(net.kind, net.static[l], h)      # R10
            static_caches.append(c)
        h, c = block_forward(net.kind, Wb, h)
        caches.append(c)
    y, r = rmsnorm(h, net.eps)
    logits = y @ net.U.T
    losses, p = cross_entropy(logits, targets)
    dlogits = p
    dlogits[np.arange(b), targets] -= 1.0
    if weights is None:
        dlogits /= b
    else:
        dlogits *= np.asarray(weights, dtype=np.float64)[:, None]
    dh = rmsnorm_backward(h, r, dlogits @ net.U)
    grads = [None] * len(fast)
    for l in range(len(fast) - 1, -1, -1):
        grads[l], dh = block_backward(net.kind, fast[l], caches[l], dh, net.fast_mats,
                                      need_dh=l > 0)
        if net.static is not None and l > 0:
            # through the frozen MLP to the fast blocks below (no gradient of its own)
            _, dh = block_backward(net.kind, net.static[l], static_caches[l], dh, (), need_dh=True)
    return losses, grads


def clip_scale(grads, clip):
    """s = min(1, c / (||g|| + 1e-6)) over one sequence's fast set (reading R4)."""
    sq = 0.0
    for g in grads:
        for v in g.values():
            sq += float(np.sum(v * v))
    norm = np.sqrt(sq)
    if clip <= 0.0:
        return 1.0, norm
    return min(1.0, clip / (norm + CLIP_EPS)), norm


def sgd_step(fast, grads, eta, s):
    """W <- W - eta * s * g on the fast matrices only (eqs. (2), (5))."""
    out = []
    for Wb, g in zip(fast, grads):
        nb = dict(Wb)
        for k, v in g.items():
            nb[k] = Wb[k] - (eta * s) * v
        out.append(nb)
    return out


def heldout_loss(net: Net, fast, q):
    """L(q, W): mean next-token CE over a held-out chunk, no update (reading R5)."""
    q = np.asarray(q)
    return float(np.mean(token_losses(net, fast, q[:-1], q[1:])))


def softmax_next(net: Net, fast, x_last, h_last=None):
    h = frozen_prefix(net, np.asarray([x_last])) if h_last is None else h_last
    logits = forward_logits(net, fast, h)
    return cross_entropy(logits, np.zeros(1, dtype=np.int64))[1][0]


# ---------------------------------------------------------------- the loop
@dataclass
class SeqState:
    """Per-sequence TTT state (reading R1)."""
    W: list
    Wc: list | None
    x_last: int
    pend_in: list = field(default_factory=list)
    pend_tgt: list = field(default_factory=list)
    chunks_done: int = 0
    norms: list = field(default_factory=list)
    scales: list = field(default_factory=list)
    reset_every: int = 0
    hist: list = field(default_factory=list)      # attention (R11): inputs x_0 .. x_last
    h_last: object = None                         # attention: prefix row of x_last
    pend_h: list = field(default_factory=list)    # attention: prefix rows of the pending inputs


def settle(net, st: SeqState, q):
    """Settlement ([SGF]): score the candidate st.W against the committed st.Wc
    on held-out q; A >= 0 commits the candidate, otherwise st.W reverts."""
    if net.attn is not None:
        raise ValueError("Settlement is not defined with attention (R11)")
    A = heldout_loss(net, st.Wc, q) - heldout_loss(net, st.W, q)
    accept = bool(A >= 0.0)
    if accept:
        st.Wc = copy.deepcopy(st.W)
    else:
        st.W = copy.deepcopy(st.Wc)
    return A, accept


def mask_weights(mask):
    """Source Masking (R8): the chunk's TTT loss is the mean over the targets
    whose mask is 1; a chunk without any contributes no gradient."""
    m = np.asarray(mask, dtype=np.float64)
    return m / max(1.0, float(m.sum()))


def _step(net, st: SeqState, x_in, tgt, eta, clip, mask=None, h_in=None):
    if h_in is None:
        h_in = frozen_prefix(net, x_in)
    w = None if mask is None else mask_weights(mask)
    losses, grads = chunk_loss_and_grads(net, st.W, h_in, tgt, w)
    s, norm = clip_scale(grads, clip)
    st.W = sgd_step(st.W, grads, eta, s)
    st.chunks_done += 1
    st.norms.append(norm)
    st.scales.append(s)
    if st.reset_every and st.chunks_done % st.reset_every == 0:
        st.W = copy.deepcopy(net.fast0)       # R9
    return losses


def prefill_sequence(net: Net, eta, clip, b, tokens, settle_every=0, settle_q=None,
                     snapshots=False, loss_mask=None, reset_every=0):
    """Run one sequence's prefill.  tokens: [T+1] with tokens[0] = BOS;
    loss_mask [T] (optional, R8): target t+1 enters the update iff mask[t];
    reset_every (R9): chunk updates between returns to W_0, 0 = never."""
    tokens = np.asarray(tokens, dtype=np.int64)
    T = len(tokens) - 1
    n_full, rem = divmod(T, b)
    if settle_every and reset_every:
        raise ValueError("reset and Settlement are alternatives (R9)")
    st = SeqState(W=copy.deepcopy(net.fast0),
                  Wc=copy.deepcopy(net.fast0) if settle_every else None,
                  x_last=int(tokens[-1]), reset_every=reset_every)
    # with attention (R11) the prefix of x_0 .. x_T is one pass over the sequence
    H = frozen_prefix(net, tokens) if net.attn is not None else None
    rows = (lambda lo, hi: None) if H is None else (lambda lo, hi: H[lo:hi])
    losses = np.zeros(T)
    snaps = [copy.deepcopy(st.W)] if snapshots else None
    A_list, acc_list = [], []
    for i in range(n_full):
        lo = i * b
        losses[lo:lo + b] = _step(net, st, tokens[lo:lo + b], tokens[lo + 1:lo + b + 1],
                                  eta, clip, None if loss_mask is None else loss_mask[lo:lo + b],
                                  rows(lo, lo + b))
        if settle_every and (i + 1) % settle_every == 0:
            e = (i + 1) // settle_every - 1
            A, accept = settle(net, st, settle_q[e])
            A_list.append(A)
            acc_list.append(accept)
        if snapshots:
            snaps.append(copy.deepcopy(st.W))
    if rem:
        lo = n_full * b
        x_in, tgt = tokens[lo:T], tokens[lo + 1:T + 1]
        losses[lo:] = token_losses(net, st.W, x_in, tgt, rows(lo, T))
        st.pend_in = list(x_in)
        st.pend_tgt = list(tgt)
        if H is not None:
            st.pend_h = list(H[lo:T])
    if H is not None:
        st.hist = [int(t) for t in tokens]
        st.h_last = H[T]
    p_next = softmax_next(net, st.W, st.x_last, rows(T, T + 1))
    return {"losses": losses, "state": st, "p_next": p_next, "A": np.array(A_list),
            "accept": np.array(acc_list, dtype=bool), "snapshots": snaps}


def prefill(net: Net, eta, clip, b, tokens, settle_every=0, settle_q=None, snapshots=False,
            seqs=None, loss_mask=None, reset_every=0):
    """Batched prefill: every sequence runs independently (reading R1).

    tokens [B, T+1]; settle_q [E, B, Lq] when settle_every > 0; loss_mask
    [B, T] (optional, R8) selects the targets whose loss enters the update;
    reset_every (R9) returns the fast weights to W_0 periodically.  `seqs`
    restricts the run to some sequences (the others are left zero / None).
    Returns losses [B, T], per-sequence final fast weights, p_next [B, V],
    A and accept [E, B].
    """
    tokens = np.asarray(tokens)
    B, T1 = tokens.shape
    seqs = range(B) if seqs is None else seqs
    n_events = ((T1 - 1) // b) // settle_every if settle_every else 0
    out = {"losses": np.zeros((B, T1 - 1)), "W": [None] * B,
           "p_next": np.zeros((B, net.vocab)), "A": np.zeros((n_events, B)),
           "accept": np.zeros((n_events, B), dtype=bool), "states": [None] * B,
           "snapshots": [None] * B}
    for s in seqs:
        r = prefill_sequence(net, eta, clip, b, tokens[s], settle_every,
                             None if settle_q is None else np.asarray(settle_q)[:, s],
                             snapshots, None if loss_mask is None else np.asarray(loss_mask)[s],
                             reset_every)
        out["losses"][s] = r["losses"]
        out["W"][s] = r["state"].W
        out["p_next"][s] = r["p_next"]
        if n_events:
            out["A"][:, s] = r["A"]
            out["accept"][:, s] = r["accept"]
        out["states"][s] = r["state"]
        out["snapshots"][s] = r["snapshots"]
    return out


def decode_step(net: Net, st: SeqState, x_new, eta, clip, b):
    """One decoded token for one sequence (reading R7; a reset of R9 applies
    to the steps taken here as well).

    Returns (l of the new token under the weights that scored it, p_next).
    """
    x_new = int(x_new)
    attn = net.attn is not None
    h_prev = st.h_last[None, :] if attn else None
    loss = float(token_losses(net, st.W, np.array([st.x_last]), np.array([x_new]), h_prev)[0])
    st.pend_in.append(st.x_last)
    st.pend_tgt.append(x_new)
    if attn:
        # R11: the new input's prefix row sees the receptive field of the
        # attention layers, (k - 1) per layer before it (the suffix alone
        # reproduces that row: no positional encoding)
        st.pend_h.append(st.h_last)
        st.hist.append(x_new)
        reach = (net.window - 1) * len(net.prefix) + 1
        st.h_last = frozen_prefix(net, np.array(st.hist[-reach:]))[-1]
    st.x_last = x_new
    if len(st.pend_in) == b:
        _step(net, st, np.array(st.pend_in), np.array(st.pend_tgt), eta, clip,
              h_in=np.array(st.pend_h) if attn else None)
        st.pend_in, st.pend_tgt, st.pend_h = [], [], []
    return loss, softmax_next(net, st.W, st.x_last, st.h_last[None, :] if attn else None)


def static_losses(net: Net, tokens):
    """Losses with W_0 throughout: the TTT-naive objective of eq. (4)."""
    tokens = np.asarray(tokens, dtype=np.int64)
    return token_losses(net, net.fast0, tokens[:-1], tokens[1:])


def weights_rel_frobenius(Wa, Wb, mats):
    """||Wa - Wb||_F / ||Wb||_F over all fast matrices of one sequence."""
    num = den = 0.0
    for a, b in zip(Wa, Wb):
        for k in mats:
            num += float(np.sum((np.asarray(a[k], np.float64) - b[k]) ** 2))
            den += float(np.sum(np.asarray(b[k], np.float64) ** 2))
    return np.sqrt(num / den)
