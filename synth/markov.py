"""Seeded sparse first-order Markov chains and token streams.

Row i of the chain has `k` distinct successor tokens drawn uniformly, with
weights w ~ Dirichlet(alpha * 1_k), mixed with a uniform draw:

    P(j | i) = (1 - u) * sum_m w_m [j == s_m] + u / V,   u = 0.05.

A stream starts at x_0 = 0 (the BOS token) and draws each x_t from
P(. | x_{t-1}).  The Markov streams stand in for the book and agent text the
pages evaluate on; none of that text is present here.

Seeds: numpy SeedSequence([workload seed id, purpose, index]) with purpose
1 = chain, 2 = stream (index = sequence), 3 = held-out chunk
(index = event * B + sequence).  Sequence s never depends on B.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

PURPOSE_WEIGHTS = 0
PURPOSE_CHAIN = 1
PURPOSE_STREAM = 2
PURPOSE_HELDOUT = 3


def rng_for(seed_id: int, purpose: int, index: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed_id, purpose, index]))


@dataclass
class Chain:
    succ: np.ndarray      # [V, k] int64, distinct per row
    w: np.ndarray         # [V, k] float64, rows sum to 1
    cdf: np.ndarray       # [V, k] float64 cumulative of w (last column forced to 1)
    uniform_mix: float

    @property
    def vocab(self) -> int:
        return self.succ.shape[0]

    def dense(self) -> np.ndarray:
        """[V, V] transition matrix; only for small V (tests)."""
        V, k = self.succ.shape
        P = np.full((V, V), self.uniform_mix / V)
        rows = np.repeat(np.arange(V), k)
        np.add.at(P, (rows, self.succ.ravel()), (1.0 - self.uniform_mix) * self.w.ravel())
        return P


def make_chain(seed_id: int, vocab: int, k: int, alpha: float,
               uniform_mix: float = 0.05) -> Chain:
    rng = rng_for(seed_id, PURPOSE_CHAIN, 0)
    if k > vocab:
        raise ValueError("k > vocab")
    succ = rng.integers(0, vocab, size=(vocab, k))
    while True:                      # redraw rows holding a repeated successor
        s = np.sort(succ, axis=1)
        bad = np.any(s[:, 1:] == s[:, :-1], axis=1)
        if not bad.any():
            break
        succ[bad] = rng.integers(0, vocab, size=(int(bad.sum()), k))
    w = rng.dirichlet(np.full(k, alpha), size=vocab)
    cdf = np.cumsum(w, axis=1)
    cdf[:, -1] = 1.0
    return Chain(succ=succ.astype(np.int64), w=w, cdf=cdf, uniform_mix=uniform_mix)


def _walk(chain: Chain, rngs: list, length: int, start: int = 0) -> np.ndarray:
    """Walk len(rngs) independent streams for `length` transitions."""
    n = len(rngs)
    V = chain.vocab
    # every stream draws its own three uniform arrays up front, so a stream's
    # tokens depend only on its own generator
    mix = np.stack([r.random(length) for r in rngs]) < chain.uniform_mix
    usucc = np.stack([r.random(length) for r in rngs])
    uni = np.stack([r.integers(0, V, size=length) for r in rngs])
    out = np.empty((n, length + 1), dtype=np.int64)
    out[:, 0] = start
    prev = out[:, 0].copy()
    for t in range(length):
        cdf = chain.cdf[prev]                                  # [n, k]
        j = (cdf < usucc[:, t:t + 1]).sum(axis=1)
        j = np.minimum(j, chain.succ.shape[1] - 1)
        nxt = chain.succ[prev, j]
        nxt = np.where(mix[:, t], uni[:, t], nxt)
        out[:, t + 1] = nxt
        prev = nxt
    return out


def sample_stream(chain: Chain, seed_id: int, B: int, T: int) -> np.ndarray:
    """Tokens [B, T+1] int32, x_0 = 0 (BOS) for every sequence."""
    rngs = [rng_for(seed_id, PURPOSE_STREAM, s) for s in range(B)]
    return _walk(chain, rngs, T).astype(np.int32)


def sample_heldout(chain: Chain, seed_id: int, events: int, B: int, L: int) -> np.ndarray:
    """Held-out chunks q [events, B, L] int32, each starting at BOS."""
    if events == 0:
        return np.zeros((0, B, L), dtype=np.int32)
    rngs = [rng_for(seed_id, PURPOSE_HELDOUT, e * B + s)
            for e in range(events) for s in range(B)]
    q = _walk(chain, rngs, L - 1)
    return q.reshape(events, B, L).astype(np.int32)
