"""Seeded initial weights: N(0, std^2) drawn in float64, rounded to the
workload's storage type (float32, or bfloat16 via float32), returned as
float32 arrays whose values are exactly representable in that type.

Layout (row-major, linear maps stored [out, in]):
  E [V, d]          embedding, row v = token v
  U [V, d]          LM head, logits = y @ U.T
  GELU block:   W1 [d_ff, d], W2 [d, d_ff]
  SwiGLU block: Wg [d_ff, d], Wu [d_ff, d], Wd [d, d_ff]

Matrix m of the workload is drawn from SeedSequence([seed id, 0, m]) with
m = 0 for E, 1 for U, then 2 + 3 * block + position-in-block over the prefix
blocks followed by the fast blocks; with static MLPs in the fast blocks, the
static MLP of fast block l continues after them at 2 + 3 * (n_prefix + n_fast
+ l) + position; with attention, prefix block p's (Wq, Wk, Wv, Wo) follow
at 2 + 3 * (n_prefix + 2 * n_fast) + 4 * p + position.  Only the generator
lives here; the arithmetic of the method does not.
"""
from __future__ import annotations

import numpy as np

from .configs import GELU_MATS, SWIGLU_MATS, Workload
from .markov import PURPOSE_WEIGHTS, rng_for


def round_to_bf16(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), as float32."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    bits = x32.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    bits = (bits + 0x7FFF + lsb) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "fp32":
        return x32
    if dtype == "bf16":
        return round_to_bf16(x32)
    raise ValueError(dtype)


def block_shapes(wl: Workload) -> dict:
    f, d = wl.d_ff, wl.d
    if wl.block == "gelu":
        return {"W1": (f, d), "W2": (d, f)}
    if wl.block == "swiglu":
        return {"Wg": (f, d), "Wu": (f, d), "Wd": (d, f)}
    raise ValueError(wl.block)


def block_mats(block: str) -> tuple:
    return GELU_MATS if block == "gelu" else SWIGLU_MATS


def _draw(wl: Workload, index: int, shape: tuple) -> np.ndarray:
    rng = rng_for(wl.seed_id, PURPOSE_WEIGHTS, index)
    rows, cols = shape
    out = np.empty(shape, dtype=np.float32)
    step = max(1, (1 << 23) // cols)      # bound the float64 scratch to ~64 MB
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = round_to(rng.normal(0.0, wl.init_std, size=(r1 - r0, cols)), wl.dtype)
    return out


def make_weights(wl: Workload) -> dict:
    shapes = block_shapes(wl)
    mats = block_mats(wl.block)
    w = {"E": _draw(wl, 0, (wl.vocab, wl.d)), "U": _draw(wl, 1, (wl.vocab, wl.d)),
         "prefix": [], "fast": []}
    for blk in range(wl.n_prefix + wl.n_fast):
        bw = {name: _draw(wl, 2 + 3 * blk + pos, shapes[name]) for pos, name in enumerate(mats)}
        (w["prefix"] if blk < wl.n_prefix else w["fast"]).append(bw)
    if wl.static_mlp:
        base = 2 + 3 * (wl.n_prefix + wl.n_fast)
        w["static"] = [{name: _draw(wl, base + 3 * l + pos, shapes[name]) for pos, name in enumerate(mats)}
                       for l in range(wl.n_fast)]
    if wl.attn_heads:
        base = 2 + 3 * (wl.n_prefix + 2 * wl.n_fast)
        w["attn"] = [{name: _draw(wl, base + 4 * p + pos, (wl.d, wl.d))
                      for pos, name in enumerate(("Wq", "Wk", "Wv", "Wo"))} for p in range(wl.n_prefix)]
    return w


def make_inputs(wl: Workload) -> dict:
    """Weights, the token stream [B, T+1] and the held-out chunks [E, B, Lq]."""
    from .markov import make_chain, sample_heldout, sample_stream
    chain = make_chain(wl.seed_id, wl.vocab, wl.chain_k, wl.chain_alpha, wl.uniform_mix)
    tokens = sample_stream(chain, wl.seed_id, wl.B, wl.T)
    q = sample_heldout(chain, wl.seed_id, wl.n_settle_events, wl.B, wl.settle_len)
    return {"weights": make_weights(wl), "tokens": tokens, "settle_q": q, "chain": chain}
