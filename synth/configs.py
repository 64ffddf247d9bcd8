"""The five synthetic workloads of the chunked next-token TTT inner loop.

Each workload is a network shape, the TTT hyper-parameters and the Markov
chain its tokens come from.  Shapes follow the TTT-E2E toy (attention-free
MLP-only network), a 125M-like and a 760M-like TTT-E2E stream (one clipped
SGD step per 1024-token chunk on the last MLP blocks, batch width 8), and an
In-Place-TTT-like block whose down projection is the only fast weight.

This module holds data only: no arithmetic of the method lives here.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    seed_id: int            # first word of every SeedSequence of this workload
    d: int                  # model width
    d_ff: int               # MLP hidden width
    vocab: int
    n_prefix: int           # frozen MLP blocks after the embedding
    n_fast: int             # MLP blocks whose (some) matrices are fast weights
    block: str              # "gelu" (W1, W2) or "swiglu" (Wg, Wu, Wd)
    fast_mats: tuple        # names of the fast matrices inside a fast block
    dtype: str              # storage/compute type: "fp32" or "bf16"
    eta: float
    clip: float             # 0 = no clipping
    chunk: int              # b, tokens per TTT mini-batch
    B: int                  # sequences
    T: int                  # tokens per sequence after BOS (tokens are [B, T+1])
    chain_k: int            # successors per row of the Markov chain
    chain_alpha: float      # Dirichlet concentration of the successor weights
    settle_every: int = 0   # chunks between Settlement events, 0 = off
    settle_len: int = 0     # tokens of each held-out chunk q
    reset_every: int = 0    # chunk updates between resets of the fast weights to W_0, 0 = off
    static_mlp: bool = False  # each fast block also holds a frozen MLP, run before its fast one
    attn_heads: int = 0     # sliding-window attention heads in every frozen prefix block, 0 = none
    attn_window: int = 0    # its window k (keys t-k+1 .. t)
    rms_eps: float = 1e-6
    uniform_mix: float = 0.05
    init_std: float = 0.02

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def n_chunks(self) -> int:
        return self.T // self.chunk

    @property
    def n_settle_events(self) -> int:
        if not self.settle_every:
            return 0
        return self.n_chunks // self.settle_every


GELU_MATS = ("W1", "W2")
SWIGLU_MATS = ("Wg", "Wu", "Wd")

TOY_BIGRAM = Workload(
    name="toy_bigram_fp32_d64_v256_b1", seed_id=1,
    d=64, d_ff=256, vocab=256, n_prefix=0, n_fast=1, block="gelu",
    fast_mats=GELU_MATS, dtype="fp32", eta=0.1, clip=0.0, chunk=1, B=1, T=1024,
    chain_k=16, chain_alpha=0.3)

CHUNKED_FP32 = Workload(
    name="chunked_fp32_d512_v4096_b256", seed_id=2,
    d=512, d_ff=2048, vocab=4096, n_prefix=2, n_fast=2, block="gelu",
    fast_mats=GELU_MATS, dtype="fp32", eta=0.05, clip=1.0, chunk=256, B=4, T=8192,
    chain_k=32, chain_alpha=0.1)

E2E_125M = Workload(
    name="e2e125m_bf16_d768_v32000_b1024", seed_id=3,
    d=768, d_ff=3072, vocab=32000, n_prefix=9, n_fast=3, block="gelu",
    fast_mats=GELU_MATS, dtype="bf16", eta=0.01, clip=1.0, chunk=1024, B=8, T=32768,
    chain_k=16, chain_alpha=0.3)

INPLACE_4B = Workload(
    name="inplace4b_bf16_d2560_v151936_b512", seed_id=4,
    d=2560, d_ff=9728, vocab=151936, n_prefix=4, n_fast=1, block="swiglu",
    fast_mats=("Wd",), dtype="bf16", eta=0.005, clip=1.0, chunk=512, B=1, T=65536,
    chain_k=32, chain_alpha=0.1)

SETTLE_760M = Workload(
    name="settle760m_bf16_d1536_v32000_b1024", seed_id=5,
    d=1536, d_ff=6144, vocab=32000, n_prefix=6, n_fast=3, block="gelu",
    fast_mats=GELU_MATS, dtype="bf16", eta=0.01, clip=1.0, chunk=1024, B=8, T=131072,
    chain_k=16, chain_alpha=0.3, settle_every=8, settle_len=1024)

WORKLOADS = (TOY_BIGRAM, CHUNKED_FP32, E2E_125M, INPLACE_4B, SETTLE_760M)

# The 125M-like stream with sliding-window attention (12 heads of 64) in its
# nine frozen blocks, window k = 2048 >= b, at T = 16384 (the pages pair
# k = 8K with b = 1K at 128K context; this keeps k / b = 2 at a length one
# GPU step measures in well under a second).
SWA_125M = E2E_125M.replace(name="swa125m_bf16_d768_v32000_b1024_k2048", seed_id=6, T=16384,
                            attn_heads=12, attn_window=2048)

EXTRA_WORKLOADS = (SWA_125M,)
BY_NAME = {w.name: w for w in WORKLOADS + EXTRA_WORKLOADS}
