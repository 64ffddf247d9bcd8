"""Seeded synthetic inputs (weights, Markov token streams, held-out chunks).

Shared by the oracle tests, the GPU parity tests and the benchmark.  Holds
no arithmetic of the TTT method itself.
"""
from .configs import BY_NAME, WORKLOADS, Workload  # noqa: F401
from .markov import Chain, make_chain, sample_heldout, sample_stream  # noqa: F401
from .weights import make_inputs, make_weights, round_to, round_to_bf16  # noqa: F401
