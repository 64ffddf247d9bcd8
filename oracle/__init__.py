"""Float64 CPU oracle of the chunked next-token TTT inner loop.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package's smoke
check and by the benchmark's CPU-baseline leg, never by the product library.
"""
from .ttt_oracle import *  # noqa: F401,F403
from .ttt_oracle import Net, SeqState, prefill, prefill_sequence  # noqa: F401
