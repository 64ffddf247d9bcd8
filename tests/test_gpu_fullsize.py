"""The bf16 workloads at their full stated sizes, in the launch configuration
the benchmark times (same B, widths, chunk, clip and eta; T as stated), through
the C ABI.  The oracle cannot replay whole streams in seconds, so the checks
are (1) sampled outputs it can compute one by one: the per-token losses of the
first two chunks of the first and last sequences, their fast weights after two
chunks (from a second, two-chunk prefill on the same handle), and for the
Settlement workload the first event's score and decision; and (2) properties
that hold at any size: every loss finite and no larger than a uniform guess by
much, and the clip bound ||W_T - W_0||_F <= eta * clip * (number of chunks)
for every sequence (each clipped step moves W by at most eta * clip)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import configs as C

from gpu_harness import TOL, compare_settlement, make, run_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.fullsize]


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _fast_delta_norm(W, W0, mats):
    return float(np.sqrt(sum(float(np.sum((np.asarray(a[k], np.float64) - b[k]) ** 2))
                             for a, b in zip(W, W0) for k in mats)))


def _check_full_size(wl, k_chunks=2):
    inp = make(wl)
    gpu = run_gpu(wl, inp)
    B, T = gpu["losses"].shape
    assert (B, T) == (wl.B, wl.T)
    # properties at any size
    assert np.all(np.isfinite(gpu["losses"]))
    assert gpu["losses"].max() < np.log(wl.vocab) + 10.0
    W0 = inp["weights"]["fast"]
    bound = wl.eta * wl.clip * wl.n_chunks
    for s in range(B):
        assert _fast_delta_norm(gpu["W"][s], W0, wl.fast_mats) <= bound * (1 + 1e-3) + 1e-6
    # sampled outputs: the first k chunks of the first and last sequences
    seqs = sorted({0, B - 1})
    kb = k_chunks * wl.chunk
    tok_k = np.ascontiguousarray(inp["tokens"][:, :kb + 1])
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps)
    ref = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, tok_k, seqs=seqs)
    short = run_gpu(wl, inp, tokens=tok_k, handle=gpu["handle"])
    tol = TOL["bf16"]
    for s in seqs:
        err = np.abs(gpu["losses"][s, :kb] - ref["losses"][s])
        assert err.mean() <= tol["loss_mean"], f"seq {s}: mean loss err {err.mean():.3e}"
        # the two-chunk run hoists its prefix over 2 chunks instead of the whole
        # group, so its GEMMs may split K differently: same tolerance, not bits
        err_short = np.abs(short["losses"][s] - ref["losses"][s])
        assert err_short.mean() <= tol["loss_mean"], f"seq {s}: two-chunk run mean loss err {err_short.mean():.3e}"
        rel = oracle.weights_rel_frobenius(short["W"][s], ref["W"][s], wl.fast_mats)
        assert rel <= tol["w_rel"], f"seq {s}: W rel-Frobenius after {k_chunks} chunks {rel:.3e}"
    return inp, gpu, net


def test_e2e125m_full_size():
    _check_full_size(C.E2E_125M)


def test_inplace4b_full_size():
    _check_full_size(C.INPLACE_4B)


def test_settle760m_full_size_first_event():
    wl = C.SETTLE_760M
    inp, gpu, net = _check_full_size(wl)
    assert gpu["A"].shape == (wl.n_settle_events, wl.B)
    assert np.all(np.isfinite(gpu["A"]))
    # the first Settlement event of sequence 0, replayed by the oracle
    n = wl.settle_every * wl.chunk
    tok = np.ascontiguousarray(inp["tokens"][:, :n + 1])
    ref = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, tok, wl.settle_every, inp["settle_q"][:1], seqs=[0])
    first = {"A": gpu["A"][:1], "accept": gpu["accept"][:1]}
    compare_settlement(first, ref, [0], noise=5e-3)
