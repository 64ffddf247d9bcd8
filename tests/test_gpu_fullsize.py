"""The bf16 workloads at their full stated sizes, in the launch configuration
the benchmark times (same B, widths, chunk, clip and eta, full T), through the
C ABI, against the float64 oracle.

The oracle needs minutes to hours of host time at these widths, so its outputs
come from tests/golden/fullsize_<workload>.npz, written by
tests/golden/make_fullsize.py (oracle and input generators only):
  * 125M-like stream: every per-token loss of the whole stream (32 chunks) of
    sequences 0 and 7, their final fast weights and p_{T+1};
  * 4B-like in-place shape: the first 16 chunks of its one sequence;
  * 760M-like stream with Settlement: the first 32 chunks of all 8 sequences,
    i.e. 4 Settlement events, 32 decisions.
Fast weights are compared on a seeded sample of 4096 elements per matrix (the
fixture holds W_final - W_0 there).  Checks:
  * the benchmark spec tolerances: mean per-token |loss error| <= 2e-2 per sequence,
    relative Frobenius error of the final fast weights <= 3e-2;
  * the update itself: the relative error of W_final - W_0 on the sample (the
    weights are dominated by W_0, so the tolerance above cannot see a wrong
    update), within DELTA_TOL, a bound taken from measurement (see below);
  * Settlement: |A_gpu - A_oracle| <= A_NOISE for every event, and every
    decision whose oracle score clears the noise bound agrees exactly; at least
    MIN_DECIDED of the 32 must clear it;
  * properties at any size over the whole stream: every loss finite, no larger
    than a uniform guess by much, and ||W_T - W_0||_F <= eta * clip * chunks.
"""
import json
import os

import numpy as np
import pytest
import torch

import synth
from synth import configs as C

from gpu_harness import TOL, run_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.fullsize]

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Relative error of the sampled update W_final - W_0 (bf16 operands, fp32
# accumulation and masters): measured on B300 at these sizes, with margin.
DELTA_TOL = 5e-2
# Settlement: bound on |A_gpu - A_oracle|.  Measured on B300 at the 760M-like
# shape over the 32 decisions of the fixture: mean -3.0e-6, standard deviation
# 8.4e-5, largest 2.1e-4 (the candidate scored as the committed bf16 copy plus
# its bf16 offset); the bound doubles the largest.  Every oracle score of the
# fixture is at least 6.4e-4, so all 32 decisions clear it and must agree.
A_NOISE = 4e-4
MIN_DECIDED = 32


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _report(name, data):
    """Measured errors, written when TTT_TEST_REPORT_DIR names a folder."""
    d = os.environ.get("TTT_TEST_REPORT_DIR")
    if d:
        os.makedirs(d, exist_ok=True)
        with open(os.path.join(d, f"fullsize_{name}.json"), "w") as f:
            json.dump(data, f, indent=1)


def _fast_delta_norm(W, W0, mats):
    return float(np.sqrt(sum(float(np.sum((np.asarray(a[k], np.float64) - b[k]) ** 2))
                             for a, b in zip(W, W0) for k in mats)))


def _check_full_size(wl):
    fx = dict(np.load(os.path.join(GOLDEN, f"fullsize_{wl.name}.npz")))
    seqs = [int(s) for s in fx["seqs"]]
    n_chunks = int(fx["n_chunks"])
    n = n_chunks * wl.chunk
    inp = synth.make_inputs(wl)
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
    # the fast weights after the fixture's chunks: the full run's own when it
    # covers the whole stream, else a prefill of that prefix on the same handle
    if n == wl.T:
        W_at = gpu["W"]
    else:
        tok_n = np.ascontiguousarray(inp["tokens"][:, :n + 1])
        W_at = run_gpu(wl, inp, tokens=tok_n, handle=gpu["handle"])["W"]
    rep = {"workload": wl.name, "chunks": n_chunks, "seqs": seqs, "per_seq": {}}
    for i, s in enumerate(seqs):
        err = np.abs(gpu["losses"][s, :n] - fx["losses"][i].astype(np.float64))
        num = den = dnum = dden = 0.0
        for l in range(wl.n_fast):
            for m in wl.fast_mats:
                idx = fx[f"idx_{l}_{m}"]
                d_or = fx[f"delta_{l}_{m}"][i].astype(np.float64)
                w0 = np.asarray(W0[l][m], np.float64).ravel()[idx]
                d_gpu = np.asarray(W_at[s][l][m], np.float64).ravel()[idx] - w0
                num += float(np.sum((d_gpu - d_or) ** 2))
                den += float(np.sum((w0 + d_or) ** 2))
                dden += float(np.sum(d_or ** 2))
        w_rel = float(np.sqrt(num / den))
        d_rel = float(np.sqrt(num / dden))
        rep["per_seq"][s] = {"loss_mean_err": float(err.mean()), "loss_max_err": float(err.max()),
                             "w_rel": w_rel, "delta_rel": d_rel}
        if "p_next" in fx:
            rep["per_seq"][s]["p_next_max_err"] = float(np.abs(gpu["p_next"][s] - fx["p_next"][i]).max())
    _report(wl.name, rep)
    return fx, gpu, rep


def _assert_full_size(rep):
    tol = TOL["bf16"]
    for s, r in rep["per_seq"].items():
        assert r["loss_mean_err"] <= tol["loss_mean"], f"seq {s}: mean loss err {r['loss_mean_err']:.3e}"
        assert r["w_rel"] <= tol["w_rel"], f"seq {s}: W rel-Frobenius {r['w_rel']:.3e}"
        assert r["delta_rel"] <= DELTA_TOL, f"seq {s}: update rel error {r['delta_rel']:.3e} ({rep})"
        if "p_next_max_err" in r:
            assert r["p_next_max_err"] <= 2e-3, f"seq {s}: p_next err {r['p_next_max_err']:.3e}"


def test_e2e125m_whole_stream():
    _assert_full_size(_check_full_size(C.E2E_125M)[2])


def test_inplace4b_sixteen_chunks():
    _assert_full_size(_check_full_size(C.INPLACE_4B)[2])


def test_settle760m_thirty_two_chunks_all_sequences():
    wl = C.SETTLE_760M
    fx, gpu, rep = _check_full_size(wl)
    assert gpu["A"].shape == (wl.n_settle_events, wl.B)
    assert np.all(np.isfinite(gpu["A"]))
    seqs = [int(s) for s in fx["seqs"]]
    E = fx["A"].shape[0]
    dA = np.abs(gpu["A"][:E][:, seqs] - fx["A"])
    decidable = np.abs(fx["A"]) > A_NOISE
    agree = gpu["accept"][:E][:, seqs] == fx["accept"]
    rep["settlement"] = {"events": int(E), "A_oracle": fx["A"].tolist(), "A_gpu": gpu["A"][:E][:, seqs].tolist(),
                         "max_abs_dA": float(dA.max()), "mean_abs_dA": float(dA.mean()),
                         "decidable": int(decidable.sum()), "agree_decidable": int((agree & decidable).sum()),
                         "agree_all": int(agree.sum())}
    _report(wl.name, rep)
    _assert_full_size(rep)
    assert dA.max() <= A_NOISE, f"|A_gpu - A_oracle| up to {dA.max():.3e} ({rep['settlement']})"
    assert np.all(agree[decidable]), f"a decidable Settlement decision differs ({rep['settlement']})"
    assert decidable.sum() >= MIN_DECIDED, f"only {int(decidable.sum())} decidable events ({rep['settlement']})"
