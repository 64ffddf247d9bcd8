"""Write the oracle fixtures of the full-size parity tests in this folder.

The float64 oracle needs minutes to hours on host cores for the bf16 workloads
at their stated widths, longer than a GPU test run may take, so it runs here
once and its outputs are stored.  Calls only the oracle and the seeded input
generators; no value comes from the CUDA library.

Per workload (inputs drawn at the workload's full T, since a stream's tokens
depend on T through the generator's draw order, then cut to the first
`n_chunks` chunks):
  losses    [n_seq, n_chunks * b] float32: the prequential per-token losses
  p_next    [n_seq, V] float32 (only when n_chunks covers the whole stream)
  scales    [n_seq, n_chunks]: the clip factor s of every step
  A, accept [E, n_seq]: Settlement scores and decisions (Settlement workloads)
  idx_<l>_<mat>    sampled flat indices into fast matrix <mat> of fast block l
  delta_<l>_<mat>  [n_seq, n_idx] float32: (W_final - W_0) at those indices

    python tests/golden/make_fullsize.py [workload name ...]
"""
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402
from synth import configs as C  # noqa: E402

# sequences and chunk prefix of each workload's fixture
CASES = {
    C.E2E_125M.name: {"seqs": (0, C.E2E_125M.B - 1), "n_chunks": C.E2E_125M.n_chunks},   # whole stream
    C.INPLACE_4B.name: {"seqs": (0,), "n_chunks": 16},
    C.SETTLE_760M.name: {"seqs": tuple(range(C.SETTLE_760M.B)), "n_chunks": 32},         # 4 Settlement events
}
W_SAMPLE = 4096          # sampled elements per fast matrix
SAMPLE_PURPOSE = 7       # SeedSequence purpose word of the element sample


def path_for(name):
    return os.path.join(HERE, f"fullsize_{name}.npz")


def sample_index(wl, l, k, n):
    rng = np.random.default_rng(np.random.SeedSequence([wl.seed_id, SAMPLE_PURPOSE, 3 * l + k]))
    return np.unique(rng.integers(0, n, size=W_SAMPLE)).astype(np.int64)


def fixture(name):
    wl = C.BY_NAME[name]
    case = CASES[name]
    seqs, n_chunks = list(case["seqs"]), case["n_chunks"]
    inp = synth.make_inputs(wl)
    tok = np.ascontiguousarray(inp["tokens"][:, :n_chunks * wl.chunk + 1])
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps)
    t0 = time.time()
    ref = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, tok, wl.settle_every,
                         inp["settle_q"] if wl.settle_every else None, seqs=seqs)
    dt = time.time() - t0
    out = {"seqs": np.array(seqs, dtype=np.int64), "n_chunks": np.int64(n_chunks),
           "oracle_seconds": np.float64(dt),
           "losses": np.stack([ref["losses"][s] for s in seqs]).astype(np.float32),
           "scales": np.stack([np.array(ref["states"][s].scales) for s in seqs])}
    if n_chunks * wl.chunk == wl.T:
        out["p_next"] = np.stack([ref["p_next"][s] for s in seqs]).astype(np.float32)
    if wl.settle_every:
        out["A"] = ref["A"][:, seqs]
        out["accept"] = ref["accept"][:, seqs]
    W0 = inp["weights"]["fast"]
    for l in range(wl.n_fast):
        for k, m in enumerate(wl.fast_mats):
            w0 = np.asarray(W0[l][m], np.float64).ravel()
            idx = sample_index(wl, l, k, w0.size)
            out[f"idx_{l}_{m}"] = idx
            out[f"delta_{l}_{m}"] = np.stack(
                [np.asarray(ref["W"][s][l][m], np.float64).ravel()[idx] - w0[idx] for s in seqs]).astype(np.float32)
    return out


if __name__ == "__main__":
    names = sys.argv[1:] or list(CASES)
    for name in names:
        fx = fixture(name)
        np.savez_compressed(path_for(name), **fx)
        print(f"{name}: {len(fx['seqs'])} sequences x {int(fx['n_chunks'])} chunks, "
              f"oracle {float(fx['oracle_seconds']):.0f} s", flush=True)
