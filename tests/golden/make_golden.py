"""Write the oracle regression fixtures in this folder.

Calls only the oracle and the seeded input generators.  The pages print no
worked numeric example, so every stored value here is the oracle's own output
on a seeded synthetic input; the fixture locks the oracle against unintended
changes (a deliberate change regenerates it and says why).

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402
from synth.configs import TOY_BIGRAM  # noqa: E402


def toy_bigram_fixture(T=256):
    wl = TOY_BIGRAM.replace(T=T)
    inp = synth.make_inputs(wl)
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps)
    out = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, inp["tokens"])
    W = out["W"][0][0]
    return {
        "workload": wl.name, "T": T,
        "source": "oracle prefill on the seeded toy bigram workload (E2E review, "
                  "Method 1: eq. (1)-(3), b = 1)",
        "tokens_head": inp["tokens"][0, :16].tolist(),
        "losses": [float(v) for v in out["losses"][0]],
        "W1_sum": float(np.sum(W["W1"])), "W1_sumsq": float(np.sum(W["W1"] ** 2)),
        "W2_sum": float(np.sum(W["W2"])), "W2_sumsq": float(np.sum(W["W2"] ** 2)),
        "p_next_head": [float(v) for v in out["p_next"][0, :16]],
    }


if __name__ == "__main__":
    fx = toy_bigram_fixture()
    with open(os.path.join(HERE, "toy_bigram_oracle_T256.json"), "w") as f:
        json.dump(fx, f, indent=1)
    print("wrote", len(fx["losses"]), "losses")
