"""The oracle against its stored regression fixture, and a sanity curve."""
import json
import os

import numpy as np

import oracle
import synth
from synth.configs import TOY_BIGRAM

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_matches_stored_toy_fixture():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    ref = json.load(open(os.path.join(HERE, "toy_bigram_oracle_T256.json")))
    got = mg.toy_bigram_fixture(ref["T"])
    assert got["tokens_head"] == ref["tokens_head"]
    np.testing.assert_allclose(got["losses"], ref["losses"], rtol=0, atol=1e-12)
    for k in ("W1_sum", "W1_sumsq", "W2_sum", "W2_sumsq"):
        assert abs(got[k] - ref[k]) <= 1e-10 * max(1.0, abs(ref[k]))
    np.testing.assert_allclose(got["p_next_head"], ref["p_next_head"], rtol=1e-10)


def test_toy_loss_stays_near_ln_V_at_random_init():
    """Sanity (not a pin): with N(0, 0.02^2) weights the logits are small, so
    every prequential loss of the toy sits near ln V; random (not
    meta-learned) W_0 gives TTT little to work with at this step size."""
    wl = TOY_BIGRAM
    inp = synth.make_inputs(wl)
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps)
    out = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, inp["tokens"])
    l = out["losses"][0]
    assert abs(l.mean() - np.log(wl.vocab)) < 0.1
    assert np.all(np.isfinite(l))
