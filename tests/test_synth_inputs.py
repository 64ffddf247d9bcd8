"""The seeded generators: Markov statistics, determinism, weight rounding."""
import numpy as np
import pytest
import torch
from scipy import stats

import synth
from synth import markov
from synth.configs import WORKLOADS


def test_chain_rows_are_distributions_with_distinct_successors():
    ch = markov.make_chain(99, 64, 8, 0.3)
    assert ch.succ.shape == (64, 8)
    assert all(len(set(r)) == 8 for r in ch.succ.tolist())
    P = ch.dense()
    np.testing.assert_allclose(P.sum(1), 1.0, rtol=1e-12)
    assert P.min() >= 0.05 / 64 - 1e-15


def test_stream_transition_counts_match_the_chain_chi_square():
    V = 12
    ch = markov.make_chain(98, V, 4, 0.3)
    tok = markov.sample_stream(ch, 98, 4, 40000)
    assert tok.dtype == np.int32 and np.all(tok[:, 0] == 0)
    counts = np.zeros((V, V))
    for s in range(tok.shape[0]):
        np.add.at(counts, (tok[s, :-1], tok[s, 1:]), 1)
    P = ch.dense()
    pvals = []
    for i in range(V):
        n = counts[i].sum()
        if n < 2000:
            continue
        pvals.append(stats.chisquare(counts[i], n * P[i]).pvalue)
    assert len(pvals) >= 6
    # under the null the p-values are uniform; a wrong sampler gives ~0 everywhere
    assert min(pvals) > 1e-6
    assert stats.kstest(pvals, "uniform").pvalue > 1e-4


def test_streams_are_seeded_and_independent_of_batch_size():
    ch = markov.make_chain(97, 50, 5, 0.3)
    a = markov.sample_stream(ch, 97, 3, 200)
    b = markov.sample_stream(ch, 97, 1, 200)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a, markov.sample_stream(ch, 97, 3, 200))
    assert not np.array_equal(a[0], a[1])
    q = markov.sample_heldout(ch, 97, 2, 3, 16)
    assert q.shape == (2, 3, 16) and np.all(q[:, :, 0] == 0)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 0.02, 100000), rng.normal(0, 50, 1000),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875])]).astype(np.float32)
    ours = synth.round_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours, ref)


@pytest.mark.parametrize("wl", WORKLOADS[:2], ids=lambda w: w.name)
def test_weights_shapes_and_statistics(wl):
    w = synth.make_weights(wl)
    assert w["E"].shape == (wl.vocab, wl.d) and w["U"].shape == (wl.vocab, wl.d)
    assert len(w["prefix"]) == wl.n_prefix and len(w["fast"]) == wl.n_fast
    assert w["fast"][0]["W1"].shape == (wl.d_ff, wl.d)
    assert abs(float(np.std(w["U"])) - 0.02) < 1e-3
    np.testing.assert_array_equal(synth.make_weights(wl)["U"], w["U"])


def test_workload_table_matches_the_stated_shapes():
    names = [w.name for w in WORKLOADS]
    assert len(set(names)) == 5
    for w in WORKLOADS:
        assert w.T % w.chunk == 0
    assert WORKLOADS[4].n_settle_events == 16
