"""libttt (CUDA, through the C ABI) against the float64 oracle on seeded inputs.

Workloads run either at their stated sizes or, where the oracle would take
minutes, at the same structure (block kind, dtype, fast set, clip, eta) with
smaller widths and a documented chunk prefix; every case spans several GEMM
tiles and ragged tile tails.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from chunked_next_token_ttt_b300 import Handle
from synth import configs as C

from gpu_harness import TOL, compare, compare_settlement, make, run_gpu, run_oracle

TOL_BF16_LOSS_MEAN = TOL["bf16"]["loss_mean"]

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def test_toy_bigram_fp32_full_size():
    """The pages' toy: b = 1, per-token update (eq. (2)), 1024 tokens."""
    wl = C.TOY_BIGRAM
    inp = make(wl)
    gpu = run_gpu(wl, inp)
    ref = run_oracle(wl, inp)
    compare(wl, gpu, ref)


@pytest.mark.parametrize("token_kernel", ["1", "0"], ids=["persistent", "general"])
def test_per_token_clipped_b1_both_paths(token_kernel):
    """b = 1 with a clip that binds, three sequences, odd widths: the persistent
    per-token kernel (closed-form outer-product norm) and the general chunk path
    both match the oracle within the fp32 tolerance."""
    wl = C.TOY_BIGRAM.replace(d=40, d_ff=100, vocab=90, B=3, T=150, clip=0.05, eta=0.2)
    inp = make(wl)
    gpu = run_gpu(wl, inp, options={"no_token_kernel": token_kernel == "0"})
    ref = run_oracle(wl, inp)
    assert max(max(st.norms) for st in ref["states"]) > wl.clip      # the clip binds
    compare(wl, gpu, ref)


@pytest.mark.parametrize("token_kernel", ["1", "0"], ids=["persistent", "general"])
def test_per_token_clipped_b1_at_the_toy_widths(token_kernel):
    """The toy's widths (d = 64, d_ff = 256, V = 256), where the persistent
    kernel keeps W1 and W2 in registers, with a clip that binds on three
    sequences: it matches the oracle, and so does the general chunk path."""
    wl = C.TOY_BIGRAM.replace(B=3, T=300, clip=0.05, eta=0.2)
    inp = make(wl)
    gpu = run_gpu(wl, inp, options={"no_token_kernel": token_kernel == "0"})
    ref = run_oracle(wl, inp)
    assert max(max(st.norms) for st in ref["states"]) > wl.clip      # the clip binds
    compare(wl, gpu, ref)


def test_decode_after_persistent_per_token_prefill():
    """The persistent kernel writes the fast weights back: decoding continues
    from them (general path) and matches the oracle token by token."""
    wl = C.TOY_BIGRAM.replace(B=2, T=64)
    inp = make(wl)
    extra = 12
    long_tok = synth.sample_stream(inp["chain"], wl.seed_id, wl.B, wl.T + extra)
    tok = np.ascontiguousarray(long_tok[:, :wl.T + 1])
    gpu = run_gpu(wl, inp, tokens=tok)
    h = gpu["handle"]
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps)
    ref = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, tok)
    p = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    loss = torch.empty((wl.B,), dtype=torch.float32, device="cuda")
    for t in range(wl.T + 1, wl.T + extra + 1):
        h.decode_step(torch.from_numpy(long_tok[:, t].copy()).cuda(), p, loss)
        torch.cuda.synchronize()
        for s in range(wl.B):
            l_ref, p_ref = oracle.decode_step(net, ref["states"][s], long_tok[s, t], wl.eta, wl.clip, wl.chunk)
            assert abs(float(loss[s]) - l_ref) <= 1e-4
            assert np.abs(p[s].cpu().numpy() - p_ref).max() <= 1e-5


def test_chunked_fp32_prefix_chunks():
    wl = C.CHUNKED_FP32.replace(T=4 * C.CHUNKED_FP32.chunk)
    inp = make(wl)
    gpu = run_gpu(wl, inp)
    ref = run_oracle(wl, inp)
    compare(wl, gpu, ref)


def test_chunked_fp32_full_size():
    """The benchmark workload at its stated size: B = 4, T = 8192, 32 chunks,
    every loss and the final fast weights within the fp32 tolerance."""
    wl = C.CHUNKED_FP32
    inp = make(wl)
    gpu = run_gpu(wl, inp)
    ref = run_oracle(wl, inp)
    compare(wl, gpu, ref)


def test_chunked_fp32_plain_storage_matches_too():
    """The same workload with fp32 storage forced (SIMT GEMMs) also passes."""
    wl = C.CHUNKED_FP32.replace(T=2 * C.CHUNKED_FP32.chunk, B=2)
    inp = make(wl)
    gpu = run_gpu(wl, inp, options={"fp32_simt": 1})
    ref = run_oracle(wl, inp)
    compare(wl, gpu, ref)


def test_chunked_fp32_odd_shapes_ragged_tail():
    """Widths that are not multiples of any tile, T not a multiple of b."""
    wl = C.CHUNKED_FP32.replace(d=72, d_ff=200, vocab=333, chunk=40, B=3, T=130, n_prefix=1)
    inp = make(wl)
    gpu = run_gpu(wl, inp)
    ref = run_oracle(wl, inp)
    compare(wl, gpu, ref)


def test_e2e125m_bf16_small_widths():
    wl = C.E2E_125M.replace(d=256, d_ff=1024, vocab=2000, chunk=256, B=3, T=3 * 256, n_prefix=2)
    inp = make(wl)
    gpu = run_gpu(wl, inp)
    ref = run_oracle(wl, inp)
    compare(wl, gpu, ref)


def test_inplace_swiglu_down_proj_bf16_small_widths():
    wl = C.INPLACE_4B.replace(d=256, d_ff=640, vocab=3000, chunk=128, B=2, T=3 * 128 + 17, n_prefix=2)
    inp = make(wl)
    gpu = run_gpu(wl, inp)
    ref = run_oracle(wl, inp)
    compare(wl, gpu, ref)


def test_settlement_bf16_small_widths():
    """Settlement after every 8th chunk; half the sequences score their candidate
    on held-out text from a different chain, so both commits and reverts occur."""
    wl = C.SETTLE_760M.replace(d=128, d_ff=512, vocab=512, chunk=64, B=4, T=16 * 64, n_prefix=1,
                               settle_len=64, eta=0.5, init_std=0.08)
    inp = make(wl)
    other = synth.make_chain(wl.seed_id + 100, wl.vocab, wl.chain_k, wl.chain_alpha)
    q = inp["settle_q"].copy()
    q_other = synth.sample_heldout(other, wl.seed_id + 100, q.shape[0], wl.B, wl.settle_len)
    q[:, 1::2] = q_other[:, 1::2]
    gpu = run_gpu(wl, inp, q=q)
    ref = run_oracle(wl, inp, q=q)
    decided = compare_settlement(gpu, ref, range(wl.B), noise=5e-3)
    assert decided >= 6
    assert ref["accept"].any() and (~ref["accept"]).any()
    compare(wl, gpu, ref)


def test_hoisted_prefix_groups_bf16():
    """The frozen prefix runs once per group of chunks; groups of 2 over 5
    chunks (2 + 2 + 1) give the same result as the oracle's chunk-by-chunk loop."""
    wl = C.E2E_125M.replace(d=128, d_ff=512, vocab=1024, chunk=128, B=3, T=5 * 128, n_prefix=2)
    inp = make(wl)
    gpu = run_gpu(wl, inp, options={"hoist_chunks": 2})
    ref = run_oracle(wl, inp)
    compare(wl, gpu, ref)


def test_hoisted_swiglu_activation_groups_ragged_tail():
    """SwiGLU block whose frozen gate/up activation is hoisted with the prefix:
    groups of 2 over 5 chunks, then a ragged tail scored by the per-call path."""
    wl = C.INPLACE_4B.replace(d=128, d_ff=384, vocab=1000, chunk=64, B=2, T=5 * 64 + 9, n_prefix=1)
    inp = make(wl)
    gpu = run_gpu(wl, inp, options={"hoist_chunks": 2})
    ref = run_oracle(wl, inp)
    compare(wl, gpu, ref)


def test_decode_swiglu_bf16_steps_with_the_per_call_prefix():
    """Decoding runs its chunk steps without the hoisted prefix (one token at a
    time): SwiGLU bf16 decode losses and final weights against the oracle."""
    wl = C.INPLACE_4B.replace(d=128, d_ff=384, vocab=1000, chunk=64, B=2, T=64 + 10, n_prefix=1)
    inp = make(wl)
    extra = 64
    long_tok = synth.sample_stream(inp["chain"], wl.seed_id, wl.B, wl.T + extra)
    tok = np.ascontiguousarray(long_tok[:, :wl.T + 1])
    gpu = run_gpu(wl, inp, tokens=tok)
    h = gpu["handle"]
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps)
    ref = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, tok)
    p = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    loss = torch.empty((wl.B,), dtype=torch.float32, device="cuda")
    errs = []
    for t in range(wl.T + 1, wl.T + extra + 1):
        h.decode_step(torch.from_numpy(long_tok[:, t].copy()).cuda(), p, loss)
        torch.cuda.synchronize()
        for s in range(wl.B):
            l_ref, p_ref = oracle.decode_step(net, ref["states"][s], long_tok[s, t], wl.eta, wl.clip, wl.chunk)
            errs.append(abs(float(loss[s]) - l_ref))
            assert np.abs(p[s].cpu().numpy() - p_ref).sum() <= 5e-2
    assert np.mean(errs) <= TOL_BF16_LOSS_MEAN
    for s in range(wl.B):
        rel = oracle.weights_rel_frobenius(h.fast_weights(s), ref["states"][s].W, wl.fast_mats)
        assert rel <= 3e-2


@pytest.mark.parametrize("block", ["gelu", "swiglu"])
def test_decode_persistent_kernel_against_the_graph_and_the_oracle(block):
    """Decoding's next-token forward as the one persistent cooperative kernel
    (bf16, eight sequences for GELU, a decode that crosses a chunk step) against
    the captured-graph path launch for launch and against the oracle; the
    persistent path is the one that ran (with device inputs, one more logged
    launch per step than the graph path: its one kernel that stages the step's
    inputs and scores the new token takes the place of the loss kernel, and
    the forward is the other)."""
    if block == "gelu":
        wl = C.E2E_125M.replace(d=128, d_ff=512, vocab=1000, chunk=32, B=8, T=2 * 32 + 5, n_prefix=2, n_fast=2)
    else:
        wl = C.INPLACE_4B.replace(d=256, d_ff=640, vocab=3000, chunk=32, B=1, T=32 + 7, n_prefix=2)
    inp = make(wl)
    extra = 40
    long_tok = synth.sample_stream(inp["chain"], wl.seed_id, wl.B, wl.T + extra)
    tok = np.ascontiguousarray(long_tok[:, :wl.T + 1])
    runs = {}
    for name, opt in (("persist", {}), ("graph", {"no_decode_persist": 1})):
        gpu = run_gpu(wl, inp, tokens=tok, options=opt)
        h = gpu["handle"]
        p = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
        loss = torch.empty((wl.B,), dtype=torch.float32, device="cuda")
        ps, ls, logged = [], [], []
        for t in range(wl.T + 1, wl.T + extra + 1):
            h.launch_log_enable(True)
            h.decode_step(torch.from_numpy(long_tok[:, t].copy()).cuda(), p, loss)
            torch.cuda.synchronize()
            logged.append(len(h.launch_log()))
            h.launch_log_enable(False)
            ps.append(p.cpu().numpy().copy())
            ls.append(loss.cpu().numpy().copy())
        runs[name] = (np.array(ps), np.array(ls), logged, h)
    (pp, lp, np_, hp), (pg, lg, ng, hg) = runs["persist"], runs["graph"]
    # the same forward up to summation order (bf16 operands, fp32 accumulation)
    assert np.abs(pp - pg).sum(axis=-1).max() <= 2e-2
    assert np.abs(lp - lg).max() <= 2e-2
    steps_without_update = [i for i in range(extra) if np_[i] == ng[i] + 1]
    assert len(steps_without_update) >= extra - 3, (np_, ng)
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps)
    ref = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, tok)
    errs = []
    for i, t in enumerate(range(wl.T + 1, wl.T + extra + 1)):
        for s in range(wl.B):
            l_ref, p_ref = oracle.decode_step(net, ref["states"][s], long_tok[s, t], wl.eta, wl.clip, wl.chunk)
            errs.append(abs(float(lp[i, s]) - l_ref))
            assert np.abs(pp[i, s] - p_ref).sum() <= 5e-2
    assert np.mean(errs) <= TOL_BF16_LOSS_MEAN
    for s in range(wl.B):
        rel = oracle.weights_rel_frobenius(hp.fast_weights(s), ref["states"][s].W, wl.fast_mats)
        assert rel <= 3e-2


def test_settle_entry_point_after_prefill():
    """ttt_settle on its own, after a prefill of 3 chunks whose 2nd chunk ended
    with an in-prefill event: the candidate is the 3rd chunk's update; A and the
    decision for every sequence, and the weights kept or restored, against the
    oracle's Settlement on the same state (half the sequences score held-out
    text from another chain, so both outcomes occur)."""
    wl = C.SETTLE_760M.replace(d=128, d_ff=512, vocab=512, chunk=64, B=4, T=3 * 64, n_prefix=1,
                               settle_len=64, settle_every=2, eta=0.5, init_std=0.08)
    inp = make(wl)
    gpu = run_gpu(wl, inp)
    h = gpu["handle"]
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps)
    ref = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, inp["tokens"], wl.settle_every, inp["settle_q"])
    other = synth.make_chain(wl.seed_id + 100, wl.vocab, wl.chain_k, wl.chain_alpha)
    q = synth.sample_heldout(inp["chain"], wl.seed_id + 7, 1, wl.B, wl.settle_len)[0]
    q[1::2] = synth.sample_heldout(other, wl.seed_id + 7, 1, wl.B, wl.settle_len)[0][1::2]
    qd = torch.from_numpy(np.ascontiguousarray(q)).cuda()
    acc = torch.empty(wl.B, dtype=torch.uint8, device="cuda")
    A = torch.empty(wl.B, dtype=torch.float32, device="cuda")
    h.settle(qd, acc, A)
    torch.cuda.synchronize()
    A_ref = np.zeros((1, wl.B))
    acc_ref = np.zeros((1, wl.B), dtype=bool)
    for s in range(wl.B):
        A_ref[0, s], acc_ref[0, s] = oracle.settle(net, ref["states"][s], q[s])
    decided = compare_settlement({"A": A.cpu().numpy()[None], "accept": acc.cpu().numpy()[None].astype(bool)},
                                 {"A": A_ref, "accept": acc_ref}, range(wl.B), noise=5e-3)
    assert decided >= 2
    for s in range(wl.B):
        rel = oracle.weights_rel_frobenius(h.fast_weights(s), ref["states"][s].W, wl.fast_mats)
        assert rel <= 3e-2, f"seq {s}: W after settle {rel:.3e}"


def _random_mask(B, T, b, seed):
    """Random per-token mask with a fully masked chunk and a fully unmasked one."""
    rng = np.random.default_rng(seed)
    m = (rng.random((B, T)) < 0.6).astype(np.uint8)
    m[0, :b] = 0
    m[-1, b:2 * b] = 1
    return m


@pytest.mark.parametrize("case", ["bf16_gelu_fused_ce", "bf16_swiglu_hoisted", "fp32_split_ce", "fp32_rows",
                                  "fp32_rows_host", "b1_persistent", "b1_general"])
def test_source_masking_against_the_oracle(case):
    """Source Masking (a per-token mask on the chunk loss): every CE path of the
    GPU (fused dlogits, bf16x3 row CE, fp32 row CE, the per-token kernel) and
    the hoisted prefix, against the oracle's masked loop; a fully masked chunk
    leaves the weights untouched, every token is still scored."""
    if case == "bf16_gelu_fused_ce":
        wl = C.E2E_125M.replace(d=128, d_ff=512, vocab=1024, chunk=128, B=3, T=3 * 128, n_prefix=1)
    elif case == "bf16_swiglu_hoisted":
        wl = C.INPLACE_4B.replace(d=128, d_ff=384, vocab=1000, chunk=64, B=2, T=3 * 64 + 9, n_prefix=1)
    elif case == "fp32_split_ce":
        wl = C.CHUNKED_FP32.replace(d=128, d_ff=256, vocab=512, chunk=128, B=2, T=3 * 128)
    elif case.startswith("fp32_rows"):
        wl = C.CHUNKED_FP32.replace(d=72, d_ff=200, vocab=333, chunk=40, B=3, T=130, n_prefix=1)
    else:
        wl = C.TOY_BIGRAM.replace(B=2, T=200, clip=0.5)
    inp = make(wl)
    mask = _random_mask(wl.B, wl.T, wl.chunk, seed=len(case) * 7 + wl.seed_id)
    gpu = run_gpu(wl, inp, device=not case.endswith("_host"), loss_mask=mask,
                  options={"no_token_kernel": case == "b1_general"})
    ref = run_oracle(wl, inp, loss_mask=mask)
    compare(wl, gpu, ref)
    # The GPU's weights sit much nearer the masked trajectory than the unmasked one.
    plain = run_oracle(wl, inp)
    for s in range(wl.B):
        for g, r, u in zip(gpu["W"][s], ref["W"][s], plain["W"][s]):
            for k in wl.fast_mats:
                d_masked = np.linalg.norm(g[k] - r[k])
                d_plain = np.linalg.norm(g[k] - u[k])
                assert d_masked < 0.5 * d_plain, (s, k, d_masked, d_plain)


@pytest.mark.parametrize("case", ["fp32_split_ce", "bf16_gelu_hoisted", "bf16_swiglu", "b1_general"])
def test_periodic_reset_against_the_oracle(case):
    """The 8-chunk-reset mitigation at reset periods that fall inside hoisted
    chunk groups, before a ragged tail, and on the b = 1 path."""
    if case == "fp32_split_ce":
        wl = C.CHUNKED_FP32.replace(d=128, d_ff=256, vocab=512, chunk=64, B=2, T=7 * 64 + 5, reset_every=2)
    elif case == "bf16_gelu_hoisted":
        wl = C.E2E_125M.replace(d=128, d_ff=512, vocab=1024, chunk=64, B=3, T=9 * 64, n_prefix=1, reset_every=4,
                                eta=0.3)
    elif case == "bf16_swiglu":
        wl = C.INPLACE_4B.replace(d=128, d_ff=384, vocab=1000, chunk=32, B=2, T=6 * 32, n_prefix=1, reset_every=3,
                                  eta=0.5)
    else:
        wl = C.TOY_BIGRAM.replace(B=2, T=150, reset_every=8)
    inp = make(wl)
    gpu = run_gpu(wl, inp)
    ref = run_oracle(wl, inp)
    compare(wl, gpu, ref)
    if wl.n_chunks % wl.reset_every == 0:       # the run ends on a reset: W_0 exactly
        for s in range(wl.B):
            for l, blk in enumerate(gpu["W"][s]):
                for k in wl.fast_mats:
                    np.testing.assert_array_equal(blk[k], np.float32(inp["weights"]["fast"][l][k]))


def test_periodic_reset_counts_decoded_chunks():
    """A reset period that ends inside decoding: the decoded chunk's step is
    followed by the reset, and decoding goes on from W_0 like the oracle."""
    wl = C.CHUNKED_FP32.replace(d=64, d_ff=128, vocab=256, chunk=8, B=2, T=3 * 8 + 3, n_prefix=1,
                                reset_every=4, eta=0.5)
    inp = make(wl)
    extra = 14
    long_tok = synth.sample_stream(inp["chain"], wl.seed_id, wl.B, wl.T + extra)
    tok = np.ascontiguousarray(long_tok[:, :wl.T + 1])
    gpu = run_gpu(wl, inp, tokens=tok)
    h = gpu["handle"]
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps)
    ref = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, tok, reset_every=wl.reset_every)
    p = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    loss = torch.empty((wl.B,), dtype=torch.float32, device="cuda")
    for t in range(wl.T + 1, wl.T + extra + 1):
        h.decode_step(torch.from_numpy(long_tok[:, t].copy()).cuda(), p, loss)
        torch.cuda.synchronize()
        for s in range(wl.B):
            l_ref, p_ref = oracle.decode_step(net, ref["states"][s], long_tok[s, t], wl.eta, wl.clip, wl.chunk)
            assert abs(float(loss[s]) - l_ref) <= TOL["fp32"]["loss_max"]
            np.testing.assert_allclose(p[s].cpu().numpy(), p_ref, atol=1e-5)
    assert ref["states"][0].chunks_done == 5
    for s in range(wl.B):
        assert oracle.weights_rel_frobenius(h.fast_weights(s), ref["states"][s].W, wl.fast_mats) <= 1e-4


@pytest.mark.parametrize("case", ["fp32_split", "fp32_rows", "bf16_hoisted", "bf16_settle", "b1"])
def test_two_mlp_fast_blocks_against_the_oracle(case):
    """Fast blocks holding a frozen MLP before the fast one: the static MLP of
    block 0 runs in the (hoisted) prefix, the later ones forward and backward
    between the fast MLPs; every storage type, Settlement and b = 1."""
    if case == "fp32_split":
        wl = C.CHUNKED_FP32.replace(d=128, d_ff=256, vocab=512, chunk=64, B=2, T=4 * 64 + 7, n_fast=3,
                                    static_mlp=True)
    elif case == "fp32_rows":
        wl = C.CHUNKED_FP32.replace(d=72, d_ff=200, vocab=333, chunk=40, B=3, T=130, n_prefix=0,
                                    static_mlp=True)
    elif case == "bf16_hoisted":
        wl = C.E2E_125M.replace(d=128, d_ff=512, vocab=1024, chunk=64, B=3, T=5 * 64, n_prefix=1,
                                static_mlp=True, eta=0.3)
    elif case == "bf16_settle":
        wl = C.SETTLE_760M.replace(d=128, d_ff=512, vocab=1000, chunk=64, B=4, T=4 * 64, n_prefix=1,
                                   settle_len=64, settle_every=2, eta=0.5, init_std=0.08, static_mlp=True)
    else:
        wl = C.TOY_BIGRAM.replace(B=2, T=100, n_fast=2, static_mlp=True)
    inp = make(wl)
    gpu = run_gpu(wl, inp, options={"hoist_chunks": 2 if case == "bf16_hoisted" else 0})
    ref = run_oracle(wl, inp)
    # the Settlement case draws 4x larger weights (to make decisions decidable) through
    # seven bf16 MLPs: its next-token probabilities carry about twice the usual bf16 error
    compare(wl, gpu, ref, check_p=not wl.settle_every)
    if wl.settle_every:
        assert np.abs(gpu["p_next"] - ref["p_next"]).max() <= 1e-2
        compare_settlement(gpu, ref, range(wl.B), noise=5e-3)


def test_two_mlp_fast_blocks_decode():
    """Decoding through static MLPs (captured graph), across a step."""
    wl = C.CHUNKED_FP32.replace(d=64, d_ff=128, vocab=256, chunk=8, B=2, T=2 * 8 + 5, n_prefix=1, n_fast=2,
                                static_mlp=True, eta=0.5)
    inp = make(wl)
    extra = 6
    long_tok = synth.sample_stream(inp["chain"], wl.seed_id, wl.B, wl.T + extra)
    tok = np.ascontiguousarray(long_tok[:, :wl.T + 1])
    gpu = run_gpu(wl, inp, tokens=tok)
    h = gpu["handle"]
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps)
    ref = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, tok)
    p = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    loss = torch.empty((wl.B,), dtype=torch.float32, device="cuda")
    for t in range(wl.T + 1, wl.T + extra + 1):
        h.decode_step(torch.from_numpy(long_tok[:, t].copy()).cuda(), p, loss)
        torch.cuda.synchronize()
        for s in range(wl.B):
            l_ref, p_ref = oracle.decode_step(net, ref["states"][s], long_tok[s, t], wl.eta, wl.clip, wl.chunk)
            assert abs(float(loss[s]) - l_ref) <= TOL["fp32"]["loss_max"]
            np.testing.assert_allclose(p[s].cpu().numpy(), p_ref, atol=1e-5)
    for s in range(wl.B):
        assert oracle.weights_rel_frobenius(h.fast_weights(s), ref["states"][s].W, wl.fast_mats) <= 1e-4


def _attention_inputs(wl, qk_scale=8.0):
    """Seeded inputs whose query and key projections are scaled by a power of
    two (exact in every storage type), so the windowed softmax is far from
    uniform."""
    inp = make(wl)
    for a in inp["weights"]["attn"]:
        a["Wq"] = a["Wq"] * np.float32(qk_scale)
        a["Wk"] = a["Wk"] * np.float32(qk_scale)
    return inp


@pytest.mark.parametrize("case", ["fp32_split", "fp32_rows", "bf16_gelu_static", "bf16_swiglu", "b1", "masked"])
def test_sliding_window_attention_prefill_against_the_oracle(case):
    """Frozen blocks with sliding-window attention: the whole-sequence prefix
    pass (tensor-core projections, the windowed-softmax kernel) feeds every
    chunk, the ragged tail and p_{T+1}; windows shorter and longer than b,
    head dimensions below and at the warp width, every storage type."""
    mask = None
    if case in ("fp32_split", "masked"):
        wl = C.CHUNKED_FP32.replace(d=128, d_ff=256, vocab=512, chunk=64, B=2, T=4 * 64 + 5, init_std=0.1,
                                    attn_heads=4, attn_window=96)
        if case == "masked":
            mask = _random_mask(wl.B, wl.T, wl.chunk, seed=5)
    elif case == "fp32_rows":
        wl = C.CHUNKED_FP32.replace(d=72, d_ff=200, vocab=333, chunk=40, B=3, T=130, n_prefix=1, init_std=0.1,
                                    attn_heads=3, attn_window=50)
    elif case == "bf16_gelu_static":
        wl = C.E2E_125M.replace(d=128, d_ff=512, vocab=1024, chunk=64, B=3, T=5 * 64, n_prefix=2, init_std=0.1,
                                attn_heads=2, attn_window=200, static_mlp=True)
    elif case == "bf16_swiglu":
        wl = C.INPLACE_4B.replace(d=128, d_ff=384, vocab=1000, chunk=64, B=2, T=3 * 64 + 9, n_prefix=1,
                                  init_std=0.1, attn_heads=4, attn_window=64)
    else:
        wl = C.TOY_BIGRAM.replace(B=2, T=64, n_prefix=1, init_std=0.1, attn_heads=2, attn_window=8)
    inp = _attention_inputs(wl)
    gpu = run_gpu(wl, inp, loss_mask=mask)
    ref = run_oracle(wl, inp, loss_mask=mask)
    compare(wl, gpu, ref)


def _attention_launches(wl, inp, options=None):
    """Kernel classes of one prefill, logged by the library, and its outputs."""
    h = Handle.from_workload(wl, inp["weights"], options=options)
    tok = torch.from_numpy(np.ascontiguousarray(inp["tokens"])).cuda()
    losses = torch.empty((wl.B, wl.T), dtype=torch.float32, device="cuda")
    p = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    h.launch_log_enable(True)
    h.prefill(tok, losses, p)
    torch.cuda.synchronize()
    log = h.launch_log()
    h.close()
    return log, losses.cpu().numpy().astype(np.float64), p.cpu().numpy()


@pytest.mark.parametrize("dh,window,T", [(64, 1, 2 * 128 + 30), (64, 100, 3 * 128 + 17), (64, 200, 5 * 128),
                                          (128, 300, 4 * 128 + 3), (64, 4096, 3 * 128 + 1)],
                         ids=["dh64_k1", "dh64_k100_ragged", "dh64_k200", "dh128_k300", "dh64_k_beyond_T"])
def test_fused_attention_against_the_oracle_and_the_unfused_path(dh, window, T):
    """The fused tensor-core attention (bf16, one launch per frozen block, scores
    on chip): head widths 64 and 128, windows of 1, below, at and beyond a
    128-key block and beyond T, several 128-query blocks with a ragged last
    one.  Against the oracle at the bf16 tolerance, and against the three-launch
    path (score GEMM, windowed softmax, P V GEMM) it replaces; the launch log
    shows which path ran.  Weights N(0, 0.05^2) and scores sharpened by 8 (4
    for the 128-wide heads, whose dot products are twice as long)."""
    heads = 2
    wl = C.E2E_125M.replace(d=heads * dh, d_ff=2 * heads * dh, vocab=1024, chunk=64, B=2, T=T, n_prefix=2,
                            init_std=0.05, attn_heads=heads, attn_window=window)
    inp = _attention_inputs(wl, qk_scale=8.0 if dh == 64 else 4.0)
    log_f, loss_f, p_f = _attention_launches(wl, inp)
    log_u, loss_u, p_u = _attention_launches(wl, inp, options={"attn_unfused": 1})
    ref = run_oracle(wl, inp)
    rep = {"attention launches (fused, unfused)": (log_f.count("attention"), log_u.count("attention")),
           "fused mean loss err": [float(np.abs(loss_f[s] - ref["losses"][s]).mean()) for s in range(wl.B)],
           "unfused mean loss err": [float(np.abs(loss_u[s] - ref["losses"][s]).mean()) for s in range(wl.B)],
           "fused p_next max err": [float(np.abs(p_f[s] - ref["p_next"][s]).max()) for s in range(wl.B)],
           "fused vs unfused mean loss diff": float(np.abs(loss_f - loss_u).mean())}
    # per frozen block: the K/V cache fill, then one fused launch (or 3 per head)
    assert rep["attention launches (fused, unfused)"] == (wl.n_prefix * 2, wl.n_prefix * (1 + 3 * heads)), rep
    assert max(rep["fused mean loss err"]) <= TOL["bf16"]["loss_mean"], rep
    assert max(rep["fused p_next max err"]) <= 2e-3, rep
    assert max(rep["unfused mean loss err"]) <= TOL["bf16"]["loss_mean"], rep
    gpu = run_gpu(wl, inp)
    compare(wl, gpu, ref)


@pytest.mark.parametrize("case", ["window1", "window_beyond_T", "single_sequence_host", "shorter_than_a_chunk",
                                  "split_dh24"])
def test_sliding_window_attention_edge_cases(case):
    """Degenerate windows (k = 1: each position sees itself; k > T: full causal
    attention), one sequence through host buffers, a prefill shorter than one
    chunk (no step: scored tail and p_{T+1} only), and a head dimension of 24
    on the split-storage tensor-core path."""
    base = C.CHUNKED_FP32.replace(d=128, d_ff=256, vocab=512, chunk=64, B=2, T=3 * 64 + 7, n_prefix=1,
                                  init_std=0.1, attn_heads=4)
    device = True
    if case == "window1":
        wl = base.replace(attn_window=1)
    elif case == "window_beyond_T":
        wl = base.replace(attn_window=4096)
    elif case == "single_sequence_host":
        wl = base.replace(B=1, attn_window=80)
        device = False
    elif case == "shorter_than_a_chunk":
        wl = base.replace(T=50, attn_window=32)
    else:
        wl = base.replace(d=96, d_ff=192, attn_window=100)
    inp = _attention_inputs(wl)
    gpu = run_gpu(wl, inp, device=device)
    ref = run_oracle(wl, inp)
    compare(wl, gpu, ref)


@pytest.mark.parametrize("case", ["fp32_split_graph", "fp32_split_launches", "fp32_rows", "bf16_swiglu",
                                  "fp32_split_window_in_four", "bf16_window_in_eight_short_prefill"])
def test_decoding_with_attention_against_the_oracle(case):
    """Decoding after an attention prefill: each new input attends through the
    K/V cache to the window's inputs, prefill's included; the pending inputs'
    prefix rows feed the decoded chunk's step; token by token against the
    oracle across a step, captured graph and launch by launch.  Windows beyond
    256 keys are split over several blocks per (head, sequence) whose states
    are merged: four splits over a partly filled 1000-key window, and eight
    over a 2048-key window after a 5-token prefill (splits without keys)."""
    if case == "fp32_split_window_in_four":
        wl = C.CHUNKED_FP32.replace(d=128, d_ff=256, vocab=512, chunk=64, B=2, T=2 * 64 + 21, n_prefix=2,
                                    init_std=0.1, attn_heads=4, attn_window=1000, eta=0.3)
    elif case == "bf16_window_in_eight_short_prefill":
        wl = C.INPLACE_4B.replace(d=128, d_ff=384, vocab=1000, chunk=16, B=2, T=5, n_prefix=1,
                                  init_std=0.1, attn_heads=2, attn_window=2048, eta=0.5)
    elif case.startswith("fp32_split"):
        wl = C.CHUNKED_FP32.replace(d=128, d_ff=256, vocab=512, chunk=64, B=2, T=2 * 64 + 21, n_prefix=2,
                                    init_std=0.1, attn_heads=4, attn_window=96, eta=0.3)
    elif case == "fp32_rows":
        wl = C.CHUNKED_FP32.replace(d=72, d_ff=200, vocab=333, chunk=8, B=3, T=2 * 8 + 3, n_prefix=1,
                                    init_std=0.1, attn_heads=3, attn_window=6, eta=0.3)
    else:
        wl = C.INPLACE_4B.replace(d=128, d_ff=384, vocab=1000, chunk=16, B=2, T=3 * 16 + 5, n_prefix=1,
                                  init_std=0.1, attn_heads=2, attn_window=24, eta=0.5)
    extra = wl.chunk + 6 - wl.T % wl.chunk       # completes the pending chunk, then some
    inp = _attention_inputs(wl)
    long_tok = synth.sample_stream(inp["chain"], wl.seed_id, wl.B, wl.T + extra)
    tok = np.ascontiguousarray(long_tok[:, :wl.T + 1])
    gpu = run_gpu(wl, inp, tokens=tok, options={"no_decode_graph": case == "fp32_split_launches"})
    h = gpu["handle"]
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps, heads=wl.attn_heads,
                                  window=wl.attn_window)
    ref = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, tok)
    p = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    loss = torch.empty((wl.B,), dtype=torch.float32, device="cuda")
    lt, pt = (1e-4, 1e-5) if wl.dtype == "fp32" else (3e-2, 3e-3)
    for t in range(wl.T + 1, wl.T + extra + 1):
        h.decode_step(torch.from_numpy(long_tok[:, t].copy()).cuda(), p, loss)
        torch.cuda.synchronize()
        for s in range(wl.B):
            l_ref, p_ref = oracle.decode_step(net, ref["states"][s], long_tok[s, t], wl.eta, wl.clip, wl.chunk)
            assert abs(float(loss[s]) - l_ref) <= lt, (t, s, float(loss[s]), l_ref)
            assert np.abs(p[s].cpu().numpy() - p_ref).max() <= pt, (t, s)
    assert ref["states"][0].chunks_done == wl.T // wl.chunk + 1
    for s in range(wl.B):
        rel = oracle.weights_rel_frobenius(h.fast_weights(s), ref["states"][s].W, wl.fast_mats)
        assert rel <= (1e-4 if wl.dtype == "fp32" else 3e-2)


def test_attention_decoding_needs_a_prefill_after_reset():
    from chunked_next_token_ttt_b300 import TTTError
    wl = C.CHUNKED_FP32.replace(d=64, d_ff=128, vocab=256, chunk=16, B=2, T=40, n_prefix=1, attn_heads=2,
                                attn_window=16)
    inp = make(wl)
    h = run_gpu(wl, inp)["handle"]
    p = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    h.decode_step(torch.zeros(wl.B, dtype=torch.int32, device="cuda"), p)
    h.reset()
    with pytest.raises(TTTError) as e:
        h.decode_step(torch.zeros(wl.B, dtype=torch.int32, device="cuda"), p)
    assert e.value.status == 8


def test_host_and_device_buffers_agree():
    wl = C.CHUNKED_FP32.replace(d=64, d_ff=128, vocab=256, chunk=32, B=2, T=100, n_prefix=1)
    inp = make(wl)
    a = run_gpu(wl, inp, device=True)
    b = run_gpu(wl, inp, device=False)
    np.testing.assert_array_equal(a["losses"], b["losses"])
    np.testing.assert_array_equal(a["p_next"], b["p_next"])


def test_sequences_are_independent_on_gpu():
    wl = C.CHUNKED_FP32.replace(d=64, d_ff=128, vocab=256, chunk=32, B=3, T=96, n_prefix=1)
    inp = make(wl)
    full = run_gpu(wl, inp)
    one = run_gpu(wl, inp, tokens=inp["tokens"][1:2])
    np.testing.assert_array_equal(one["losses"][0], full["losses"][1])
    for l in range(wl.n_fast):
        for k in wl.fast_mats:
            np.testing.assert_array_equal(one["W"][0][l][k], full["W"][1][l][k])


@pytest.mark.parametrize("graph", ["1", "0"], ids=["graph", "launches"])
def test_decode_completes_the_ragged_chunk_and_continues(graph):
    """Decoding after a prefill with a ragged tail: every step's loss and p_next
    against the oracle, through the captured next-token graph and launch by
    launch."""
    wl = C.CHUNKED_FP32.replace(d=64, d_ff=128, vocab=256, chunk=16, B=2, T=16 * 3 + 5, n_prefix=1)
    inp = make(wl)
    extra = 16 + 11 + 16
    chain = inp["chain"]
    long_tok = synth.sample_stream(chain, wl.seed_id, wl.B, wl.T + extra)
    tok = np.ascontiguousarray(long_tok[:, :wl.T + 1])
    gpu = run_gpu(wl, inp, tokens=tok, options={"no_decode_graph": graph == "0"})
    h = gpu["handle"]
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps)
    ref = oracle.prefill(net, wl.eta, wl.clip, wl.chunk, tok)
    p = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device="cuda")
    loss = torch.empty((wl.B,), dtype=torch.float32, device="cuda")
    for t in range(wl.T + 1, wl.T + extra + 1):
        x = torch.from_numpy(long_tok[:, t].copy()).cuda()
        if t == wl.T + 8:
            # a state round trip drops the cached next-token softmax: this step
            # scores its token with a forward pass instead
            h.set_state(h.get_state())
        h.decode_step(x, p, loss)
        torch.cuda.synchronize()
        for s in range(wl.B):
            l_ref, p_ref = oracle.decode_step(net, ref["states"][s], long_tok[s, t], wl.eta, wl.clip, wl.chunk)
            assert abs(float(loss[s]) - l_ref) <= 1e-4
            assert np.abs(p[s].cpu().numpy() - p_ref).max() <= 1e-5
    for s in range(wl.B):
        rel = oracle.weights_rel_frobenius(h.fast_weights(s), ref["states"][s].W, wl.fast_mats)
        assert rel <= 1e-4


def test_state_roundtrip_and_reset():
    wl = C.CHUNKED_FP32.replace(d=64, d_ff=128, vocab=256, chunk=16, B=2, T=40, n_prefix=1)
    inp = make(wl)
    gpu = run_gpu(wl, inp)
    h = gpu["handle"]
    blob = h.get_state()
    W_before = h.fast_weights(1)
    h.reset()
    W0 = h.fast_weights(1)
    for l in range(wl.n_fast):
        np.testing.assert_array_equal(W0[l]["W1"], inp["weights"]["fast"][l]["W1"])
    h.set_state(blob)
    W_after = h.fast_weights(1)
    for l in range(wl.n_fast):
        for k in wl.fast_mats:
            np.testing.assert_array_equal(W_after[l][k], W_before[l][k])


def test_bad_arguments_raise_status_codes():
    from chunked_next_token_ttt_b300 import TTTError
    wl = C.CHUNKED_FP32.replace(d=64, d_ff=128, vocab=256, chunk=16, B=2, T=32, n_prefix=1)
    inp = make(wl)
    gpu = run_gpu(wl, inp)
    h = gpu["handle"]
    bad = torch.zeros((3, 33), dtype=torch.int32, device="cuda")
    losses = torch.empty((3, 32), device="cuda")
    with pytest.raises(TTTError) as e:
        h.prefill(bad, losses)
    assert e.value.status == 2
    with pytest.raises(TTTError) as e:
        wl2 = wl.replace(block="swiglu", fast_mats=("Wg", "Wd"))
        from chunked_next_token_ttt_b300 import Handle
        Handle.from_workload(wl2, synth.make_weights(wl2))
    assert e.value.status == 7
