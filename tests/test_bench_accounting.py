"""The benchmark's algorithmic accounting (CPU only): the FLOPs and bytes it
divides by measured times, checked against direct counts on small shapes."""
import numpy as np

import bench
from synth import configs as C


def test_attention_pairs_count_the_window():
    """(query, key) pairs of a sliding window k over n positions, by brute force."""
    for n in (1, 5, 17, 64):
        for k in (1, 3, 16, 100):
            brute = sum(1 for t in range(n) for s in range(n) if t - k < s <= t)
            assert bench.attention_pairs(n, k) == brute


def test_gelu_chunk_flops_by_counting_the_gemms():
    """Per chunk: prefix 2 GEMMs per block, fast forward 2 per block, backward
    dX 2 per block but the first block's input gradient, dW 2 per block, head
    forward and backward: each 2 M N K."""
    wl = C.CHUNKED_FP32.replace(d=8, d_ff=24, vocab=40, chunk=4, B=3, n_prefix=2, n_fast=3)
    M, d, f, V = wl.B * wl.chunk, wl.d, wl.d_ff, wl.vocab
    g = lambda m, n, k: 2.0 * m * n * k
    fl = bench.chunk_flops(wl)
    assert fl["gemm_prefix"] == 2 * (g(M, f, d) + g(M, d, f))
    assert fl["gemm_fast_fwd"] == 3 * (g(M, f, d) + g(M, d, f))
    assert fl["gemm_bwd_dx"] == 3 * g(M, f, d) + 2 * g(M, d, f)
    assert fl["gemm_dw"] == 3 * (g(d, f, M) + g(f, d, M))
    assert fl["gemm_head"] == fl["gemm_head_bwd"] == g(M, V, d)


def test_static_mlps_and_attention_add_their_gemms():
    wl = C.CHUNKED_FP32.replace(d=8, d_ff=24, vocab=40, chunk=4, B=3, T=20, n_prefix=2, n_fast=3)
    M, d, f = wl.B * wl.chunk, wl.d, wl.d_ff
    base = bench.chunk_flops(wl)
    st = bench.chunk_flops(wl.replace(static_mlp=True))
    assert st["gemm_prefix"] - base["gemm_prefix"] == 2 * 2.0 * M * d * f
    assert st["gemm_fast_fwd"] - base["gemm_fast_fwd"] == 2 * 2 * 2.0 * M * d * f
    assert st["gemm_bwd_dx"] - base["gemm_bwd_dx"] == 2 * 2 * 2.0 * M * d * f
    at = bench.chunk_flops(wl.replace(attn_heads=2, attn_window=6))
    assert at["gemm_prefix"] - base["gemm_prefix"] == wl.n_prefix * 4 * 2.0 * M * d * d
    pairs = sum(1 for t in range(wl.T + 1) for s in range(wl.T + 1) if t - 6 < s <= t)
    np.testing.assert_allclose(at["attention"] * wl.n_chunks, wl.n_prefix * 4.0 * d * wl.B * pairs)


def test_update_bytes_per_parameter():
    """Clip + SGD reads the fp32 master and dW, writes the master and the
    operand copy (2 B bf16, 4 B for two bf16 planes or fp32)."""
    for dtype, es in (("bf16", 2), ("fp32", 4)):
        wl = C.E2E_125M.replace(d=8, d_ff=16, chunk=4, B=2, n_fast=3, dtype=dtype)
        params = len(wl.fast_mats) * wl.n_fast * wl.B * wl.d * wl.d_ff
        assert bench.chunk_bytes(wl)["clip_sgd_update"] == params * (12 + es)


def test_both_arms_name_the_same_workload_config():
    """The reference arm's config keys are a subset of ours with equal values,
    and ours adds only how it was measured."""
    wl = C.SWA_125M
    pk = bench.peaks()
    ref = bench.workload_config(wl, 1)
    ours = bench.measured_config(wl, 1, 0.1, 0.002, pk)
    assert all(ours[k] == v for k, v in ref.items())
    assert set(ours) - set(ref) == {"l2", "chunk_roofline_frac", "chunk_roofline_ms", "peaks"}
    assert ref["attn_window"] == 2048 and ref["tokens_per_step"] == wl.B * wl.T
    t_roof, fl, by = bench.chunk_roofline_seconds(C.CHUNKED_FP32, pk)
    assert t_roof > 0 and fl > 0 and by > 0


def test_settlement_flops_count_one_prefix_and_two_forwards():
    """A Settlement event runs the frozen prefix over the held-out chunks once
    and the fast blocks and the head forward twice (committed and current
    weights); a whole step adds every chunk, every event and p_{T+1}."""
    wl = C.SETTLE_760M.replace(d=8, d_ff=24, vocab=40, chunk=4, B=3, T=64, n_prefix=2, n_fast=3,
                               settle_every=2, settle_len=6)
    Mq, d, f, V = wl.B * wl.settle_len, wl.d, wl.d_ff, wl.vocab
    g = lambda m, n, k: 2.0 * m * n * k
    sf = bench.settle_flops(wl)
    assert sf["gemm_prefix"] == 2 * (g(Mq, f, d) + g(Mq, d, f))
    assert sf["gemm_fast_fwd"] == 2 * 3 * (g(Mq, f, d) + g(Mq, d, f))
    assert sf["gemm_head"] == 2 * g(Mq, V, d)
    step = bench.step_flops(wl)
    ch, one = bench.chunk_flops(wl), bench.chunk_flops(wl, rows=1)
    assert wl.n_chunks == 16 and wl.n_settle_events == 8
    assert step["gemm_prefix"] == 16 * ch["gemm_prefix"] + 8 * sf["gemm_prefix"] + one["gemm_prefix"]
    assert step["gemm_dw"] == 16 * ch["gemm_dw"]
    assert bench.settle_flops(wl.replace(settle_every=0)) == {}


def test_peak_choice_follows_the_clock_record():
    pk = {"bf16_tflops": 1700.0, "bf16_tflops_sustained": 1300.0}
    fast = {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": []}
    assert bench.choose_peak(pk, fast, 0.4) == (1700.0, "burst")
    assert bench.choose_peak(pk, fast, 3.0) == (1300.0, "sustained")
    assert bench.choose_peak(pk, dict(fast, reasons=["sw_power_cap"]), 0.4) == (1300.0, "sustained")
    assert bench.choose_peak(pk, dict(fast, sm_mhz=1500.0), 0.4) == (1300.0, "sustained")
