"""Benchmark: TTT prefill tokens/s (forward + backward + clipped update) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

One step is one full prefill of the workload's B sequences of T tokens: every
chunk runs the frozen prefix, the fast blocks forward, RMSNorm, the LM head, the
fused cross-entropy, the backward to the fast weights and the clipped SGD step
(and, for the Settlement workload, the Settlement events).  The default workload
is the largest: the 760M-like stream, B = 8, T = 131072, one clipped step per
1024-token chunk on the last three MLP blocks, Settlement after every 8th chunk.
Inputs (seeded synthetic Markov tokens, N(0, 0.02^2) weights) are resident on
the device before the timed region; L2 is flushed (a 512 MB write) before every
timed step, outside the step's events.  The timed steps carry no profiling
events: the per-class times and the dominant class's launch times come from
separate, untimed profiled steps.  `e2e` times the same call with pinned host
buffers (tokens and held-out chunks in; losses, p_{T+1}, scores and decisions
out) through the C ABI.

With --gpus N under torchrun every rank runs its own B sequences (weak scaling:
the sequences are independent, so no collective is on the data path); rank 0
prints the max-over-ranks time.  --impl reference times the float64 CPU oracle
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402
from synth import configs as C  # noqa: E402

METRIC = "TTT prefill tokens/s (fwd+bwd+update) on 1 B300; % of chunk roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "sm_max_mhz": 2032.0}


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")

# the sources that define each family of kernels (kernel identity for counters
# taken by a profiler: a change elsewhere leaves a family's counters valid)
KERNEL_FAMILIES = {
    "gemm": ("common.cuh", "epilogue.cuh", "gemm.h", "gemm.cu", "gemm_tc.cu", "gemm_tc_kernel.cuh", "gemm_tc_kk.cu",
             "gemm_tc_km.cu", "gemm_tc_mk.cu", "gemm_tc_mm.cu", "gemm_simt.cu", "gemm_small.cu"),
    "elementwise": ("common.cuh", "kernels.h", "kernels.cu", "clip_sgd.h", "clip_sgd.cu"),
    "attention": ("common.cuh", "kernels.h", "gemm_tc_kernel.cuh", "attention.cu", "attention_fused.cu"),
    "token": ("common.cuh", "kernels.h", "token_step.cu"),
}


def class_family(kernel_class):
    if kernel_class.startswith("gemm_"):
        return "gemm"
    return {"attention": "attention", "token_step": "token"}.get(kernel_class, "elementwise")


def source_hash(family):
    """SHA-256 over the sources of one kernel family."""
    import hashlib
    hsh = hashlib.sha256()
    for name in sorted(KERNEL_FAMILIES[family]):
        hsh.update(name.encode())
        with open(os.path.join(ROOT, "chunked_next_token_ttt_b300", "csrc", name), "rb") as fh:
            hsh.update(fh.read())
    return hsh.hexdigest()[:16]


def profiled_traffic(workload, kernel_class):
    """DRAM bytes per launch of a kernel class from profiles/traffic.json (ncu's
    dram__bytes_read.sum + dram__bytes_write.sum per launch), or None when there
    is none or the class's kernel family changed since the counters were taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        entry = json.load(f).get(workload, {}).get(kernel_class)
    if not entry or entry.get("source_hash") != source_hash(class_family(kernel_class)):
        return None
    return float(entry["dram_bytes_per_launch"])


def choose_peak(pk, clocks, timed_s):
    """The bf16 denominator for a class timed inside the measured steps: the
    burst peak when the timed region is sub-second at the maximum clock with no
    power-cap sample, the sustained (power-capped) peak otherwise."""
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    at_max = sm is not None and smax and sm >= 0.97 * smax
    if timed_s < 1.0 and at_max and "sw_power_cap" not in clocks.get("reasons", []):
        return pk["bf16_tflops"], "burst"
    return pk.get("bf16_tflops_sustained", pk["bf16_tflops"]), "sustained"


def peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        p["source"] = "measured"
        return p
    p = dict(FALLBACK)
    p["source"] = "fallback"
    return p


# ---------------------------------------------------------------- accounting
def chunk_flops(wl, rows=None):
    """Dense-contraction FLOPs of one chunk step for all B sequences, by class."""
    M = wl.B * (wl.chunk if rows is None else rows)
    mdf = 2.0 * M * wl.d * wl.d_ff
    per = {}
    if wl.block == "gelu":
        per["gemm_prefix"] = wl.n_prefix * 2 * mdf
        per["gemm_fast_fwd"] = wl.n_fast * 2 * mdf
        per["gemm_bwd_dx"] = (2 * wl.n_fast - 1) * mdf
        per["gemm_dw"] = 2 * wl.n_fast * mdf
        if wl.static_mlp:
            # fast block 0's static MLP joins the prefix; the later ones run forward and dX backward
            per["gemm_prefix"] += 2 * mdf
            per["gemm_fast_fwd"] += (wl.n_fast - 1) * 2 * mdf
            per["gemm_bwd_dx"] += (wl.n_fast - 1) * 2 * mdf
    else:
        per["gemm_prefix"] = wl.n_prefix * 3 * mdf
        per["gemm_fast_fwd"] = wl.n_fast * 3 * mdf
        per["gemm_bwd_dx"] = 0.0
        per["gemm_dw"] = wl.n_fast * mdf
    per["gemm_head"] = 2.0 * M * wl.d * wl.vocab
    per["gemm_head_bwd"] = 2.0 * M * wl.d * wl.vocab
    if wl.chunk == 1:
        # the persistent per-token kernel: W1 and W2 forward, head, dy = U^T dl,
        # da = W2^T dh, and the two outer-product updates (2 FLOP per FMA)
        per["token_step"] = wl.B * (10.0 * wl.d * wl.d_ff + 4.0 * wl.d * wl.vocab)
    if wl.attn_heads:
        # the Q|K|V and Wo projections of every frozen block, and the windowed
        # attention (Q K^T and P V: 4 d FLOP per (query, key) pair), as a
        # per-chunk share of the whole-sequence pass over x_0 .. x_T
        per["gemm_prefix"] += wl.n_prefix * 8.0 * M * wl.d * wl.d
        per["attention"] = wl.n_prefix * 4.0 * wl.d * wl.B * attention_pairs(wl.T + 1, wl.attn_window) / wl.n_chunks
    return per


def attention_pairs(n, k):
    """Number of (query, key) pairs of a sliding window k over n positions."""
    m = min(n, k)
    return m * (m + 1) // 2 + (n - m) * k




def chunk_flops_fwd_one(wl):
    """FLOPs of the p_{T+1} forward (one row per sequence) by class."""
    f = chunk_flops(wl, rows=1)
    return {k: f[k] for k in ("gemm_prefix", "gemm_fast_fwd", "gemm_head")}


def chunk_bytes(wl):
    """Algorithmic HBM bytes of one chunk step, by class (see DESIGN: each
    tensor read or written once; the V-wide logits buffer counted once in
    the CE class as read + write)."""
    es = 2 if wl.dtype == "bf16" else 4
    M = wl.B * wl.chunk
    nf = len(wl.fast_mats) * wl.n_fast
    params = nf * wl.B * wl.d * wl.d_ff
    return {
        "ce_fused": 2.0 * M * wl.vocab * es,
        "clip_sgd_update": params * (4 + 4 + 4 + es),   # read W32, dW; write W32 and the operand copy
        "rmsnorm_fwd": M * wl.d * (4 + es),
        "rmsnorm_bwd": M * wl.d * (4 * 3 + 4 + es),
        "embed": M * wl.d * (es + 4 + es),
        "grad_norm": 0.0,
    }


def settle_flops(wl):
    """FLOPs of one Settlement event for all B sequences, by class: one pass of
    the frozen prefix over the held-out chunks (shared by both scores), then
    the fast blocks and the LM head forward twice (committed and current)."""
    if not wl.settle_every:
        return {}
    f = chunk_flops(wl, rows=wl.settle_len)
    return {"gemm_prefix": f["gemm_prefix"], "gemm_fast_fwd": 2 * f["gemm_fast_fwd"], "gemm_head": 2 * f["gemm_head"]}


def step_flops(wl):
    """Dense-contraction FLOPs of one whole prefill step (every chunk, every
    Settlement event and the p_{T+1} forward), by kernel class."""
    out = {k: v * wl.n_chunks for k, v in chunk_flops(wl).items()}
    for k, v in settle_flops(wl).items():
        out[k] = out.get(k, 0.0) + v * wl.n_settle_events
    for k, v in chunk_flops_fwd_one(wl).items():
        out[k] = out.get(k, 0.0) + v
    return out


def chunk_roofline_seconds(wl, pk):
    """Roofline time of one chunk step, max(FLOPs / bf16 burst peak, bytes / HBM
    peak), with the Settlement events' FLOPs spread over the chunks."""
    fl = sum(chunk_flops(wl).values())
    if wl.settle_every:
        fl += sum(settle_flops(wl).values()) / wl.settle_every
    es = 2 if wl.dtype == "bf16" else 4
    M = wl.B * wl.chunk
    nf = len(wl.fast_mats) * wl.n_fast
    params = nf * wl.B * wl.d * wl.d_ff
    # weights read once per chunk (frozen prefix, head, fast masters r+w), token ids, losses,
    # and the block inputs written and read once
    n_frozen_blocks = wl.n_prefix + (wl.n_fast if wl.static_mlp else 0)
    frozen = (n_frozen_blocks * (2 if wl.block == "gelu" else 3) * wl.d * wl.d_ff + wl.vocab * wl.d) * es
    by = frozen + params * 8 + M * 8 + M * wl.d * es * 2
    return max(fl / (pk["bf16_tflops"] * 1e12), by / (pk["hbm_gbs"] * 1e9)), fl, by


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.path = tempfile.mktemp(suffix=".csv")
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(wl, inp, n_seq, n_chunks):
    import oracle
    net = oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps,
                                  heads=wl.attn_heads, window=wl.attn_window)
    tok = inp["tokens"][:n_seq, :n_chunks * wl.chunk + 1]
    t0 = time.perf_counter()
    oracle.prefill(net, wl.eta, wl.clip, wl.chunk, tok)
    dt = time.perf_counter() - t0
    return n_seq * n_chunks * wl.chunk / dt, dt


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


# ---------------------------------------------------------------- ranks
def rank_inputs(wl, rank):
    """Seeded inputs of one rank: every rank owns its own B sequences (the
    sequences are independent), so rank r > 0 draws its streams with a seed
    shifted by 1000 r; weights and the chain are shared."""
    inp = synth.make_inputs(wl)
    if rank:
        inp["tokens"] = synth.sample_stream(inp["chain"], wl.seed_id + 1000 * rank, wl.B, wl.T)
    return inp


def max_over_ranks(x, world, device):
    """Largest x over the ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- arms
def workload_config(wl, world):
    """The workload keys of the JSON line's config, the same for both arms."""
    cfg = {"workload": wl.name, "B": wl.B, "T": wl.T, "chunk": wl.chunk, "d": wl.d, "d_ff": wl.d_ff,
           "vocab": wl.vocab, "n_prefix": wl.n_prefix, "n_fast": wl.n_fast, "tokens_per_step": wl.B * wl.T * world}
    if wl.attn_heads:
        cfg.update(attn_heads=wl.attn_heads, attn_window=wl.attn_window)
    return cfg


def measured_config(wl, world, chunk_frac, t_roof, pk):
    """The config of our arm's line: the workload keys plus how it was measured."""
    return dict(workload_config(wl, world), l2="flushed (512 MB write) before every step",
                chunk_roofline_frac=chunk_frac, chunk_roofline_ms=t_roof * 1e3,
                peaks={"bf16_tflops": pk["bf16_tflops"], "hbm_gbs": pk["hbm_gbs"], "source": pk["source"]})


def run_reference(args, wl, rank):
    if rank != 0:
        return
    inp = synth.make_inputs(wl.replace(B=1))
    # chunks per step: at most 4, and about 8e11 FLOP (a few seconds of the
    # float64 oracle on host cores) so that the whole run ends in minutes
    per_chunk = sum(chunk_flops(wl).values()) / wl.B
    n_chunks = max(1, min(wl.n_chunks, 4, int(8e11 // per_chunk)))
    for _ in range(args.warmup):
        oracle_sample(wl, inp, 1, 1)
    vals, times = [], []
    for _ in range(args.steps):
        v, dt = oracle_sample(wl, inp, 1, n_chunks)
        vals.append(v)
        times.append(dt)
    v = len(vals) * n_chunks * wl.chunk / sum(times)
    sample = f"1 sequence x {n_chunks} chunk(s) ({n_chunks * wl.chunk} tokens) of {wl.name} per step"
    if wl.settle_every:
        sample += " (no Settlement event falls inside the sample)"
    line = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": workload_config(wl, args.gpus),
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, wl, rank, world, local_rank):
    import torch

    from chunked_next_token_ttt_b300 import Handle, kernel_classes

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pk = peaks()
    inp = rank_inputs(wl, rank)
    h = Handle.from_workload(wl, inp["weights"], options=args.options)
    storage = h.operand_storage()
    tok = torch.from_numpy(inp["tokens"]).to(dev)
    losses = torch.empty((wl.B, wl.T), dtype=torch.float32, device=dev)
    p = torch.empty((wl.B, wl.vocab), dtype=torch.float32, device=dev)
    n_ev = wl.n_settle_events
    q = torch.from_numpy(inp["settle_q"]).to(dev) if n_ev else None
    acc = torch.empty((max(1, n_ev), wl.B), dtype=torch.uint8, device=dev)
    A = torch.empty((max(1, n_ev), wl.B), dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream(dev)
    classes = kernel_classes()

    def step():
        h.prefill(tok, losses, p, q, acc if n_ev else None, A if n_ev else None)

    # warm-up; the first step logs the class of every launch
    seen = []
    for w in range(args.warmup):
        if w == 0:
            h.launch_log_enable(True)
        step()
        if w == 0:
            log = h.launch_log()
            h.launch_log_enable(False)
            seen = [c for c in classes if c in set(log)]
            if args.launch_log:
                with open(args.launch_log, "w") as f:
                    f.write("\n".join(log) + "\n")
    torch.cuda.synchronize(dev)

    # timed region: K steps with no profiling events, L2 flushed before each
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    launches = 0
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(st)
            step()
            ev[i][1].record(st)
            launches += h.last_launch_count()
        torch.cuda.synchronize(dev)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    tokens = wl.B * wl.T * world * args.steps
    value = tokens / (total_ms / 1e3)
    clk_sum = clk.summary()

    # per-class device time: one untimed step per class, its launches bracketed by events
    per_class = {}
    for name in seen or classes:
        h.profile_enable(classes.index(name))
        flush.zero_()
        step()
        n, ms = h.profile_read()
        if n:
            per_class[name] = (n, ms)
    h.profile_enable(-1)
    dom = max(per_class, key=lambda k: per_class[k][1])
    # the dominant class's launch times over further untimed steps
    dom_steps = max(1, min(3, args.steps))
    h.profile_enable(classes.index(dom))
    for _ in range(dom_steps):
        flush.zero_()
        step()
    dom_n, dom_ms = h.profile_read()
    h.profile_enable(-1)

    # end to end: pinned host buffers through the C ABI
    tok_h = torch.from_numpy(inp["tokens"]).pin_memory()
    loss_h = torch.empty((wl.B, wl.T), dtype=torch.float32).pin_memory()
    p_h = torch.empty((wl.B, wl.vocab), dtype=torch.float32).pin_memory()
    q_h = torch.from_numpy(inp["settle_q"]).pin_memory() if n_ev else None
    acc_h = torch.empty((max(1, n_ev), wl.B), dtype=torch.uint8).pin_memory()
    A_h = torch.empty((max(1, n_ev), wl.B), dtype=torch.float32).pin_memory()
    h.prefill(tok_h, loss_h, p_h, q_h, acc_h if n_ev else None, A_h if n_ev else None)
    e2e_t = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        h.prefill(tok_h, loss_h, p_h, q_h, acc_h if n_ev else None, A_h if n_ev else None)
        e2e_t.append(time.perf_counter() - t0)
    e2e_total = max_over_ranks(sum(e2e_t), world, dev)
    e2e_value = tokens / e2e_total
    h2d = tok_h.numel() * 4 + (q_h.numel() * 4 if n_ev else 0)
    d2h = loss_h.numel() * 4 + p_h.numel() * 4 + (n_ev * wl.B * 5 if n_ev else 0)

    # decoding: one full cycle of b steps (one TTT update) after the prefill,
    # device buffers through ttt_decode_step; every call scores the new token,
    # steps when b are pending and returns p_{t+1}
    dec = None
    if not args.no_decode and wl.settle_every == 0:
        h.prefill(tok, losses, p)
        xs = torch.from_numpy(np.ascontiguousarray(inp["tokens"][:, 1:wl.chunk + 1].T)).to(dev)   # [b, B]
        dloss = torch.empty((wl.B,), dtype=torch.float32, device=dev)
        for t in range(min(3, wl.chunk)):
            h.decode_step(xs[t], p, dloss)
        h.prefill(tok, losses, p)
        dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(wl.chunk)]
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for t in range(wl.chunk):
            dev_ev[t][0].record(st)
            h.decode_step(xs[t], p, dloss)
            dev_ev[t][1].record(st)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        dms = sum(a.elapsed_time(b) for a, b in dev_ev)
        es = 2 if wl.dtype == "bf16" else 4
        nf = len(wl.fast_mats) * wl.n_fast
        frozen = ((wl.n_prefix + (wl.n_fast if wl.static_mlp else 0)) * (2 if wl.block == "gelu" else 3)
                  * wl.d * wl.d_ff
                  + wl.n_fast * ((2 if wl.block == "gelu" else 3) - len(wl.fast_mats)) * wl.d * wl.d_ff
                  + wl.vocab * wl.d) * es
        fast = wl.B * nf * wl.d * wl.d_ff * es
        by = frozen + fast + wl.B * wl.vocab * 4 * 2
        if wl.attn_heads:
            # the attention weights and the fp32 K/V cache of every frozen block's window
            by += wl.n_prefix * (4 * wl.d * wl.d * es + wl.B * 2 * min(wl.T + 1, wl.attn_window) * wl.d * 4)
        bound = wl.B / (by / (pk["hbm_gbs"] * 1e9))
        v = wl.B * wl.chunk / (dms / 1e3)
        dec = {"tokens_per_s": v, "tokens_per_s_wall": wl.B * wl.chunk / wall, "steps": wl.chunk,
               "ms_per_step": dms / wl.chunk,
               "weight_stream_bound_tokens_per_s": bound, "frac_of_bound": v / bound,
               "note": "b decode steps (one TTT update amortised); bound = every weight read once per step"}

    # roofline of the dominant class: its algorithmic work per launch over its
    # average launch time in the untimed profiled steps
    sflops = step_flops(wl)
    byts = chunk_bytes(wl)
    timed_s = total_ms / 1e3
    dom_avg_s = dom_ms / 1e3 / max(1, dom_n)
    if dom_n % dom_steps:
        raise RuntimeError("profiled launches are not a whole number per step")
    launches_per_step_dom = dom_n / dom_steps
    fma_peak = 148 * 128 * 2 * pk.get("sm_max_mhz", 2032.0) * 1e6 / 1e12
    if dom in sflops:
        per_launch = sflops[dom] / launches_per_step_dom
        achieved = per_launch / dom_avg_s / 1e12
        if dom == "token_step":
            # one CTA per sequence: the FP32 FMA lanes of the SMs it occupies
            sms = min(wl.B, 148)
            roof = {"bound": "alu", "achieved": achieved, "peak": fma_peak * sms / 148, "unit": "TFLOP/s",
                    "peak_source": f"fp32 FMA: {sms} SM(s) x 128 lanes x 2 x max SM clock"}
        elif storage == "f32":
            # fp32 FMA on the SIMT pipes: 148 SMs x 128 lanes x 2 FLOP x max SM clock
            roof = {"bound": "alu", "achieved": achieved, "peak": fma_peak, "unit": "TFLOP/s",
                    "peak_source": "fp32 FMA: 148 SMs x 128 lanes x 2 x max SM clock"}
        else:
            peak, regime = choose_peak(pk, clk_sum, timed_s)
            if regime == "burst":
                why = "sub-second timed region at max clock, no power cap"
            else:
                why = f"{timed_s:.1f} s timed region, median {clk_sum.get('sm_mhz')} MHz"
            src = f"{pk['source']} bf16 {regime} ({why})"
            if storage == "bf16x3":
                peak /= 3.0
                src += " / 3 (bf16x3: three bf16 products per product)"
            roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "peak_source": src}
    else:
        per_launch = byts.get(dom, 0.0) * wl.n_chunks / max(1e-9, launches_per_step_dom)
        achieved = per_launch / dom_avg_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "peak_source": f"{pk['source']} copy bandwidth"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = dom
    roof["traffic"] = profiled_traffic(wl.name, dom)
    roof["traffic_source"] = ("profiles/traffic.json (ncu dram__bytes_read.sum + dram__bytes_write.sum per launch); "
                              "null when the kernels changed since")
    roof["launches_per_step"] = launches_per_step_dom
    roof["avg_launch_ms"] = dom_avg_s * 1e3
    roof["timing"] = f"CUDA events around each launch of the class in {dom_steps} untimed step(s)"
    t_roof, fl_chunk, by_chunk = chunk_roofline_seconds(wl, pk)
    chunk_frac = t_roof * wl.n_chunks / (total_ms / 1e3 / args.steps)

    cfg = measured_config(wl, world, chunk_frac, t_roof, pk)
    cfg["arith"] = storage
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": storage,
            "data": "synthetic",
            "config": cfg,
            "roofline": roof, "clocks": clk_sum,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "decode": dec,
            "per_class_ms": {k: round(v[1], 3) for k, v in sorted(per_class.items(), key=lambda kv: -kv[1][1])}}
    if n_ev:
        line["settlement"] = {"events": n_ev, "accepted": int(acc.cpu().numpy()[:n_ev].sum()),
                              "decisions": n_ev * wl.B}
    if rank == 0 and not args.no_cpu_baseline:
        n_chunks = 12 if wl.name == C.CHUNKED_FP32.name else 2
        n_seq = min(wl.B, 4)
        v, dt = oracle_sample(wl, inp, n_seq, min(n_chunks, wl.n_chunks))
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                                "sample": f"{n_seq} sequences x {min(n_chunks, wl.n_chunks)} chunks of "
                                          f"{wl.name} ({dt:.1f} s)"}
    h.close()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=C.SETTLE_760M.name, choices=list(C.BY_NAME))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode measurement")
    ap.add_argument("--launch-log", default=None,
                    help="write the kernel class of every launch of the first prefill to this file")
    ap.add_argument("--T", type=int, default=None,
                    help="tokens per sequence instead of the workload's (small cases for profiler captures)")
    ap.add_argument("--B", type=int, default=None,
                    help="sequences instead of the workload's (small cases for profiler captures)")
    ap.add_argument("--option", action="append", default=[], metavar="NAME=VALUE",
                    help="a ttt_options field of the handle (e.g. hoist_chunks=2), for profiler captures")
    args = ap.parse_args()
    wl = C.BY_NAME[args.workload]
    if args.T is not None:
        wl = wl.replace(T=args.T)
    if args.B is not None:
        wl = wl.replace(B=args.B)
    args.options = {k: int(v) for k, v in (o.split("=", 1) for o in args.option)}
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, wl, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, wl, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
