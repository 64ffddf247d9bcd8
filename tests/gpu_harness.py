"""Shared helpers of the GPU parity tests: run libttt and the oracle on the same
seeded inputs and compare them with the stated tolerances.

Tolerances (fp32-accurate workloads): per-token loss |err| <= 1e-4 and final
fast-weight relative Frobenius error <= 1e-4.  bf16 workloads: mean per-token
|err| <= 2e-2 and relative Frobenius error <= 3e-2.  Settlement decisions must
agree exactly wherever the oracle's |A| exceeds the measured noise of A.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from chunked_next_token_ttt_b300 import Handle

TOL = {"fp32": {"loss_max": 1e-4, "w_rel": 1e-4}, "bf16": {"loss_mean": 2e-2, "w_rel": 3e-2}}


def make(wl):
    return synth.make_inputs(wl)


def oracle_net(wl, inp):
    return oracle.Net.from_weights(inp["weights"], wl.block, wl.fast_mats, wl.rms_eps,
                                   heads=wl.attn_heads, window=wl.attn_window)


def run_oracle(wl, inp, seqs=None, tokens=None, q=None, loss_mask=None):
    net = oracle_net(wl, inp)
    tok = inp["tokens"] if tokens is None else tokens
    sq = inp["settle_q"] if q is None else q
    return oracle.prefill(net, wl.eta, wl.clip, wl.chunk, tok, wl.settle_every,
                          sq if wl.settle_every else None, seqs=seqs, loss_mask=loss_mask,
                          reset_every=wl.reset_every)


def run_gpu(wl, inp, device=True, tokens=None, q=None, handle=None, loss_mask=None, options=None):
    tok = inp["tokens"] if tokens is None else tokens
    sq = inp["settle_q"] if q is None else q
    B, T1 = tok.shape
    h = handle or Handle.from_workload(wl, inp["weights"], B=B, options=options)
    n_ev = ((T1 - 1) // wl.chunk) // wl.settle_every if wl.settle_every else 0
    if device:
        t = torch.from_numpy(np.ascontiguousarray(tok)).cuda()
        losses = torch.empty((B, T1 - 1), dtype=torch.float32, device="cuda")
        p = torch.empty((B, wl.vocab), dtype=torch.float32, device="cuda")
        qd = torch.from_numpy(np.ascontiguousarray(sq[:n_ev])).cuda() if n_ev else None
        A = torch.empty((max(n_ev, 1), B), dtype=torch.float32, device="cuda")
        acc = torch.empty((max(n_ev, 1), B), dtype=torch.uint8, device="cuda")
        md = None if loss_mask is None else torch.from_numpy(np.ascontiguousarray(loss_mask, dtype=np.uint8)).cuda()
        h.prefill(t, losses, p, qd, acc if n_ev else None, A if n_ev else None, loss_mask=md)
        torch.cuda.synchronize()
        out = {"losses": losses.cpu().numpy().astype(np.float64), "p_next": p.cpu().numpy(),
               "A": A.cpu().numpy()[:n_ev], "accept": acc.cpu().numpy()[:n_ev].astype(bool)}
    else:
        losses = np.empty((B, T1 - 1), dtype=np.float32)
        p = np.empty((B, wl.vocab), dtype=np.float32)
        A = np.empty((max(n_ev, 1), B), dtype=np.float32)
        acc = np.empty((max(n_ev, 1), B), dtype=np.uint8)
        h.prefill(np.ascontiguousarray(tok), losses, p,
                  np.ascontiguousarray(sq[:n_ev]) if n_ev else None,
                  acc if n_ev else None, A if n_ev else None,
                  loss_mask=None if loss_mask is None else np.ascontiguousarray(loss_mask, dtype=np.uint8))
        out = {"losses": losses.astype(np.float64), "p_next": p, "A": A[:n_ev],
               "accept": acc[:n_ev].astype(bool)}
    out["W"] = [h.fast_weights(s) for s in range(B)]
    out["handle"] = h
    return out


def compare(wl, gpu, ref, seqs=None, check_p=True):
    seqs = range(len(gpu["W"])) if seqs is None else seqs
    tol = TOL[wl.dtype]
    report = {}
    for s in seqs:
        err = np.abs(gpu["losses"][s] - ref["losses"][s])
        assert np.all(np.isfinite(gpu["losses"][s])), f"seq {s}: non-finite loss"
        if wl.dtype == "fp32":
            assert err.max() <= tol["loss_max"], f"seq {s}: max loss err {err.max():.3e}"
        else:
            assert err.mean() <= tol["loss_mean"], f"seq {s}: mean loss err {err.mean():.3e}"
        rel = oracle.weights_rel_frobenius(gpu["W"][s], ref["W"][s], wl.fast_mats)
        assert rel <= tol["w_rel"], f"seq {s}: W rel-Frobenius {rel:.3e}"
        if check_p:
            perr = np.abs(gpu["p_next"][s] - ref["p_next"][s]).max()
            assert perr <= (1e-5 if wl.dtype == "fp32" else 2e-3), f"seq {s}: p_next err {perr:.3e}"
        report[s] = (float(err.max()), float(err.mean()), rel)
    return report


def compare_settlement(gpu, ref, seqs, noise):
    """Decisions agree wherever the oracle's |A| clears the noise bound;
    returns the number of events that were decidable."""
    decided = 0
    for s in seqs:
        for e in range(ref["A"].shape[0]):
            a_ref, a_gpu = ref["A"][e, s], gpu["A"][e, s]
            assert abs(a_gpu - a_ref) <= noise, f"event {e} seq {s}: A {a_gpu:.4e} vs {a_ref:.4e}"
            if abs(a_ref) > 2 * noise:
                assert bool(gpu["accept"][e, s]) == bool(ref["accept"][e, s]), f"event {e} seq {s}"
                decided += 1
    return decided
