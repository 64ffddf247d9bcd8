"""ttt_clip_sgd_noalloc against ttt_clip_sgd, through the C ABI.

The no-allocation variant serves callers that cannot allocate device memory
(their device memory belongs to their own allocator or budget, or cudaMalloc's
implicit synchronisation is not acceptable in their loop).  It must give the
same result as the workspace entry point; two calls in a row check that the
shared scratch array carries nothing over from one call to the next.  This file
is collected last so a stop-at-first-failure run has run every other test.
"""
import numpy as np
import pytest
import torch

from chunked_next_token_ttt_b300 import ttt as T

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _case(seed, nslots, B, n, clip):
    rng = np.random.default_rng(seed)
    W = torch.from_numpy(rng.normal(0, 0.02, (nslots, B, n)).astype(np.float32)).cuda()
    G = torch.from_numpy(rng.normal(0, 0.01 * (seed + 1), (nslots, B, n)).astype(np.float32)).cuda()
    return W, G, clip


def _call(fn, W, G, clip, dtype="bf16", **kw):
    """(W32, Wop, norm, scale) after the call, and the call's status."""
    W32 = W.clone()
    Wop = torch.zeros(W.shape, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32, device="cuda")
    norm = torch.full((W.shape[1],), -1.0, device="cuda")
    scale = torch.full((W.shape[1],), -1.0, device="cuda")
    status = 0
    try:
        fn(dtype, W32, Wop, G, 0.05, clip, norm, scale, **kw)
    except T.TTTError as e:
        status = e.status
    torch.cuda.synchronize()
    return (W32, Wop, norm, scale), status


def _run(fn, W, G, clip, dtype="bf16", **kw):
    out, status = _call(fn, W, G, clip, dtype, **kw)
    assert status == 0, T.STATUS.get(status, status)
    return out


def _same(got, ref):
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a.float().cpu().numpy(), b.float().cpu().numpy(), rtol=1e-6, atol=1e-9)


def _workspace(W):
    return torch.empty(T.clip_sgd_workspace_size(*W.shape), dtype=torch.uint8, device="cuda")


def test_no_alloc_clip_sgd_matches_workspace_entry_point_twice():
    cases = [_case(0, 6, 8, 300000, 1.0), _case(1, 2, 3, 20000, 1e-3)]
    for W, G, clip in cases:   # two calls in a row on different sizes
        ref = _run(T.clip_sgd, W, G, clip, workspace=_workspace(W))
        got = _run(T.clip_sgd_noalloc, W, G, clip)
        _same(got, ref)


def test_no_alloc_fp32_operand_copy_matches_workspace_entry_point():
    W, G, clip = _case(2, 3, 4, 50001, 0.5)
    ref = _run(T.clip_sgd, W, G, clip, "fp32", workspace=_workspace(W))
    got = _run(T.clip_sgd_noalloc, W, G, clip, "fp32")
    _same(got, ref)
    np.testing.assert_array_equal(got[1].cpu().numpy(), got[0].cpu().numpy())


def test_no_alloc_nonfinite_gradient_skips_that_sequence_then_recovers():
    """A NaN in one sequence's gradient: status NONFINITE, that sequence's
    weights unchanged (scale 0), the others updated as by the workspace entry
    point; the next call on finite gradients succeeds and matches again."""
    nonfinite = next(k for k, v in T.STATUS.items() if v.startswith("non-finite"))
    W, G, clip = _case(3, 2, 4, 30000, 1.0)
    bad = G.clone()
    bad[1, 2, 777] = float("nan")
    got, st = _call(T.clip_sgd_noalloc, W, bad, clip)
    ref, st_ref = _call(T.clip_sgd, W, bad, clip, workspace=_workspace(W))
    assert st == st_ref == nonfinite
    W32, _, norm, scale = (x.float().cpu().numpy() for x in got)
    np.testing.assert_array_equal(W32[:, 2], W.cpu().numpy()[:, 2])
    assert scale[2] == 0.0 and not np.isfinite(norm[2])
    keep = [0, 1, 3]
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a.float().cpu().numpy()[..., keep, :] if a.dim() == 3 else a.cpu().numpy()[keep],
                                   b.float().cpu().numpy()[..., keep, :] if b.dim() == 3 else b.cpu().numpy()[keep],
                                   rtol=1e-6, atol=1e-9)
    assert np.all(scale[keep] > 0)
    _same(_run(T.clip_sgd_noalloc, W, G, clip), _run(T.clip_sgd, W, G, clip, workspace=_workspace(W)))


def test_no_alloc_rejects_sizes_beyond_its_fixed_scratch():
    n = 8192 * 70000        # 70000 pieces per (slot, sequence): beyond 2^20 floats
    W = torch.zeros((2, 8, 1), device="cuda")
    lib = T._ops_lib()
    st = lib.ttt_clip_sgd_noalloc(1, 2, 8, n, W.data_ptr(), W.data_ptr(), W.data_ptr(), 0.1, 1.0,
                                  None, None, None)
    assert st == 2
    assert b"fixed maximum" in lib.ttt_last_error()
