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


def _run(fn, W, G, clip, **kw):
    W32 = W.clone()
    Wop = torch.zeros(W.shape, dtype=torch.bfloat16, device="cuda")
    norm = torch.full((W.shape[1],), -1.0, device="cuda")
    scale = torch.full((W.shape[1],), -1.0, device="cuda")
    fn("bf16", W32, Wop, G, 0.05, clip, norm, scale, **kw)
    torch.cuda.synchronize()
    return W32, Wop, norm, scale


def test_no_alloc_clip_sgd_matches_workspace_entry_point_twice():
    cases = [_case(0, 6, 8, 300000, 1.0), _case(1, 2, 3, 20000, 1e-3)]
    for W, G, clip in cases:   # two calls in a row on different sizes
        ws = torch.empty(T.clip_sgd_workspace_size(*W.shape), dtype=torch.uint8, device="cuda")
        ref = _run(T.clip_sgd, W, G, clip, workspace=ws)
        got = _run(T.clip_sgd_noalloc, W, G, clip)
        for a, b in zip(got, ref):
            np.testing.assert_allclose(a.float().cpu().numpy(), b.float().cpu().numpy(), rtol=1e-6, atol=1e-9)


def test_no_alloc_rejects_sizes_beyond_its_fixed_scratch():
    n = 8192 * 70000        # 70000 pieces per (slot, sequence): beyond 2^20 floats
    W = torch.zeros((2, 8, 1), device="cuda")
    lib = T._ops_lib()
    st = lib.ttt_clip_sgd_noalloc(1, 2, 8, n, W.data_ptr(), W.data_ptr(), W.data_ptr(), 0.1, 1.0,
                                  None, None, None)
    assert st == 2
    assert b"fixed maximum" in lib.ttt_last_error()
