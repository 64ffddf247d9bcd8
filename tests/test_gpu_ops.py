"""Single-kernel tests through the op-level C ABI (include/ttt_ops.h).

GEMMs (SIMT and tcgen05, every operand major-ness, batched, ragged tails,
every epilogue) against float64 products of the same (bf16-exact) inputs;
cross-entropy, RMSNorm and the clipped SGD step against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from chunked_next_token_ttt_b300 import ttt as T

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def bf16_exact(shape, rng, scale=1.0):
    x = torch.from_numpy(rng.normal(0, scale, shape).astype(np.float32)).to(torch.bfloat16)
    return x


def to64(t):
    return t.float().cpu().numpy().astype(np.float64)


def operands(rng, M, N, K, batch, a_k, b_k, dtype):
    """A(m,k) and B(n,k) stored K-major or MN-major; returns device tensors and
    the float64 [batch, M, K] / [batch, N, K] views."""
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    A = bf16_exact((batch, M, K), rng).to(tdt)
    B = bf16_exact((batch, N, K), rng).to(tdt)
    A_store = A if a_k else A.transpose(1, 2)
    B_store = B if b_k else B.transpose(1, 2)
    return A_store.contiguous().cuda(), B_store.contiguous().cuda(), to64(A), to64(B)


def run_gemm(M, N, K, batch, a_k, b_k, impl, epi="store_f32", dtype="bf16", seed=0, **kw):
    rng = np.random.default_rng(seed)
    Ad, Bd, A64, B64 = operands(rng, M, N, K, batch, a_k, b_k, dtype)
    ref = np.einsum("bmk,bnk->bmn", A64, B64)
    out = torch.zeros((batch, M, N), dtype=torch.float32, device="cuda")
    args = T.gemm_args(M, N, K, Ad, Bd, out, batch=batch, dtype=dtype, a_kmajor=a_k, b_kmajor=b_k,
                       epi=epi, impl=impl, sA=M * K, sB=N * K, sO=M * N, **kw)
    T.op_gemm(args)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), ref


def test_tensor_core_gemm_single_tile_first():
    """Smallest tcgen05 case first: one 128x128 tile, K = 64, both K-major."""
    got, ref = run_gemm(128, 128, 64, 1, True, True, "tensor")
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max() + 1e-6


@pytest.mark.parametrize("a_k", [True, False], ids=["A_kmaj", "A_mnmaj"])
@pytest.mark.parametrize("b_k", [True, False], ids=["B_kmaj", "B_mnmaj"])
@pytest.mark.parametrize("impl", ["tensor", "simt"])
def test_gemm_every_major_batched(a_k, b_k, impl):
    got, ref = run_gemm(256, 384, 320, 2, a_k, b_k, impl, seed=1)
    assert np.abs(got - ref).max() <= 2e-5 * np.abs(ref).max()


@pytest.mark.parametrize("a_k", [True, False], ids=["A_kmaj", "A_mnmaj"])
@pytest.mark.parametrize("b_k", [True, False], ids=["B_kmaj", "B_mnmaj"])
def test_tensor_core_gemm_ragged_tails(a_k, b_k):
    """M, N, K not multiples of the 128 x 128 x 64 tile (TMA zero-fills the rest)."""
    got, ref = run_gemm(200, 136, 72, 3, a_k, b_k, "tensor", seed=2)
    assert np.abs(got - ref).max() <= 2e-5 * np.abs(ref).max()


def test_tensor_core_gemm_long_k_pipeline_wraps():
    """K = 2048: 32 k-slices through the 4-deep ring (every slot reused 8 times)."""
    got, ref = run_gemm(128, 256, 2048, 1, True, False, "tensor", seed=3)
    assert np.abs(got - ref).max() <= 2e-5 * np.abs(ref).max()


def test_fp32_simt_gemm_exact_inputs():
    got, ref = run_gemm(70, 90, 50, 2, False, True, "simt", dtype="fp32", seed=4)
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max()


def _bf(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


@pytest.mark.parametrize("impl", ["tensor", "simt"])
def test_epilogues(impl):
    rng = np.random.default_rng(5)
    M, N, K, batch = 256, 256, 128, 2
    Ad, Bd, A64, B64 = operands(rng, M, N, K, batch, True, True, "bf16")
    acc = np.einsum("bmk,bnk->bmn", A64, B64)
    common = dict(batch=batch, impl=impl, sA=M * K, sB=N * K, sO=M * N)
    bf = torch.bfloat16

    # GELU: stash z and a
    z = torch.zeros((batch, M, N), dtype=bf, device="cuda")
    a = torch.zeros((batch, M, N), dtype=bf, device="cuda")
    T.op_gemm(T.gemm_args(M, N, K, Ad, Bd, z, epi="gelu", out2=a, ldo2=N, sO2=M * N, **common))
    torch.cuda.synchronize()
    np.testing.assert_allclose(to64(z), _bf(acc), rtol=1e-2, atol=1e-2)
    np.testing.assert_allclose(to64(a), _bf(oracle.gelu(acc)), rtol=1e-2, atol=1e-2)

    # RESID: fp32 out = aux + acc, and its bf16 copy
    r = torch.from_numpy(rng.normal(0, 1, (batch, M, N)).astype(np.float32)).cuda()
    out = torch.zeros_like(r)
    cp = torch.zeros((batch, M, N), dtype=bf, device="cuda")
    T.op_gemm(T.gemm_args(M, N, K, Ad, Bd, out, epi="resid", aux=r, ldx=N, sX=M * N, out2=cp, ldo2=N,
                          sO2=M * N, **common))
    torch.cuda.synchronize()
    want = r.cpu().numpy().astype(np.float64) + acc
    np.testing.assert_allclose(out.cpu().numpy(), want, rtol=1e-5, atol=1e-4)
    np.testing.assert_allclose(to64(cp), _bf(want), rtol=1e-2, atol=1e-2)

    # SWIGLU: silu(aux) * acc
    g = torch.from_numpy(rng.normal(0, 1, (batch, M, N)).astype(np.float32)).cuda()
    sw = torch.zeros((batch, M, N), dtype=bf, device="cuda")
    T.op_gemm(T.gemm_args(M, N, K, Ad, Bd, sw, epi="swiglu", aux=g, ldx=N, sX=M * N, **common))
    torch.cuda.synchronize()
    np.testing.assert_allclose(to64(sw), _bf(oracle.silu(g.cpu().numpy().astype(np.float64)) * acc),
                               rtol=2e-2, atol=2e-2)

    # DGELU: acc * GELU'(aux), in place over aux
    zz = torch.from_numpy(rng.normal(0, 1, (batch, M, N)).astype(np.float32)).to(bf).cuda()
    z64 = to64(zz)
    T.op_gemm(T.gemm_args(M, N, K, Ad, Bd, zz, epi="dgelu", aux=zz, ldx=N, sX=M * N, **common))
    torch.cuda.synchronize()
    np.testing.assert_allclose(to64(zz), _bf(acc * oracle.gelu_grad(z64)), rtol=2e-2, atol=2e-2)

    # DW: the gradient in the storage's dW type (bf16 here) and per-tile sums
    # of squares of the fp32 accumulators
    dw = torch.zeros((batch, M, N), dtype=bf, device="cuda")
    args = T.gemm_args(M, N, K, Ad, Bd, dw, epi="dw", **common)
    tiles = T.op_gemm_partial_tiles(args)
    part = torch.zeros((batch, tiles), dtype=torch.float32, device="cuda")
    args = T.gemm_args(M, N, K, Ad, Bd, dw, epi="dw", partials=part, **common)
    T.op_gemm(args)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to64(dw), acc, rtol=2.0 ** -8, atol=1e-3)   # one bf16 rounding
    np.testing.assert_allclose(part.cpu().numpy().sum(1), (acc ** 2).sum(axis=(1, 2)), rtol=1e-5)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_cross_entropy_op(dtype):
    rng = np.random.default_rng(6)
    M, V = 37, 3001
    logits = rng.normal(0, 2, (M, V)).astype(np.float32)
    tgt = rng.integers(0, V, M).astype(np.int32)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    L = torch.from_numpy(logits).to(tdt).cuda()
    L64 = to64(L)
    losses = torch.zeros(M, dtype=torch.float32, device="cuda")
    T.op_cross_entropy(dtype, L, torch.from_numpy(tgt).cuda(), 0.25, True, losses)
    torch.cuda.synchronize()
    ref_l, p = oracle.cross_entropy(L64, tgt.astype(np.int64))
    dl = p.copy()
    dl[np.arange(M), tgt] -= 1
    tol = 1e-5 if dtype == "fp32" else 1e-2
    np.testing.assert_allclose(losses.cpu().numpy(), ref_l, rtol=tol, atol=tol)
    np.testing.assert_allclose(to64(L), dl * 0.25, atol=1e-6 if dtype == "fp32" else 1e-3)


def test_rmsnorm_ops():
    rng = np.random.default_rng(7)
    M, d, eps = 33, 777, 1e-6
    x = torch.from_numpy(rng.normal(0, 0.05, (M, d)).astype(np.float32)).cuda()
    y = torch.zeros_like(x)
    r = torch.zeros(M, device="cuda")
    T.op_rmsnorm_forward("fp32", x, eps, y, r)
    dy = torch.from_numpy(rng.normal(0, 1, (M, d)).astype(np.float32)).cuda()
    dx = torch.zeros_like(x)
    T.op_rmsnorm_backward("fp32", x, r, dy, dx)
    torch.cuda.synchronize()
    x64 = x.cpu().numpy().astype(np.float64)
    y_ref, r_ref = oracle.rmsnorm(x64, eps)
    np.testing.assert_allclose(y.cpu().numpy(), y_ref, rtol=1e-5, atol=1e-6)
    dx_ref = oracle.rmsnorm_backward(x64, r_ref, dy.cpu().numpy().astype(np.float64))
    np.testing.assert_allclose(dx.cpu().numpy(), dx_ref, rtol=1e-4, atol=1e-4 * np.abs(dx_ref).max())


@pytest.mark.parametrize("clip", [0.0, 1e-3, 1e6])
def test_clip_sgd_op_matches_oracle(clip):
    rng = np.random.default_rng(8)
    nslots, B, n, eta = 3, 4, 10000, 0.05
    W = rng.normal(0, 0.02, (nslots, B, n)).astype(np.float32)
    G = rng.normal(0, 0.01, (nslots, B, n)).astype(np.float32)
    W32 = torch.from_numpy(W).cuda()
    Wop = torch.zeros((nslots, B, n), dtype=torch.bfloat16, device="cuda")
    dW = torch.from_numpy(G).cuda()
    ws = torch.empty(T.clip_sgd_workspace_size(nslots, B, n), dtype=torch.uint8, device="cuda")
    norm = torch.zeros(B, device="cuda")
    scale = torch.zeros(B, device="cuda")
    T.clip_sgd("bf16", W32, Wop, dW, eta, clip, norm, scale, ws)
    for s in range(B):
        grads = [{"g": G[j, s].astype(np.float64)} for j in range(nslots)]
        sc, nr = oracle.clip_scale(grads, clip)
        assert abs(float(norm[s]) - nr) <= 1e-5 * nr
        assert abs(float(scale[s]) - sc) <= 1e-5 * sc
        want = W[:, s].astype(np.float64) - eta * sc * G[:, s].astype(np.float64)
        np.testing.assert_allclose(W32[:, s].cpu().numpy(), want, rtol=1e-6, atol=1e-8)
        np.testing.assert_array_equal(Wop[:, s].float().cpu().numpy(),
                                      W32[:, s].to(torch.bfloat16).float().cpu().numpy())


def test_clip_sgd_nonfinite_sequence_is_skipped():
    nslots, B, n = 2, 3, 5000
    W = torch.ones((nslots, B, n), device="cuda")
    Wop = torch.zeros((nslots, B, n), dtype=torch.bfloat16, device="cuda")
    dW = torch.full((nslots, B, n), 0.5, device="cuda")
    dW[1, 1, 7] = float("nan")
    ws = torch.empty(T.clip_sgd_workspace_size(nslots, B, n), dtype=torch.uint8, device="cuda")
    with pytest.raises(T.TTTError) as e:
        T.clip_sgd("bf16", W, Wop, dW, 0.1, 1.0, workspace=ws)
    assert e.value.status == 5
    assert torch.all(W[:, 1] == 1.0)
    assert torch.all(W[:, 0] < 1.0) and torch.all(W[:, 2] < 1.0)


def split_planes(x64):
    """fp32 values as bf16 hi/lo planes stacked [2, ...] (hi = bf16(v), lo = bf16(v - hi))."""
    v = torch.from_numpy(np.asarray(x64, dtype=np.float32))
    hi = v.to(torch.bfloat16)
    lo = (v - hi.float()).to(torch.bfloat16)
    return torch.stack([hi, lo]).contiguous()


@pytest.mark.parametrize("a_k", [True, False], ids=["A_kmaj", "A_mnmaj"])
@pytest.mark.parametrize("b_k", [True, False], ids=["B_kmaj", "B_mnmaj"])
@pytest.mark.parametrize("impl", ["tensor", "simt"])
def test_bf16x3_split_gemm_is_fp32_accurate(a_k, b_k, impl):
    """hi*hi + hi*lo + lo*hi on the tensor cores: error ~2^-17 of the operands'
    scale, far inside the fp32 workloads' 1e-4 tolerance (plain bf16 would be
    ~2^-9)."""
    rng = np.random.default_rng(9)
    M, N, K, batch = 256, 200, 320, 2
    A = rng.normal(0, 1, (batch, M, K)).astype(np.float32)
    Bm = rng.normal(0, 1, (batch, N, K)).astype(np.float32)
    ref = np.einsum("bmk,bnk->bmn", A.astype(np.float64), Bm.astype(np.float64))
    As = split_planes(A if a_k else A.transpose(0, 2, 1)).cuda()
    Bs = split_planes(Bm if b_k else Bm.transpose(0, 2, 1)).cuda()
    out = torch.zeros((batch, M, N), dtype=torch.float32, device="cuda")
    args = T.gemm_args(M, N, K, As, Bs, out, batch=batch, dtype="bf16x3", a_kmajor=a_k, b_kmajor=b_k,
                       epi="store_f32", impl=impl, sA=M * K, sB=N * K, sO=M * N,
                       loA=batch * M * K, loB=batch * N * K)
    T.op_gemm(args)
    torch.cuda.synchronize()
    err = np.abs(out.cpu().numpy() - ref).max()
    # per product: dropped lo*lo and the two lo roundings, about 3 * 2^-18 of |a b|;
    # summed over K random-sign terms and taken as the max over ~1e5 outputs
    scale = np.sqrt(K)
    assert err <= 6e-5 * scale, err
    hi_only = np.einsum("bmk,bnk->bmn", _bf(A), _bf(Bm))
    assert err * 20 < np.abs(hi_only - ref).max()
    # and the split store epilogue writes hi/lo planes that add back to the value
    o2 = torch.zeros((2, batch, M, N), dtype=torch.bfloat16, device="cuda")
    args = T.gemm_args(M, N, K, As, Bs, o2, batch=batch, dtype="bf16x3", a_kmajor=a_k, b_kmajor=b_k,
                       epi="store", impl=impl, sA=M * K, sB=N * K, sO=M * N,
                       loA=batch * M * K, loB=batch * N * K, loO=batch * M * N)
    T.op_gemm(args)
    torch.cuda.synchronize()
    v = (o2[0].float() + o2[1].float()).cpu().numpy()
    assert np.abs(v - ref).max() <= 6e-5 * scale + 1e-5 * np.abs(ref).max()


@pytest.mark.parametrize("dtype", ["bf16", "bf16x3"])
def test_split_k_narrow_long_k_gemm(dtype):
    """N = 512, K = 2048, 2 x 2 tiles per batch: the tensor-core path splits K
    into workspace slices and reduces them in a fixed order; results equal the
    unsplit kernel's within fp32 rounding, and the GELU epilogue sees the sum."""
    rng = np.random.default_rng(10)
    M, N, K, batch = 256, 512, 2048, 2
    A = rng.normal(0, 1, (batch, M, K)).astype(np.float32)
    Bm = rng.normal(0, 1, (batch, N, K)).astype(np.float32)
    if dtype == "bf16":
        A, Bm = _bf(A).astype(np.float32), _bf(Bm).astype(np.float32)
        Ad = torch.from_numpy(A).to(torch.bfloat16).cuda()
        Bd = torch.from_numpy(Bm).to(torch.bfloat16).cuda()
        lo = {}
    else:
        Ad, Bd = split_planes(A).cuda(), split_planes(Bm).cuda()
        lo = dict(loA=batch * M * K, loB=batch * N * K)
    ref = np.einsum("bmk,bnk->bmn", A.astype(np.float64), Bm.astype(np.float64))
    ws = torch.zeros(16 * batch * M * N, dtype=torch.float32, device="cuda")
    outs = []
    for w in (None, ws):
        out = torch.zeros((batch, M, N), dtype=torch.float32, device="cuda")
        T.op_gemm(T.gemm_args(M, N, K, Ad, Bd, out, batch=batch, dtype=dtype, epi="store_f32", impl="tensor",
                              sA=M * K, sB=N * K, sO=M * N, workspace=w, **lo))
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy().astype(np.float64))
    tol = (6e-5 if dtype == "bf16x3" else 2e-5) * np.sqrt(K)
    assert np.abs(outs[0] - ref).max() <= tol * (1 if dtype == "bf16x3" else np.abs(ref).max() / np.sqrt(K))
    np.testing.assert_allclose(outs[1], outs[0], rtol=1e-5, atol=1e-3)
    # the workspace was used: its slices are non-zero
    assert float(ws.abs().sum()) > 0


def test_split_k_ragged_residual_twice_in_a_row():
    """Split K with ragged row and column tiles (M = 200, N = 136) and the
    residual epilogue, issued twice back to back: the last CTA of each tile sums
    the partials in split order, so both calls give the same bits, and both
    match the unsplit kernel within fp32 rounding (the per-tile arrival counters
    are back at zero after each call)."""
    rng = np.random.default_rng(11)
    M, N, K, batch = 200, 136, 1536, 3
    A = _bf(rng.normal(0, 1, (batch, M, K))).astype(np.float32)
    Bm = _bf(rng.normal(0, 1, (batch, N, K))).astype(np.float32)
    X = rng.normal(0, 1, (batch, M, N)).astype(np.float32)
    Ad = torch.from_numpy(A).to(torch.bfloat16).cuda()
    Bd = torch.from_numpy(Bm).to(torch.bfloat16).cuda()
    Xd = torch.from_numpy(X).cuda()
    ref = X + np.einsum("bmk,bnk->bmn", A.astype(np.float64), Bm.astype(np.float64))
    ws = torch.zeros(16 * batch * M * N, dtype=torch.float32, device="cuda")
    outs = []
    for w in (None, ws, ws):
        out = torch.zeros((batch, M, N), dtype=torch.float32, device="cuda")
        T.op_gemm(T.gemm_args(M, N, K, Ad, Bd, out, batch=batch, dtype="bf16", epi="resid", impl="tensor",
                              sA=M * K, sB=N * K, sO=M * N, aux=Xd, ldx=N, sX=M * N, workspace=w))
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy().astype(np.float64))
    assert float(ws.abs().sum()) > 0
    np.testing.assert_array_equal(outs[1], outs[2])
    np.testing.assert_allclose(outs[1], outs[0], rtol=1e-5, atol=2e-3)
    assert np.abs(outs[0] - ref).max() <= 2e-3 * np.abs(ref).max()


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "bf16x3"])
@pytest.mark.parametrize("K", [768, 4096])
def test_small_m_gemm_long_k_split_over_warps(dtype, K):
    """Eight rows, shared weights, few output columns (a frozen block of a
    one-token forward): several warps share each column's K range."""
    rng = np.random.default_rng(12)
    M, N = 8, 200
    A = rng.normal(0, 1, (M, K)).astype(np.float32)
    Bm = rng.normal(0, 1, (N, K)).astype(np.float32)
    X = rng.normal(0, 1, (M, N)).astype(np.float32)
    if dtype == "fp32":
        Ad, Bd, lo = torch.from_numpy(A).cuda(), torch.from_numpy(Bm).cuda(), {}
        A64, B64 = A.astype(np.float64), Bm.astype(np.float64)
    elif dtype == "bf16":
        Ad, Bd, lo = torch.from_numpy(A).to(torch.bfloat16).cuda(), torch.from_numpy(Bm).to(torch.bfloat16).cuda(), {}
        A64, B64 = _bf(A), _bf(Bm)
    else:
        Ad, Bd = split_planes(A).cuda(), split_planes(Bm).cuda()
        lo = dict(loA=M * K, loB=N * K)
        A64, B64 = A.astype(np.float64), Bm.astype(np.float64)
    ref = A64 @ B64.T + X
    out = torch.from_numpy(X.copy()).cuda()
    T.op_gemm(T.gemm_args(M, N, K, Ad, Bd, out, dtype=dtype, epi="resid", aux=out, ldx=N, **lo))
    torch.cuda.synchronize()
    tol = {"fp32": 1e-5, "bf16": 1e-5, "bf16x3": 6e-5}[dtype] * np.sqrt(K) * (np.abs(ref).max() if dtype != "bf16x3" else 1)
    assert np.abs(out.cpu().numpy() - ref).max() <= tol


@pytest.mark.parametrize("N", [1000, 9000], ids=["narrow", "wide"])
@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("b_k", [True, False], ids=["B_kmaj", "B_nmaj"])
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "bf16x3"])
def test_small_m_gemm(M, b_k, dtype, N):
    """A few rows per batch entry (one token per sequence): weight-streaming kernel."""
    rng = np.random.default_rng(11)
    K, batch = 520, 3   # N = 9000 with M <= 2: four columns per warp, ragged last group
    A = rng.normal(0, 1, (batch, M, K)).astype(np.float32)
    Bm = rng.normal(0, 1, (batch, N, K)).astype(np.float32)
    Bs = Bm if b_k else np.ascontiguousarray(Bm.transpose(0, 2, 1))
    if dtype == "fp32":
        Ad, Bd, lo = torch.from_numpy(A).cuda(), torch.from_numpy(Bs).cuda(), {}
        A64, B64 = A.astype(np.float64), Bm.astype(np.float64)
    elif dtype == "bf16":
        Ad, Bd, lo = (torch.from_numpy(A).to(torch.bfloat16).cuda(), torch.from_numpy(Bs).to(torch.bfloat16).cuda(), {})
        A64, B64 = _bf(A), _bf(Bm)
    else:
        Ad, Bd = split_planes(A).cuda(), split_planes(Bs).cuda()
        lo = dict(loA=batch * M * K, loB=batch * N * K)
        A64, B64 = A.astype(np.float64), Bm.astype(np.float64)
    ref = np.einsum("bmk,bnk->bmn", A64, B64)
    out = torch.zeros((batch, M, N), dtype=torch.float32, device="cuda")
    T.op_gemm(T.gemm_args(M, N, K, Ad, Bd, out, batch=batch, dtype=dtype, b_kmajor=b_k, epi="store_f32",
                          sA=M * K, sB=N * K, sO=M * N, **lo))
    torch.cuda.synchronize()
    tol = {"fp32": 1e-5, "bf16": 1e-5, "bf16x3": 6e-5}[dtype] * np.sqrt(K) * (np.abs(ref).max() if dtype != "bf16x3" else 1)
    assert np.abs(out.cpu().numpy() - ref).max() <= tol


@pytest.mark.parametrize("dh,window,rows", [(64, 1, 200), (64, 100, 300), (64, 300, 300), (128, 130, 257),
                                            (64, 5000, 260)],
                         ids=["dh64_k1", "dh64_k100", "dh64_k300", "dh128_k130", "dh64_k_beyond_rows"])
def test_fused_sliding_window_attention_op(dh, window, rows):
    """The fused attention kernel alone against a float64 evaluation of
    windowed softmax attention on the same bf16 Q, K, V: several 128-query
    blocks with a ragged last one, windows of 1, below, at and beyond a
    128-key block and beyond the sequence, head widths 64 and 128."""
    rng = np.random.default_rng(21)
    B, H, pad = 2, 2, 256
    d = H * dh
    nqb = -(-rows // 128)
    L = pad + nqb * 128
    qkv = np.zeros((B, L, 3 * d), dtype=np.float32)
    qkv[:, pad:pad + rows] = rng.normal(0, 1, (B, rows, 3 * d))
    qkv[:, pad:pad + rows, :2 * d] *= 2.0          # sharper softmax
    qkv = _bf(qkv).astype(np.float32)
    qd = torch.from_numpy(qkv).to(torch.bfloat16).cuda()
    out = torch.zeros((B, L, d), dtype=torch.bfloat16, device="cuda")
    T.op_sliding_window_attention(qd, rows, H, window, pad, out)
    torch.cuda.synchronize()
    got = to64(out)[:, pad:pad + rows]
    x = qkv[:, pad:pad + rows].astype(np.float64)
    ref = np.zeros((B, rows, d))
    p = np.arange(rows)
    mask = (p[None, :] <= p[:, None]) & (p[None, :] > p[:, None] - window)
    for s in range(B):
        for h in range(H):
            c = slice(h * dh, (h + 1) * dh)
            S = x[s, :, c] @ x[s, :, d:2 * d][:, c].T / np.sqrt(dh)
            S = np.where(mask, S, -np.inf)
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            ref[s, :, c] = P @ x[s, :, 2 * d:][:, c]
    err = np.abs(got - ref)
    # where it goes wrong, by sequence, 128-query block and head
    blocks = {(s, b, h): float(err[s, b * 128:(b + 1) * 128, h * dh:(h + 1) * dh].max())
              for s in range(B) for b in range(nqb) for h in range(H)}
    assert err.max() <= 3e-2, f"max err {err.max():.3e}; per (seq, query block, head): {blocks}"
    # the padding rows of out are never written
    assert float(out[:, :pad].abs().max()) == 0.0
