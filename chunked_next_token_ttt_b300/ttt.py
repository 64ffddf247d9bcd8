"""Thin ctypes binding of libttt (argument marshalling only).

Every step of the TTT inner loop runs inside libttt's CUDA kernels; this
module only converts numpy arrays / torch tensors into pointers and sizes,
calls the C ABI declared in include/ttt.h, and raises TTTError on a non-OK
status.  There is no CPU fallback: without the built library (or without a
GPU) every call fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libttt.so")

STATUS = {0: "ok", 1: "bad argument", 2: "bad shape", 3: "out of device memory", 4: "CUDA error",
          5: "non-finite gradient norm", 6: "timeout", 7: "unsupported", 8: "call out of order"}
BLOCK = {"gelu": 0, "swiglu": 1}
DTYPE = {"fp32": 0, "bf16": 1}
MATS = {"gelu": ("W1", "W2"), "swiglu": ("Wg", "Wu", "Wd")}
FAST_BIT = {"W1": 1, "W2": 2, "Wg": 1, "Wd": 2, "Wu": 4}


class TTTError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}" + (f" ({detail})" if detail else ""))


class Dims(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("d_ff", ctypes.c_int), ("vocab", ctypes.c_int),
                ("n_prefix", ctypes.c_int), ("n_fast", ctypes.c_int), ("block_kind", ctypes.c_int),
                ("fast_mask", ctypes.c_int), ("dtype", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("static_mlp", ctypes.c_int), ("attn_heads", ctypes.c_int), ("attn_window", ctypes.c_int)]


class HParams(ctypes.Structure):
    _fields_ = [("eta", ctypes.c_float), ("clip", ctypes.c_float), ("chunk", ctypes.c_int),
                ("settle_every", ctypes.c_int), ("max_batch", ctypes.c_int), ("settle_len", ctypes.c_int),
                ("reset_every", ctypes.c_int)]


class Options(ctypes.Structure):
    """ttt_options: zero fields are the library's defaults."""
    _fields_ = [("no_pdl", ctypes.c_int), ("no_decode_graph", ctypes.c_int), ("fp32_simt", ctypes.c_int),
                ("hoist_chunks", ctypes.c_int), ("no_token_kernel", ctypes.c_int), ("max_ctas", ctypes.c_int),
                ("no_dw_stream", ctypes.c_int), ("attn_unfused", ctypes.c_int), ("no_decode_persist", ctypes.c_int)]


class Weights(ctypes.Structure):
    _fields_ = [("E", ctypes.c_void_p), ("U", ctypes.c_void_p),
                ("prefix", ctypes.POINTER(ctypes.c_void_p)), ("fast", ctypes.POINTER(ctypes.c_void_p)),
                ("statics", ctypes.POINTER(ctypes.c_void_p)), ("attn", ctypes.POINTER(ctypes.c_void_p))]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libttt.so; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libttt.so is not built ({path}); run "
                           "`python -m chunked_next_token_ttt_b300.build`")
    lib = ctypes.CDLL(path)
    sig = {
        "ttt_create": ([ctypes.POINTER(Dims), ctypes.POINTER(HParams), ctypes.POINTER(Weights),
                        ctypes.POINTER(_P)], _I),
        "ttt_create_ex": ([ctypes.POINTER(Dims), ctypes.POINTER(HParams), ctypes.POINTER(Weights),
                           ctypes.POINTER(Options), ctypes.POINTER(_P)], _I),
        "ttt_destroy": ([_P], _I),
        "ttt_prefill": ([_P, _P, _I, _I, _P, _P, _P, _I, _P, _P, _P], _I),
        "ttt_prefill_masked": ([_P, _P, _P, _I, _I, _P, _P, _P, _I, _P, _P, _P], _I),
        "ttt_decode_step": ([_P, _P, _P, _P, _P], _I),
        "ttt_settle": ([_P, _P, _I, _P, _P, _P], _I),
        "ttt_get_fast_weights": ([_P, _I, _I, _I, _P, _P], _I),
        "ttt_reset": ([_P, _P], _I),
        "ttt_state_size": ([_P, ctypes.POINTER(ctypes.c_size_t)], _I),
        "ttt_get_state": ([_P, _P, ctypes.c_size_t, _P], _I),
        "ttt_set_state": ([_P, _P, ctypes.c_size_t, _P], _I),
        "ttt_profile_enable": ([_P, _I], _I),
        "ttt_profile_read": ([_P, ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_double)], _I),
        "ttt_kernel_class_name": ([_I], ctypes.c_char_p),
        "ttt_kernel_class_count": ([], _I),
        "ttt_last_launch_count": ([_P, ctypes.POINTER(ctypes.c_longlong)], _I),
        "ttt_operand_storage": ([_P], _I),
        "ttt_launch_log_enable": ([_P, _I], _I),
        "ttt_launch_log_read": ([_P, ctypes.POINTER(ctypes.c_int8), _I], _I),
        "ttt_status_string": ([_I], ctypes.c_char_p),
        "ttt_last_error": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != 0:
        detail = _lib.ttt_last_error().decode(errors="replace") if _lib else ""
        raise TTTError(status, where, detail)


def _ptr(x):
    """Data pointer of a torch tensor or numpy array (None -> NULL)."""
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        if not x.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays passed to libttt must be C-contiguous")
        return x.ctypes.data
    raise TypeError(f"unsupported buffer type {type(x)}")


def _stream(stream):
    if stream is not None:
        return stream
    try:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
    except Exception:
        pass
    return None


def kernel_classes() -> list:
    lib = load_library()
    return [lib.ttt_kernel_class_name(i).decode() for i in range(lib.ttt_kernel_class_count())]


class Handle:
    """One libttt handle: a network, its TTT hyper-parameters and B sequences."""

    def __init__(self, *, d, d_ff, vocab, n_prefix, n_fast, block, fast_mats, dtype, eta, clip, chunk,
                 B, weights, settle_every=0, settle_len=0, rms_eps=1e-6, reset_every=0, static_mlp=False,
                 attn_heads=0, attn_window=0, options=None):
        """weights: {"E", "U", "prefix": [block dicts], "fast": [block dicts]};
        with static_mlp, "static": one frozen MLP (block dict) per fast block;
        with attn_heads > 0, "attn": one {"Wq", "Wk", "Wv", "Wo"} per prefix block.
        options: {field of ttt_options: int} (omitted fields keep the defaults)."""
        self.lib = load_library()
        self.block = block
        self.mats = MATS[block]
        self.B, self.V, self.chunk = B, vocab, chunk
        self.d, self.d_ff, self.n_fast = d, d_ff, n_fast
        self.fast_mats = tuple(fast_mats)
        mask = 0
        for m in fast_mats:
            mask |= FAST_BIT[m]
        self._dims = Dims(d, d_ff, vocab, n_prefix, n_fast, BLOCK[block], mask, DTYPE[dtype], rms_eps,
                          1 if static_mlp else 0, attn_heads, attn_window)
        self._hp = HParams(eta, clip, chunk, settle_every, B, settle_len, reset_every)
        keep = []

        def f32(a):
            if hasattr(a, "data_ptr"):
                import torch
                t = a.detach().to(torch.float32).contiguous()
                keep.append(t)
                return t.data_ptr()
            arr = np.ascontiguousarray(a, dtype=np.float32)
            keep.append(arr)
            return arr.ctypes.data

        pre = [f32(b[m]) for b in weights["prefix"] for m in self.mats]
        fst = [f32(b[m]) for b in weights["fast"] for m in self.mats]
        pre_arr = (ctypes.c_void_p * max(1, len(pre)))(*pre)
        fst_arr = (ctypes.c_void_p * len(fst))(*fst)
        sta = [f32(b[m]) for b in weights["static"] for m in self.mats] if static_mlp else []
        sta_arr = (ctypes.c_void_p * max(1, len(sta)))(*sta)
        att = [f32(b[m]) for b in weights["attn"] for m in ("Wq", "Wk", "Wv", "Wo")] if attn_heads else []
        att_arr = (ctypes.c_void_p * max(1, len(att)))(*att)
        w = Weights(f32(weights["E"]), f32(weights["U"]),
                    ctypes.cast(pre_arr, ctypes.POINTER(ctypes.c_void_p)),
                    ctypes.cast(fst_arr, ctypes.POINTER(ctypes.c_void_p)),
                    ctypes.cast(sta_arr, ctypes.POINTER(ctypes.c_void_p)) if static_mlp else None,
                    ctypes.cast(att_arr, ctypes.POINTER(ctypes.c_void_p)) if attn_heads else None)
        h = ctypes.c_void_p()
        self._opt = Options(**{k: int(v) for k, v in (options or {}).items()})
        _check(self.lib.ttt_create_ex(ctypes.byref(self._dims), ctypes.byref(self._hp), ctypes.byref(w),
                                      ctypes.byref(self._opt), ctypes.byref(h)), "ttt_create_ex")
        self._h = h
        del keep

    @classmethod
    def from_workload(cls, wl, weights, B=None, options=None):
        return cls(d=wl.d, d_ff=wl.d_ff, vocab=wl.vocab, n_prefix=wl.n_prefix, n_fast=wl.n_fast,
                   block=wl.block, fast_mats=wl.fast_mats, dtype=wl.dtype, eta=wl.eta, clip=wl.clip,
                   chunk=wl.chunk, B=wl.B if B is None else B, weights=weights,
                   settle_every=wl.settle_every, settle_len=wl.settle_len, rms_eps=wl.rms_eps,
                   reset_every=wl.reset_every, static_mlp=wl.static_mlp, attn_heads=wl.attn_heads,
                   attn_window=wl.attn_window, options=options)

    def close(self):
        if getattr(self, "_h", None):
            self.lib.ttt_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---------------------------------------------------------------- calls
    def prefill(self, tokens, losses, p_next=None, settle_q=None, accept=None, A=None, stream=None,
                loss_mask=None):
        """tokens [B, T+1] int32; losses [B, T] float32 out; the rest optional.
        loss_mask [B, T] uint8 (Source Masking): only targets whose entry is
        non-zero enter the updates (every token is still scored)."""
        B, T1 = tokens.shape
        Lq = 0 if settle_q is None else settle_q.shape[-1]
        if loss_mask is None:
            _check(self.lib.ttt_prefill(self._h, _ptr(tokens), B, T1 - 1, _ptr(losses), _ptr(p_next),
                                        _ptr(settle_q), Lq, _ptr(accept), _ptr(A), _stream(stream)),
                   "ttt_prefill")
        else:
            _check(self.lib.ttt_prefill_masked(self._h, _ptr(tokens), _ptr(loss_mask), B, T1 - 1, _ptr(losses),
                                               _ptr(p_next), _ptr(settle_q), Lq, _ptr(accept), _ptr(A),
                                               _stream(stream)), "ttt_prefill_masked")

    def decode_step(self, x_new, p_next, loss=None, stream=None):
        _check(self.lib.ttt_decode_step(self._h, _ptr(x_new), _ptr(p_next), _ptr(loss), _stream(stream)),
               "ttt_decode_step")

    def settle(self, q, accept, A, stream=None):
        _check(self.lib.ttt_settle(self._h, _ptr(q), q.shape[-1], _ptr(accept), _ptr(A), _stream(stream)),
               "ttt_settle")

    def fast_weight(self, seq, block, mat, out=None):
        """fp32 master of one fast matrix of one sequence (numpy unless `out` given)."""
        mi = self.mats.index(mat) if isinstance(mat, str) else mat
        shape = (self.d_ff, self.d) if self.mats[mi] in ("W1", "Wg", "Wu") else (self.d, self.d_ff)
        dst = np.empty(shape, dtype=np.float32) if out is None else out
        _check(self.lib.ttt_get_fast_weights(self._h, seq, block, mi, _ptr(dst), _stream(None)),
               "ttt_get_fast_weights")
        return dst

    def fast_weights(self, seq):
        return [{m: self.fast_weight(seq, l, m) for m in self.fast_mats} for l in range(self.n_fast)]

    def reset(self):
        _check(self.lib.ttt_reset(self._h, _stream(None)), "ttt_reset")

    def get_state(self) -> bytes:
        n = ctypes.c_size_t()
        _check(self.lib.ttt_state_size(self._h, ctypes.byref(n)), "ttt_state_size")
        buf = np.empty(n.value, dtype=np.uint8)
        _check(self.lib.ttt_get_state(self._h, buf.ctypes.data, n.value, _stream(None)), "ttt_get_state")
        return buf

    def set_state(self, blob):
        blob = np.ascontiguousarray(blob, dtype=np.uint8)
        _check(self.lib.ttt_set_state(self._h, blob.ctypes.data, blob.size, _stream(None)), "ttt_set_state")

    def profile_enable(self, kernel_class):
        if isinstance(kernel_class, str):
            kernel_class = kernel_classes().index(kernel_class)
        _check(self.lib.ttt_profile_enable(self._h, kernel_class), "ttt_profile_enable")

    def profile_read(self):
        n = ctypes.c_int()
        ms = ctypes.c_double()
        _check(self.lib.ttt_profile_read(self._h, ctypes.byref(n), ctypes.byref(ms)), "ttt_profile_read")
        return n.value, ms.value

    def operand_storage(self) -> str:
        """The arithmetic of the handle's GEMMs: "f32", "bf16" or "bf16x3"."""
        return {0: "f32", 1: "bf16", 2: "bf16x3"}[self.lib.ttt_operand_storage(self._h)]

    def last_launch_count(self) -> int:
        n = ctypes.c_longlong()
        _check(self.lib.ttt_last_launch_count(self._h, ctypes.byref(n)), "ttt_last_launch_count")
        return n.value

    def launch_log_enable(self, on: bool = True):
        _check(self.lib.ttt_launch_log_enable(self._h, int(on)), "ttt_launch_log_enable")

    def launch_log(self) -> list:
        """Kernel class names of the logged launches, in launch order."""
        n = self.lib.ttt_launch_log_read(self._h, None, 0)
        buf = (ctypes.c_int8 * max(n, 1))()
        self.lib.ttt_launch_log_read(self._h, buf, n)
        names = kernel_classes()
        return [names[buf[i]] for i in range(n)]


# ---------------------------------------------------------------- single operations
EPI = {"store": 0, "store_f32": 1, "gelu": 2, "resid": 3, "swiglu": 4, "dgelu": 5, "dw": 6}
GEMM_IMPL = {"auto": 0, "simt": 1, "tensor": 2}


class GemmArgs(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int), ("batch", ctypes.c_int),
                ("dtype", ctypes.c_int), ("a_kmajor", ctypes.c_int), ("b_kmajor", ctypes.c_int),
                ("epi", ctypes.c_int), ("impl", ctypes.c_int),
                ("A", ctypes.c_void_p), ("lda", ctypes.c_longlong), ("sA", ctypes.c_longlong),
                ("B", ctypes.c_void_p), ("ldb", ctypes.c_longlong), ("sB", ctypes.c_longlong),
                ("out", ctypes.c_void_p), ("ldo", ctypes.c_longlong), ("sO", ctypes.c_longlong),
                ("out2", ctypes.c_void_p), ("ldo2", ctypes.c_longlong), ("sO2", ctypes.c_longlong),
                ("aux", ctypes.c_void_p), ("ldx", ctypes.c_longlong), ("sX", ctypes.c_longlong),
                ("partials", ctypes.c_void_p),
                ("loA", ctypes.c_longlong), ("loB", ctypes.c_longlong), ("loO", ctypes.c_longlong),
                ("loO2", ctypes.c_longlong), ("loX", ctypes.c_longlong),
                ("workspace", ctypes.c_void_p), ("workspace_elems", ctypes.c_longlong)]


def _ops_lib():
    lib = load_library()
    if not getattr(lib, "_ops_ready", False):
        sig = {
            "ttt_op_gemm": ([ctypes.POINTER(GemmArgs), _P], _I),
            "ttt_op_gemm_partial_tiles": ([ctypes.POINTER(GemmArgs)], _I),
            "ttt_op_cross_entropy": ([_I, _I, _I, _P, _P, ctypes.c_float, _I, _P, _P], _I),
            "ttt_op_rmsnorm_forward": ([_I, _I, _I, _P, ctypes.c_float, _P, _P, _P], _I),
            "ttt_op_rmsnorm_backward": ([_I, _I, _I, _P, _P, _P, _P, _P, _P], _I),
            "ttt_clip_sgd": ([_I, _I, _I, ctypes.c_longlong, _P, _P, _P, ctypes.c_float, ctypes.c_float,
                              _P, _P, _P, ctypes.c_size_t, _P], _I),
            "ttt_clip_sgd_workspace_size": ([_I, _I, ctypes.c_longlong], ctypes.c_size_t),
            "ttt_op_sliding_window_attention": ([_I, _I, _I, _I, _I, _I, _P, _I, ctypes.c_longlong, _P, _P], _I),
            "ttt_clip_sgd_noalloc": ([_I, _I, _I, ctypes.c_longlong, _P, _P, _P, ctypes.c_float,
                                      ctypes.c_float, _P, _P, _P], _I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        lib._ops_ready = True
    return lib


def gemm_args(M, N, K, A, B, out, *, batch=1, dtype="bf16", a_kmajor=True, b_kmajor=True, epi="store",
              impl="auto", lda=None, sA=0, ldb=None, sB=0, ldo=None, sO=0, out2=None, ldo2=0, sO2=0,
              aux=None, ldx=0, sX=0, partials=None, loA=0, loB=0, loO=0, loO2=0, loX=0, workspace=None):
    """dtype: "fp32", "bf16" or "bf16x3" (fp32 values as bf16 hi/lo planes, lo offsets lo*)."""
    code = {"fp32": 0, "bf16": 1, "bf16x3": 2}[dtype]
    return GemmArgs(M, N, K, batch, code, int(a_kmajor), int(b_kmajor), EPI[epi], GEMM_IMPL[impl],
                    _ptr(A), lda if lda is not None else (K if a_kmajor else M), sA,
                    _ptr(B), ldb if ldb is not None else (K if b_kmajor else N), sB,
                    _ptr(out), ldo if ldo is not None else N, sO, _ptr(out2), ldo2, sO2,
                    _ptr(aux), ldx, sX, _ptr(partials), loA, loB, loO, loO2, loX,
                    _ptr(workspace), 0 if workspace is None else workspace.numel())


def op_gemm(args: GemmArgs, stream=None):
    _check(_ops_lib().ttt_op_gemm(ctypes.byref(args), _stream(stream)), "ttt_op_gemm")


def op_gemm_partial_tiles(args: GemmArgs) -> int:
    return _ops_lib().ttt_op_gemm_partial_tiles(ctypes.byref(args))


def op_cross_entropy(dtype, logits, targets, scale, grad, losses, stream=None):
    M, V = logits.shape
    _check(_ops_lib().ttt_op_cross_entropy(DTYPE[dtype], M, V, _ptr(logits), _ptr(targets), scale, int(grad),
                                           _ptr(losses), _stream(stream)), "ttt_op_cross_entropy")


def op_rmsnorm_forward(dtype, x, eps, y, rstd, stream=None):
    M, d = x.shape
    _check(_ops_lib().ttt_op_rmsnorm_forward(DTYPE[dtype], M, d, _ptr(x), eps, _ptr(y), _ptr(rstd),
                                             _stream(stream)), "ttt_op_rmsnorm_forward")


def op_rmsnorm_backward(dtype, x, rstd, dy, dx, dx_op=None, stream=None):
    M, d = x.shape
    _check(_ops_lib().ttt_op_rmsnorm_backward(DTYPE[dtype], M, d, _ptr(x), _ptr(rstd), _ptr(dy), _ptr(dx),
                                              _ptr(dx_op), _stream(stream)), "ttt_op_rmsnorm_backward")


def op_sliding_window_attention(qkv, rows, heads, window, pad, out, stream=None):
    """qkv [B, L, 3d] bf16 device tensor (position p at row pad + p); out [B, L, d]."""
    B, L, d3 = qkv.shape
    d = d3 // 3
    _check(_ops_lib().ttt_op_sliding_window_attention(1, B, rows, heads, d // heads, window, _ptr(qkv), pad, L,
                                                      _ptr(out), _stream(stream)), "ttt_op_sliding_window_attention")


def clip_sgd_workspace_size(nslots, B, n) -> int:
    return _ops_lib().ttt_clip_sgd_workspace_size(nslots, B, n)


def clip_sgd(dtype, W32, Wop, dW, eta, clip, norm_out=None, scale_out=None, workspace=None, stream=None):
    """W32, Wop, dW: [nslots, B, n] device tensors; workspace: device byte tensor."""
    nslots, B, n = W32.shape
    _check(_ops_lib().ttt_clip_sgd(DTYPE[dtype], nslots, B, n, _ptr(W32), _ptr(Wop), _ptr(dW), eta, clip,
                                   _ptr(norm_out), _ptr(scale_out), _ptr(workspace),
                                   0 if workspace is None else workspace.numel() * workspace.element_size(),
                                   _stream(stream)), "ttt_clip_sgd")


def clip_sgd_noalloc(dtype, W32, Wop, dW, eta, clip, norm_out=None, scale_out=None, stream=None):
    """ttt_clip_sgd with the library's fixed device scratch instead of a workspace."""
    nslots, B, n = W32.shape
    _check(_ops_lib().ttt_clip_sgd_noalloc(DTYPE[dtype], nslots, B, n, _ptr(W32), _ptr(Wop), _ptr(dW), eta,
                                           clip, _ptr(norm_out), _ptr(scale_out), _stream(stream)),
           "ttt_clip_sgd_noalloc")
