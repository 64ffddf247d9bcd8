"""The C ABI library loads without a GPU and exports every function that
include/*.h declares (no compute calls here)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(ttt_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from chunked_next_token_ttt_b300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_headers_declare_the_boundary():
    names = declared_functions()
    for required in ("ttt_create", "ttt_prefill", "ttt_decode_step", "ttt_settle", "ttt_get_fast_weights",
                     "ttt_reset", "ttt_destroy", "ttt_status_string", "ttt_op_gemm", "ttt_clip_sgd"):
        assert required in names


def test_every_declared_function_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_only_calls_work_without_a_gpu(lib):
    lib.ttt_status_string.restype = ctypes.c_char_p
    assert lib.ttt_status_string(0) == b"ok"
    assert lib.ttt_status_string(5).startswith(b"non-finite")
    lib.ttt_kernel_class_count.restype = ctypes.c_int
    assert lib.ttt_kernel_class_count() > 5
    lib.ttt_clip_sgd_workspace_size.restype = ctypes.c_size_t
    lib.ttt_clip_sgd_workspace_size.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_longlong]
    assert lib.ttt_clip_sgd_workspace_size(2, 3, 10000) == (2 * 3 * 2 + 3 + 1) * 4
    # argument validation happens before any CUDA call
    lib.ttt_create.restype = ctypes.c_int
    assert lib.ttt_create(None, None, None, None) == 1


def test_binding_fails_loudly_without_the_library(tmp_path):
    from chunked_next_token_ttt_b300 import ttt
    with pytest.raises(RuntimeError):
        ttt._lib_saved = ttt._lib
        ttt._lib = None
        try:
            ttt.load_library(str(tmp_path / "missing.so"))
        finally:
            ttt._lib = ttt._lib_saved


def test_reset_with_settlement_is_rejected_before_any_cuda_call():
    """The periodic reset and Settlement are alternatives: ttt_create refuses
    the pair with BAD_ARG during validation, which runs without a GPU."""
    import synth
    from synth import configs as C
    from chunked_next_token_ttt_b300 import Handle, TTTError
    wl = C.SETTLE_760M.replace(d=16, d_ff=32, vocab=64, n_prefix=1, n_fast=1, B=2, reset_every=8)
    with pytest.raises(TTTError) as e:
        Handle.from_workload(wl, synth.make_weights(wl))
    assert e.value.status == 1


def test_static_mlp_outside_gelu_blocks_is_unsupported_before_any_cuda_call():
    import synth
    from synth import configs as C
    from chunked_next_token_ttt_b300 import Handle, TTTError
    wl = C.INPLACE_4B.replace(d=16, d_ff=32, vocab=64, n_prefix=1, B=1, static_mlp=True)
    with pytest.raises(TTTError) as e:
        Handle.from_workload(wl, synth.make_weights(wl))
    assert e.value.status == 7


def test_no_environment_variable_steers_the_library():
    """Execution choices are ttt_options fields: no library source reads the
    environment, so a caller's environment cannot change results or speed."""
    import glob
    csrc = os.path.join(ROOT, "chunked_next_token_ttt_b300", "csrc")
    for path in glob.glob(os.path.join(csrc, "*")):
        with open(path) as f:
            assert "getenv" not in f.read(), path
