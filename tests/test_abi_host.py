"""Host-only checks of the C-ABI library: it builds, loads without a GPU,
exports every symbol include/gemm.h declares, and validates arguments exactly
as documented (no device needed, nothing launched)."""
import ctypes
import re
from pathlib import Path

import pytest
import torch

from dnn_linear_layers_gb300 import build as B
from dnn_linear_layers_gb300 import gemm as G

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def lib():
    B.build()
    return G.lib()


def declared_functions():
    text = (ROOT / "include" / "gemm.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\*]+\s+\**\s*(gemm_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for core in ("gemm_plan_create", "gemm_run", "gemm_plan_status", "gemm_plan_destroy", "gemm_strerror"):
        assert core in names
    assert set(names) == set(G.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert G.strerror(code) and G.strerror(code) != "unknown error"
    assert G.strerror(17) == "unknown error"


P = ctypes.c_void_p(0x1000)   # any non-null, 16-byte aligned host value: validate never dereferences


def val(flags=0, M=64, N=64, K=64, A=P, lda=64, Bp=P, ldb=64, bias=None, C=P, ldc=64, epi=0, dtype=1):
    return G.lib().gemm_validate(flags, M, N, K, A, lda, Bp, ldb, bias, C, ldc, epi, dtype)


def test_validate_accepts_good_arguments(lib):
    assert val() == G.OK
    assert val(flags=G.B_NK, N=32, ldb=64, ldc=32) == G.OK
    assert val(epi=G.EPI_BIAS_RELU, bias=P) == G.OK


def test_validate_rejects_bad_arguments(lib):
    assert val(M=-1) == G.ERR_INVALID_ARG
    assert val(K=-5) == G.ERR_INVALID_ARG
    assert val(epi=4) == G.ERR_INVALID_ARG
    assert val(dtype=10) == G.ERR_INVALID_ARG
    assert val(dtype=G.TF32_F32OUT) == G.OK and val(dtype=G.TF32_BF16OUT) == G.OK
    assert val(flags=16) == G.ERR_INVALID_ARG
    assert val(flags=4) == G.ERR_INVALID_ARG             # not a flag
    # A stored K x M: lda counts M
    assert val(flags=G.A_KM, M=96, K=32, lda=96, ldc=64) == G.OK
    assert val(flags=G.A_KM, M=96, K=32, lda=95, ldc=64) == G.ERR_INVALID_ARG    # lda < M
    assert val(flags=G.A_KM, M=32, K=96, lda=32, ldc=64) == G.OK                 # lda < K is fine here
    assert val(flags=G.B_NK | G.B_CONST, N=32, ldb=64, ldc=32) == G.OK
    assert val(lda=63) == G.ERR_INVALID_ARG               # lda < K
    assert val(ldb=63) == G.ERR_INVALID_ARG               # ldb < N (K x N layout)
    assert val(flags=G.B_NK, K=128, lda=128, ldb=64) == G.ERR_INVALID_ARG   # ldb < K (N x K layout)
    assert val(ldc=10) == G.ERR_INVALID_ARG
    assert val(A=None) == G.ERR_INVALID_ARG
    assert val(Bp=None) == G.ERR_INVALID_ARG
    assert val(C=None) == G.ERR_INVALID_ARG
    assert val(epi=G.EPI_BIAS, bias=None) == G.ERR_INVALID_ARG
    assert val(M=2 ** 31, lda=64) == G.ERR_UNSUPPORTED


def test_validate_rejects_pointers_off_their_element_boundary(lib):
    odd, two = ctypes.c_void_p(0x1001), ctypes.c_void_p(0x1002)
    assert val(A=odd) == G.ERR_INVALID_ARG                       # bf16 A one byte off
    assert val(Bp=odd) == G.ERR_INVALID_ARG
    assert val(A=two, Bp=two) == G.OK                            # 2-byte boundary: fine for bf16
    assert val(C=two, dtype=G.BF16_F32OUT) == G.ERR_INVALID_ARG  # fp32 C two bytes off
    assert val(C=two, dtype=G.BF16_BF16OUT) == G.OK
    assert val(epi=G.EPI_BIAS, bias=odd) == G.ERR_INVALID_ARG
    assert val(A=two, dtype=G.TF32_F32OUT) == G.ERR_INVALID_ARG  # fp32 operands: 4-byte boundary
    assert val(A=odd, Bp=odd, dtype=G.E4M3_F32OUT) == G.OK        # fp8: any byte
    assert val(epi=G.EPI_BIAS, bias=two, dtype=G.E4M3_F32OUT) == G.OK   # bf16 bias of an fp8 product
    assert val(K=0, A=odd, Bp=odd) == G.OK                       # A and B not read


def test_validate_size_zero_is_a_noop(lib):
    assert val(M=0, A=None, Bp=None, C=None) == G.OK
    assert val(N=0, A=None, Bp=None, C=None) == G.OK
    # K == 0: A and B are not read, but C is written (epilogue of 0)
    assert val(K=0, A=None, Bp=None, lda=0) == G.OK
    assert val(K=0, A=None, Bp=None, C=None) == G.ERR_INVALID_ARG


def test_null_plan_is_rejected(lib):
    assert lib.gemm_run(None, 1, 1, 1, P, 1, P, 1, None, P, 1, 0, 1, None) == G.ERR_INVALID_ARG
    assert lib.gemm_plan_status(None) == G.ERR_INVALID_ARG
    assert lib.gemm_plan_destroy(None) == G.OK
    assert lib.gemm_plan_set_kernel(None, 0) == G.ERR_INVALID_ARG
    assert lib.gemm_plan_last_kernel(None) == -1
    assert lib.gemm_plan_set_option(None, G.OPT_GROUP_M, 8) == G.ERR_INVALID_ARG
    v = ctypes.c_int64(-7)
    assert lib.gemm_plan_get_option(None, G.OPT_GROUP_M, ctypes.byref(v)) == G.ERR_INVALID_ARG
    assert v.value == -7


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks behaviour on a host without a GPU")
def test_plan_create_without_gpu_returns_error(lib):
    h = ctypes.c_void_p()
    rc = lib.gemm_plan_create(ctypes.byref(h), 0, 0)
    assert rc in (G.ERR_CUDA, G.ERR_INVALID_ARG)
    assert h.value is None
    assert lib.gemm_plan_create(None, 0, 0) == G.ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(G, "LIB_PATH", tmp_path / "missing.so")
    monkeypatch.setattr(G, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        G.lib()


def test_conv2d_rejects_null_plan(lib):
    assert G.lib().gemm_conv2d(None, 1, 8, 8, 64, 64, 3, 3, 1, P, P, P, 64, None, 1, None) == G.ERR_INVALID_ARG


def test_run_ex_rejects_null_plan_and_args(lib):
    ea = G.EpilogueArgs(1.0, 0.0, None, None, 0)
    assert G.lib().gemm_run_ex(None, 8, 8, 8, P, 8, P, 8, P, 8, ctypes.byref(ea), 1, None) == G.ERR_INVALID_ARG


def test_noalloc_refuses_the_operand_forms_it_does_not_take(lib):
    # checked after argument validation and before any CUDA call
    args = dict(M=64, N=64, K=64, lda=64, ldb=64, ldc=64)
    def call(dtype, flags):
        return lib.gemm_run_noalloc(args["M"], args["N"], args["K"], P, args["lda"], P, args["ldb"], None, P,
                                    args["ldc"], 0, dtype, flags, None, None)
    for dtype in (G.E4M3_F32OUT, G.E5M2_BF16OUT, G.TF32_F32OUT, G.TF32_BF16OUT):
        assert call(dtype, G.B_NK) == G.ERR_UNSUPPORTED
    # only the B-layout flag applies without a plan
    for flags in (G.A_KM, G.B_CONST, G.B_NK | G.B_CONST, 4):
        assert call(G.BF16_F32OUT, flags) == G.ERR_INVALID_ARG


def test_attention_rejects_null_plan_and_bad_arguments(lib):
    assert lib.gemm_attention(None, 1, 1, 8, 8, 64, P, P, P, P, 0.0, 0, G.BF16_F32OUT, None) == G.ERR_INVALID_ARG


def test_conv2d_maxpool_rejects_null_plan(lib):
    assert lib.gemm_conv2d_maxpool(None, 1, 4, 4, 64, 64, 3, 3, 1, P, P, P, 64, None, G.BF16_BF16OUT,
                                   None) == G.ERR_INVALID_ARG
