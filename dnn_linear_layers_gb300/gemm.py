"""ctypes binding of the C-ABI library (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module
turns torch tensors into (pointer, shape, leading dimension) triples and the
current torch stream into a ``cudaStream_t``.  It never computes a result on
its own: if the library is missing or a call fails, it raises.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libgb300gemm.so"

EPI_NONE, EPI_BIAS, EPI_RELU, EPI_BIAS_RELU = 0, 1, 2, 3
BF16_F32OUT, BF16_BF16OUT, F16_F32OUT, F16_F16OUT = 0, 1, 2, 3
E4M3_F32OUT, E4M3_BF16OUT, E5M2_F32OUT, E5M2_BF16OUT = 4, 5, 6, 7
TF32_F32OUT, TF32_BF16OUT = 8, 9   # fp32 A and B, multiplied at tf32 precision
FP8_DTYPES = (torch.float8_e4m3fn, torch.float8_e5m2)
B_KN, B_NK, B_CONST, A_KM = 0, 1, 2, 8
OPT_GROUP_M, OPT_TAIL_SPLIT, OPT_K_SNAKE, OPT_PDL, OPT_L2_POLICY = 1, 2, 3, 4, 5
OPT_SKINNY_SPLITS, OPT_SKINNY_STAGES, OPT_LOG, OPT_GEMV_MAX_M, OPT_STREAM_K = 6, 7, 9, 10, 11
OPT_WARP_MMA_MAX_M = 12
OPTIONS = (OPT_GROUP_M, OPT_TAIL_SPLIT, OPT_K_SNAKE, OPT_PDL, OPT_L2_POLICY, OPT_SKINNY_SPLITS, OPT_SKINNY_STAGES,
           OPT_LOG, OPT_GEMV_MAX_M, OPT_STREAM_K, OPT_WARP_MMA_MAX_M)
KERNEL_AUTO, KERNEL_TC_PAIR, KERNEL_TC_SINGLE, KERNEL_FILL, KERNEL_SKINNY, KERNEL_GEMV = 0, 1, 2, 3, 4, 5
KERNEL_WARP_MMA = 6
OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_NO_MEMORY = (
    0, -1, -2, -3, -4, -5, -6)

# Every symbol include/gemm.h declares, with its ctypes signature.
_vp, _i64, _int, _uint, _u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint, ctypes.c_uint64


class EpilogueArgs(ctypes.Structure):
    """gemm_epilogue_args_t: t = alpha*acc; t *= scale[j]; t += bias[j];
    t += beta*C_old[i][j]; ReLU; cast."""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("scale", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("relu", ctypes.c_int)]


_epi_p = ctypes.POINTER(EpilogueArgs)
SIGNATURES = {
    "gemm_plan_create": (_int, [ctypes.POINTER(_vp), _int, _uint]),
    "gemm_run": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i64, _int, _int, _vp]),
    "gemm_plan_status": (_int, [_vp]),
    "gemm_plan_destroy": (_int, [_vp]),
    "gemm_strerror": (ctypes.c_char_p, [_int]),
    "gemm_plan_set_kernel": (_int, [_vp, _int]),
    "gemm_plan_last_kernel": (_int, [_vp]),
    "gemm_plan_launch_count": (_i64, [_vp]),
    "gemm_plan_last_cuda_error": (_int, [_vp]),
    "gemm_plan_set_timeout_ns": (_int, [_vp, _u64]),
    "gemm_plan_set_packing": (_int, [_vp, _int]),
    "gemm_plan_set_debug": (_int, [_vp, _uint]),
    "gemm_plan_workspace_bytes": (_i64, [_vp]),
    "gemm_plan_set_option": (_int, [_vp, _int, _i64]),
    "gemm_plan_get_option": (_int, [_vp, _int, ctypes.POINTER(_i64)]),
    "gemm_validate": (_int, [_uint, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i64, _int, _int]),
    "gemm_im2col": (_int, [_vp, _i64, _i64, _i64, _i64, _int, _int, _int, _int, _vp, _i64, _int, _vp]),
    "gemm_run_noalloc": (_int, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i64, _int, _int, _uint, _vp, _vp]),
    "gemm_conv2d": (_int, [_vp, _i64, _i64, _i64, _i64, _i64, _int, _int, _int, _vp, _vp, _vp, _i64, _epi_p, _int,
                           _vp]),
    "gemm_run_ex": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _epi_p, _int, _vp]),
    "gemm_attention": (_int, [_vp, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, ctypes.c_float, _int, _int, _vp]),
    "gemm_conv2d_maxpool": (_int, [_vp, _i64, _i64, _i64, _i64, _i64, _int, _int, _int, _vp, _vp, _vp, _i64, _epi_p,
                                   _int, _vp]),
}

_lib = None


class GemmError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})" if what else f"{strerror(code)} ({code})")


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run dnn_linear_layers_gb300/build.py or __graft_entry__.build())")
        l = ctypes.CDLL(str(LIB_PATH))
        for name, (res, args) in SIGNATURES.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def strerror(code: int) -> str:
    return lib().gemm_strerror(code).decode()


def _check(code: int, what: str):
    if code != OK:
        raise GemmError(code, what)


def dtype_code(in_dtype: torch.dtype, out_dtype: torch.dtype) -> int:
    table = {(torch.bfloat16, torch.float32): BF16_F32OUT, (torch.bfloat16, torch.bfloat16): BF16_BF16OUT,
             (torch.float16, torch.float32): F16_F32OUT, (torch.float16, torch.float16): F16_F16OUT,
             (torch.float8_e4m3fn, torch.float32): E4M3_F32OUT, (torch.float8_e4m3fn, torch.bfloat16): E4M3_BF16OUT,
             (torch.float8_e5m2, torch.float32): E5M2_F32OUT, (torch.float8_e5m2, torch.bfloat16): E5M2_BF16OUT,
             (torch.float32, torch.float32): TF32_F32OUT, (torch.float32, torch.bfloat16): TF32_BF16OUT}
    try:
        return table[(in_dtype, out_dtype)]
    except KeyError:
        raise ValueError(f"unsupported dtype pair {in_dtype} -> {out_dtype}") from None


def vector_dtype(in_dtype: torch.dtype) -> torch.dtype:
    """dtype of the bias and scale vectors for an input dtype (bf16 for fp8 and fp32 / tf32 inputs)."""
    return torch.bfloat16 if in_dtype in FP8_DTYPES or in_dtype == torch.float32 else in_dtype


def _ld(t: torch.Tensor) -> int:
    """Leading dimension (elements) of a row-major 2-D view with unit column stride."""
    if t.dim() != 2 or (t.stride(1) != 1 and t.shape[1] > 1):
        raise ValueError("operands must be 2-D row-major views with unit column stride")
    return max(t.stride(0), t.shape[1], 1)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


class Plan:
    """Owner of a ``gemm_plan_t``.  ``b_layout`` is "kn" (B is K x N) or "nk"
    (B is a Linear weight W, N x K); ``a_layout`` is "mk" (A is M x K) or "km"
    (A is stored K x M, the transposed operand)."""

    def __init__(self, device: int | torch.device = 0, b_layout: str = "kn", b_const: bool = False,
                 a_layout: str = "mk"):
        if isinstance(device, torch.device):
            device = device.index if device.index is not None else torch.cuda.current_device()
        self.device = int(device)
        if b_layout not in ("kn", "nk") or a_layout not in ("mk", "km"):
            raise ValueError("b_layout is 'kn' or 'nk', a_layout 'mk' or 'km'")
        self.b_nk = b_layout == "nk"
        self.a_km = a_layout == "km"
        flags = (B_NK if self.b_nk else B_KN) | (B_CONST if b_const else 0) | (A_KM if self.a_km else 0)
        h = _vp()
        _check(lib().gemm_plan_create(ctypes.byref(h), self.device, flags), "gemm_plan_create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            lib().gemm_plan_destroy(self._h)
            self._h = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- controls ---------------------------------------------------------
    def set_kernel(self, kernel: int):
        _check(lib().gemm_plan_set_kernel(self._h, kernel), "gemm_plan_set_kernel")

    def set_timeout_ns(self, ns: int):
        _check(lib().gemm_plan_set_timeout_ns(self._h, int(ns)), "gemm_plan_set_timeout_ns")

    def set_packing(self, enabled: bool):
        _check(lib().gemm_plan_set_packing(self._h, int(bool(enabled))), "gemm_plan_set_packing")

    def set_debug(self, flags: int):
        _check(lib().gemm_plan_set_debug(self._h, int(flags)), "gemm_plan_set_debug")

    def set_option(self, option: int, value: int):
        """Set a GEMM_OPT_* scheduling option (sweeps and tests)."""
        _check(lib().gemm_plan_set_option(self._h, int(option), int(value)), "gemm_plan_set_option")

    def get_option(self, option: int) -> int:
        v = ctypes.c_int64()
        _check(lib().gemm_plan_get_option(self._h, int(option), ctypes.byref(v)), "gemm_plan_get_option")
        return v.value

    @property
    def last_kernel(self) -> int:
        return lib().gemm_plan_last_kernel(self._h)

    @property
    def launch_count(self) -> int:
        return lib().gemm_plan_launch_count(self._h)

    @property
    def workspace_bytes(self) -> int:
        return lib().gemm_plan_workspace_bytes(self._h)

    def status(self) -> int:
        """Synchronise and return the device status (0 or a GEMM_ERR_* code)."""
        return lib().gemm_plan_status(self._h)

    # -- the call -----------------------------------------------------------
    def run_raw(self, M, N, K, A_ptr, lda, B_ptr, ldb, bias_ptr, C_ptr, ldc, epilogue, dtype, stream=None) -> int:
        return lib().gemm_run(self._h, M, N, K, A_ptr, lda, B_ptr, ldb, bias_ptr, C_ptr, ldc,
                              epilogue, dtype, _stream_handle(stream))

    def run(self, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, bias: torch.Tensor | None = None,
            relu: bool = False, stream=None, alpha: float = 1.0, beta: float = 0.0,
            scale: torch.Tensor | None = None):
        """C = relu?(alpha * (A . B) * scale + bias + beta * C), written into the
        caller's C (gemm_run, or gemm_run_ex when alpha, beta or scale is set)."""
        M, K = (A.shape[1], A.shape[0]) if self.a_km else (A.shape[0], A.shape[1])
        N = B.shape[0] if self.b_nk else B.shape[1]
        if (B.shape[1] if self.b_nk else B.shape[0]) != K or tuple(C.shape) != (M, N):
            raise ValueError(f"shape mismatch: A {tuple(A.shape)} B {tuple(B.shape)} C {tuple(C.shape)}")
        if A.dtype != B.dtype or (bias is not None and bias.dtype != vector_dtype(A.dtype)):
            raise ValueError("A and B must share one input dtype; bias takes that dtype (bf16 for fp8)")
        for t in (A, B, C) + ((bias,) if bias is not None else ()):
            if t.device.type != "cuda":
                raise ValueError("operands must be CUDA tensors")
        if bias is not None and (bias.dim() != 1 or bias.shape[0] != N or bias.stride(0) != 1):
            raise ValueError("bias must be a contiguous vector of length N")
        if scale is not None and (scale.dim() != 1 or scale.shape[0] != N or scale.stride(0) != 1
                                  or scale.dtype != vector_dtype(A.dtype) or scale.device.type != "cuda"):
            raise ValueError("scale must be a contiguous CUDA vector of length N in the bias dtype")
        if alpha != 1.0 or beta != 0.0 or scale is not None:
            ea = _epilogue_args(alpha, beta, scale, bias, relu)
            rc = lib().gemm_run_ex(self._h, M, N, K, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), C.data_ptr(), _ld(C),
                                   ctypes.byref(ea), dtype_code(A.dtype, C.dtype), _stream_handle(stream))
            _check(rc, "gemm_run_ex")
            return C
        epi = (EPI_BIAS if bias is not None else 0) | (EPI_RELU if relu else 0)
        rc = self.run_raw(M, N, K, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B),
                          bias.data_ptr() if bias is not None else None, C.data_ptr(), _ld(C), epi,
                          dtype_code(A.dtype, C.dtype), stream)
        _check(rc, "gemm_run")
        return C

    def conv2d(self, x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, bias: torch.Tensor | None = None,
               relu: bool = False, pad: int = 0, stream=None, alpha: float = 1.0, beta: float = 0.0,
               scale: torch.Tensor | None = None):
        """Stride-1 convolution of the NHWC tensor x (Nb x H x W x C) with
        w (Cout x R x S x C) into y ((Nb*OH*OW) x Cout, row-major)."""
        if x.dim() != 4 or w.dim() != 4 or not x.is_contiguous() or not w.is_contiguous():
            raise ValueError("x (NHWC) and w (Cout x R x S x C) must be contiguous 4-D tensors")
        Nb, H, W, C = x.shape
        Cout, R, S, Cw = w.shape
        OH, OW = H + 2 * pad - R + 1, W + 2 * pad - S + 1
        if Cw != C or tuple(y.shape) != (Nb * OH * OW, Cout):
            raise ValueError(f"shape mismatch: x {tuple(x.shape)} w {tuple(w.shape)} y {tuple(y.shape)}")
        if x.dtype != w.dtype or (bias is not None and bias.dtype != x.dtype):
            raise ValueError("x, w and bias must share one input dtype")
        for t in (x, w, y) + ((bias,) if bias is not None else ()):
            if t.device.type != "cuda":
                raise ValueError("operands must be CUDA tensors")
        if bias is not None and (bias.dim() != 1 or bias.shape[0] != Cout or bias.stride(0) != 1):
            raise ValueError("bias must be a contiguous vector of length Cout")
        if scale is not None and (scale.dim() != 1 or scale.shape[0] != Cout or scale.stride(0) != 1
                                  or scale.dtype != x.dtype or scale.device.type != "cuda"):
            raise ValueError("scale must be a contiguous CUDA vector of length Cout in the input dtype")
        ea = _epilogue_args(alpha, beta, scale, bias, relu)
        rc = lib().gemm_conv2d(self._h, Nb, H, W, C, Cout, R, S, pad, x.data_ptr(), w.data_ptr(),
                               y.data_ptr(), _ld(y), ctypes.byref(ea), dtype_code(x.dtype, y.dtype),
                               _stream_handle(stream))
        _check(rc, "gemm_conv2d")
        return y

    def attention(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                  scale: float = 0.0, causal: bool = False, stream=None):
        """o = softmax(scale * q k^T) v per (batch, head); q, o: [B, H, Sq, D],
        k, v: [B, H, Sk, D], contiguous; scale 0 means 1 / sqrt(D)."""
        if q.dim() != 4 or k.dim() != 4 or v.dim() != 4 or o.dim() != 4:
            raise ValueError("q, k, v, o must be [B, H, S, D]")
        B, H, Sq, D = q.shape
        Sk = k.shape[2]
        if tuple(k.shape) != (B, H, Sk, D) or tuple(v.shape) != (B, H, Sk, D) or tuple(o.shape) != (B, H, Sq, D):
            raise ValueError("shape mismatch")
        for t in (q, k, v, o):
            if not t.is_contiguous() or t.device.type != "cuda":
                raise ValueError("q, k, v, o must be contiguous CUDA tensors")
        if k.dtype != q.dtype or v.dtype != q.dtype:
            raise ValueError("q, k, v must share one dtype")
        rc = lib().gemm_attention(self._h, B, H, Sq, Sk, D, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  float(scale), int(bool(causal)), dtype_code(q.dtype, o.dtype),
                                  _stream_handle(stream))
        _check(rc, "gemm_attention")
        return o

    def conv2d_maxpool(self, x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, bias: torch.Tensor | None = None,
                       relu: bool = False, pad: int = 0, stream=None, alpha: float = 1.0,
                       scale: torch.Tensor | None = None):
        """Stride-1 convolution, epilogue (alpha, scale, bias, ReLU) and 2 x 2
        max-pool in one kernel; y is ((Nb*OH/2*OW/2) x Cout)."""
        if x.dim() != 4 or w.dim() != 4 or not x.is_contiguous() or not w.is_contiguous():
            raise ValueError("x (NHWC) and w (Cout x R x S x C) must be contiguous 4-D tensors")
        Nb, H, W, C = x.shape
        Cout, R, S, Cw = w.shape
        OH, OW = H + 2 * pad - R + 1, W + 2 * pad - S + 1
        if Cw != C or tuple(y.shape) != (Nb * (OH // 2) * (OW // 2), Cout):
            raise ValueError(f"shape mismatch: x {tuple(x.shape)} w {tuple(w.shape)} y {tuple(y.shape)}")
        ea = _epilogue_args(alpha, 0.0, scale, bias, relu)
        rc = lib().gemm_conv2d_maxpool(self._h, Nb, H, W, C, Cout, R, S, pad, x.data_ptr(), w.data_ptr(),
                                       y.data_ptr(), _ld(y), ctypes.byref(ea), dtype_code(x.dtype, y.dtype),
                                       _stream_handle(stream))
        _check(rc, "gemm_conv2d_maxpool")
        return y


def _epilogue_args(alpha, beta, scale, bias, relu) -> EpilogueArgs:
    return EpilogueArgs(float(alpha), float(beta), scale.data_ptr() if scale is not None else None,
                        bias.data_ptr() if bias is not None else None, int(bool(relu)))


_plans: dict = {}


def _plan_for(device: torch.device, b_layout: str) -> Plan:
    key = (device.index if device.index is not None else torch.cuda.current_device(), b_layout)
    p = _plans.get(key)
    if p is None:
        p = _plans[key] = Plan(key[0], b_layout)
    return p


def matmul(A: torch.Tensor, B: torch.Tensor, out_dtype: torch.dtype | None = None,
           bias: torch.Tensor | None = None, relu: bool = False, out: torch.Tensor | None = None):
    """C = A . B (+bias) (ReLU) with B stored K x N."""
    out_dtype = out_dtype or A.dtype
    if out is None:
        out = torch.empty(A.shape[0], B.shape[1], device=A.device, dtype=out_dtype)
    return _plan_for(A.device, "kn").run(A, B, out, bias, relu)


def linear(x: torch.Tensor, weight: torch.Tensor, bias: torch.Tensor | None = None, relu: bool = False,
           out_dtype: torch.dtype | None = None, out: torch.Tensor | None = None):
    """Linear layer y = x W^T + b (W stored out x in, as ``torch.nn.Linear`` keeps it)."""
    out_dtype = out_dtype or x.dtype
    if out is None:
        out = torch.empty(x.shape[0], weight.shape[0], device=x.device, dtype=out_dtype)
    return _plan_for(x.device, "nk").run(x, weight, out, bias, relu)


def conv2d(x: torch.Tensor, w: torch.Tensor, bias: torch.Tensor | None = None, relu: bool = False, pad: int = 0,
           out_dtype: torch.dtype | None = None, out: torch.Tensor | None = None):
    """Stride-1 convolution, NHWC activations, weights Cout x R x S x C; returns
    the (Nb*OH*OW) x Cout output (NHWC flattened)."""
    Nb, H, W, _ = x.shape
    Cout, R, S, _ = w.shape
    if out is None:
        out = torch.empty(Nb * (H + 2 * pad - R + 1) * (W + 2 * pad - S + 1), Cout, device=x.device,
                          dtype=out_dtype or x.dtype)
    return _plan_for(x.device, "nk").conv2d(x, w, out, bias, relu, pad)


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
              scale: float | None = None, out_dtype: torch.dtype | None = None, out: torch.Tensor | None = None):
    """Attention forward o = softmax(scale * q k^T) v per (batch, head): q is
    [B, H, Sq, D], k and v [B, H, Sk, D] (D 64 or 128, bf16 or fp16); scale None
    means 1 / sqrt(D); causal: key j visible to query i iff j <= i + (Sk - Sq)."""
    if out is None:
        out = torch.empty(tuple(q.shape), device=q.device, dtype=out_dtype or q.dtype)
    return _plan_for(q.device, "nk").attention(q, k, v, out, scale=0.0 if scale is None else scale, causal=causal)


def im2col(x: torch.Tensor, R: int, S: int, pad: int = 0, stride: int = 1, out: torch.Tensor | None = None):
    """Explicit-GEMM matrix of an R x S convolution of the NHWC tensor ``x``."""
    if x.dim() != 4 or not x.is_contiguous() or x.device.type != "cuda":
        raise ValueError("x must be a contiguous NHWC CUDA tensor")
    Nb, H, W, C = x.shape
    OH = (H + 2 * pad - R) // stride + 1
    OW = (W + 2 * pad - S) // stride + 1
    if out is None:
        out = torch.empty((Nb * OH * OW, R * S * C), dtype=x.dtype, device=x.device)
    _check(lib().gemm_im2col(x.data_ptr(), Nb, H, W, C, R, S, pad, stride, out.data_ptr(), _ld(out),
                             x.element_size(), _stream_handle(None)), "gemm_im2col")
    return out
