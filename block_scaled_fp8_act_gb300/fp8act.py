"""ctypes binding of libfp8act.so (argument marshalling only).

Each function takes CUDA torch tensors, checks dtype / device / contiguity,
passes raw device pointers, sizes and the current CUDA stream to the C entry
point of the same name (include/fp8act.h) and raises Fp8ActError on a
non-zero status. All arithmetic runs in the library's CUDA kernels; there is
no fallback: if the library is not built, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

G = 128
_lib = None

STATUS = {0: "FP8ACT_OK", 1: "FP8ACT_ERR_NULL", 2: "FP8ACT_ERR_SHAPE", 3: "FP8ACT_ERR_ALIGN",
          4: "FP8ACT_ERR_LAUNCH", 5: "FP8ACT_ERR_TIMEOUT", 6: "FP8ACT_ERR_DEVICE", 7: "FP8ACT_ERR_CUDA"}


class Fp8ActError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {STATUS.get(status, status)}: {msg}")
        self.status = status


def header_symbols() -> list[str]:
    """Names of the entry points include/fp8act.h declares."""
    text = open(os.path.join(_build.INCLUDE, "fp8act.h"), encoding="utf-8").read()
    return re.findall(r"FP8ACT_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def lib_path() -> str:
    return _build.LIB_PATH


def load(build: bool = False) -> ctypes.CDLL:
    """Load libfp8act.so (compiling it first when build=True)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build else _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libfp8act.so is not built ({path}); run block_scaled_fp8_act_gb300.build.build()")
    L = ctypes.CDLL(path)
    p, i = ctypes.c_void_p, ctypes.c_int
    L.fp8_act_quant.argtypes = [p, i, i, p, p, p]
    L.fp8_weight_quant.argtypes = [p, i, i, p, p, p]
    L.fp8_block_gemm.argtypes = [p, p, p, p, i, i, i, p, p]
    L.fp8_block_gemm_f32.argtypes = [p, p, p, p, i, i, i, p, p]
    L.fp8_block_gemm_w8a16.argtypes = [p, p, p, i, i, i, p, p]
    L.fp8_block_gemm_w8a16_f32.argtypes = [p, p, p, i, i, i, p, p]
    L.fp8_linear.argtypes = [p, p, p, i, i, i, p, p]
    L.fp8_linear_f32.argtypes = [p, p, p, i, i, i, p, p]
    L.fp8_act_quant_grouped.argtypes = [p, i, p]
    L.fp8_block_gemm_grouped.argtypes = [p, i, p]
    L.fp8_block_gemm_grouped_f32.argtypes = [p, i, p]
    L.fp8act_strerror.argtypes = [i]
    L.fp8act_strerror.restype = ctypes.c_char_p
    L.fp8act_check_status.argtypes = [p]
    L.fp8act_set_wait_limit.argtypes = [ctypes.c_longlong, i]
    L.fp8act_stream_read.argtypes = [p, ctypes.c_size_t, p, p]
    for fn in (L.fp8_act_quant, L.fp8_weight_quant, L.fp8_block_gemm, L.fp8_block_gemm_f32,
               L.fp8_block_gemm_w8a16, L.fp8_block_gemm_w8a16_f32,
               L.fp8_act_quant_grouped, L.fp8_block_gemm_grouped, L.fp8_block_gemm_grouped_f32,
               L.fp8_linear, L.fp8_linear_f32,
               L.fp8act_check_status, L.fp8act_set_wait_limit, L.fp8act_version, L.fp8act_stream_read):
        fn.restype = ctypes.c_int
    _lib = L
    return L


def strerror(status: int) -> str:
    return load().fp8act_strerror(int(status)).decode()


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream))


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise Fp8ActError(fn, status, strerror(status))


def _cuda2d(t: torch.Tensor, dtypes, name: str) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D tensor")


_CODES = (torch.uint8, torch.float8_e4m3fn)


def fp8_act_quant(x: torch.Tensor, q: torch.Tensor | None = None, sa: torch.Tensor | None = None, stream=None):
    """x bf16 [M, K] -> (q uint8 E4M3 codes [M, K], sa fp32 [M, K/128])."""
    _cuda2d(x, (torch.bfloat16,), "x")
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device) if q is None else q
    sa = torch.empty((M, K // G), dtype=torch.float32, device=x.device) if sa is None else sa
    _cuda2d(q, _CODES, "q")
    _cuda2d(sa, (torch.float32,), "sa")
    if q.shape != (M, K) or sa.shape != (M, K // G):
        raise ValueError("q / sa have the wrong shape")
    _check("fp8_act_quant", load().fp8_act_quant(x.data_ptr(), M, K, q.data_ptr(), sa.data_ptr(), _stream(stream)))
    return q, sa


def fp8_weight_quant(W: torch.Tensor, w: torch.Tensor | None = None, sw: torch.Tensor | None = None, stream=None):
    """W bf16 [N, K] -> (w uint8 E4M3 codes [N, K], sw fp32 [ceil(N/128), K/128])."""
    _cuda2d(W, (torch.bfloat16,), "W")
    N, K = W.shape
    NB = (N + G - 1) // G
    w = torch.empty((N, K), dtype=torch.uint8, device=W.device) if w is None else w
    sw = torch.empty((NB, K // G), dtype=torch.float32, device=W.device) if sw is None else sw
    _cuda2d(w, _CODES, "w")
    _cuda2d(sw, (torch.float32,), "sw")
    if w.shape != (N, K) or sw.shape != (NB, K // G):
        raise ValueError("w / sw have the wrong shape")
    _check("fp8_weight_quant", load().fp8_weight_quant(W.data_ptr(), N, K, w.data_ptr(), sw.data_ptr(),
                                                       _stream(stream)))
    return w, sw


def _gemm(fn_name: str, out_dtype, q, sa, w, sw, out, stream):
    for t, n, d in ((q, "q", _CODES), (sa, "sa", (torch.float32,)), (w, "w", _CODES), (sw, "sw", (torch.float32,))):
        _cuda2d(t, d, n)
    M, K = q.shape
    N = w.shape[0]
    if w.shape[1] != K or sa.shape != (M, K // G) or sw.shape != ((N + G - 1) // G, K // G):
        raise ValueError("inconsistent q / sa / w / sw shapes")
    out = torch.empty((M, N), dtype=out_dtype, device=q.device) if out is None else out
    _cuda2d(out, (out_dtype,), "out")
    if out.shape != (M, N):
        raise ValueError("out has the wrong shape")
    fn = getattr(load(), fn_name)
    _check(fn_name, fn(q.data_ptr(), sa.data_ptr(), w.data_ptr(), sw.data_ptr(), M, N, K, out.data_ptr(),
                       _stream(stream)))
    return out


def fp8_block_gemm(q, sa, w, sw, out=None, stream=None) -> torch.Tensor:
    """bf16 [M, N] = block-scaled q [M, K] x w [N, K]^T."""
    return _gemm("fp8_block_gemm", torch.bfloat16, q, sa, w, sw, out, stream)


def fp8_block_gemm_f32(q, sa, w, sw, out=None, stream=None) -> torch.Tensor:
    """fp32 [M, N] output of the same kernels (no bf16 cast)."""
    return _gemm("fp8_block_gemm_f32", torch.float32, q, sa, w, sw, out, stream)


def fp8_linear(x, w, sw, out=None, stream=None) -> torch.Tensor:
    """bf16 [M, N] = fp8_block_gemm(fp8_act_quant(x), w, sw) in one launch (decode-sized M)."""
    return _gemm_w8a16("fp8_linear", torch.bfloat16, x, w, sw, out, stream)


def fp8_linear_f32(x, w, sw, out=None, stream=None) -> torch.Tensor:
    """fp32 [M, N] output of the fused kernels (no bf16 cast)."""
    return _gemm_w8a16("fp8_linear_f32", torch.float32, x, w, sw, out, stream)


def _gemm_w8a16(fn_name: str, out_dtype, x, w, sw, out, stream):
    _cuda2d(x, (torch.bfloat16,), "x")
    _cuda2d(w, _CODES, "w")
    _cuda2d(sw, (torch.float32,), "sw")
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K or sw.shape != ((N + G - 1) // G, K // G):
        raise ValueError("inconsistent x / w / sw shapes")
    out = torch.empty((M, N), dtype=out_dtype, device=x.device) if out is None else out
    _cuda2d(out, (out_dtype,), "out")
    if out.shape != (M, N):
        raise ValueError("out has the wrong shape")
    fn = getattr(load(), fn_name)
    _check(fn_name, fn(x.data_ptr(), w.data_ptr(), sw.data_ptr(), M, N, K, out.data_ptr(), _stream(stream)))
    return out


def fp8_block_gemm_w8a16(x, w, sw, out=None, stream=None) -> torch.Tensor:
    """bf16 [M, N] = bf16 x [M, K] times block-scaled E4M3 w [N, K]^T (no activation quantisation)."""
    return _gemm_w8a16("fp8_block_gemm_w8a16", torch.bfloat16, x, w, sw, out, stream)


def fp8_block_gemm_w8a16_f32(x, w, sw, out=None, stream=None) -> torch.Tensor:
    """fp32 [M, N] output of the weight-only kernels (no bf16 cast)."""
    return _gemm_w8a16("fp8_block_gemm_w8a16_f32", torch.float32, x, w, sw, out, stream)


class QuantProblem(ctypes.Structure):
    """fp8act_quant_problem of include/fp8act.h."""
    _fields_ = [("x_bf16", ctypes.c_void_p), ("q_e4m3", ctypes.c_void_p), ("sa", ctypes.c_void_p),
                ("M", ctypes.c_int), ("K", ctypes.c_int)]


class GemmProblem(ctypes.Structure):
    """fp8act_gemm_problem of include/fp8act.h."""
    _fields_ = [("q_e4m3", ctypes.c_void_p), ("sa", ctypes.c_void_p), ("w_e4m3", ctypes.c_void_p),
                ("sw", ctypes.c_void_p), ("out", ctypes.c_void_p), ("M", ctypes.c_int), ("N", ctypes.c_int),
                ("K", ctypes.c_int)]


MAX_GROUPED = 16


def fp8_act_quant_grouped(xs, outs=None, stream=None):
    """Quantise several bf16 activations [M_i, K_i] in one launch.

    Returns [(q_i, sa_i)]; `outs` may supply them."""
    if len(xs) > MAX_GROUPED:
        raise ValueError(f"at most {MAX_GROUPED} problems per grouped call")
    res = []
    arr = (QuantProblem * max(1, len(xs)))()
    for i, x in enumerate(xs):
        _cuda2d(x, (torch.bfloat16,), "x")
        M, K = x.shape
        if outs is None:
            q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
            sa = torch.empty((M, K // G), dtype=torch.float32, device=x.device)
        else:
            q, sa = outs[i]
        _cuda2d(q, _CODES, "q")
        _cuda2d(sa, (torch.float32,), "sa")
        if q.shape != (M, K) or sa.shape != (M, K // G):
            raise ValueError("q / sa have the wrong shape")
        arr[i] = QuantProblem(x.data_ptr(), q.data_ptr(), sa.data_ptr(), M, K)
        res.append((q, sa))
    _check("fp8_act_quant_grouped", load().fp8_act_quant_grouped(ctypes.byref(arr), len(xs), _stream(stream)))
    return res


def _gemm_grouped(fn_name: str, out_dtype, problems, outs, stream):
    if len(problems) > MAX_GROUPED:
        raise ValueError(f"at most {MAX_GROUPED} problems per grouped call")
    res = []
    arr = (GemmProblem * max(1, len(problems)))()
    for i, (q, sa, w, sw) in enumerate(problems):
        for t, n, d in ((q, "q", _CODES), (sa, "sa", (torch.float32,)), (w, "w", _CODES),
                        (sw, "sw", (torch.float32,))):
            _cuda2d(t, d, n)
        M, K = q.shape
        N = w.shape[0]
        if w.shape[1] != K or sa.shape != (M, K // G) or sw.shape != ((N + G - 1) // G, K // G):
            raise ValueError("inconsistent q / sa / w / sw shapes")
        out = torch.empty((M, N), dtype=out_dtype, device=q.device) if outs is None else outs[i]
        _cuda2d(out, (out_dtype,), "out")
        if out.shape != (M, N):
            raise ValueError("out has the wrong shape")
        arr[i] = GemmProblem(q.data_ptr(), sa.data_ptr(), w.data_ptr(), sw.data_ptr(), out.data_ptr(), M, N, K)
        res.append(out)
    _check(fn_name, getattr(load(), fn_name)(ctypes.byref(arr), len(problems), _stream(stream)))
    return res


def fp8_block_gemm_grouped(problems, outs=None, stream=None) -> list:
    """Several block GEMMs [(q, sa, w, sw), ...] in one launch; returns the bf16 outputs."""
    return _gemm_grouped("fp8_block_gemm_grouped", torch.bfloat16, problems, outs, stream)


def fp8_block_gemm_grouped_f32(problems, outs=None, stream=None) -> list:
    """fp32 outputs of the grouped kernels (no bf16 cast)."""
    return _gemm_grouped("fp8_block_gemm_grouped_f32", torch.float32, problems, outs, stream)


def check_status(stream=None) -> int:
    """Synchronise the stream and return the library's device-side status."""
    return int(load().fp8act_check_status(_stream(stream)))


def set_wait_limit(limit_ns: int, withhold_first_load: bool = False) -> None:
    """Test hook of the tcgen05 kernels' failure path (see fp8act_set_wait_limit):
    the wall-time bound of their waits (negative = the 2 s default) and whether
    each CTA skips its first operand copy."""
    _check("fp8act_set_wait_limit", load().fp8act_set_wait_limit(int(limit_ns), 1 if withhold_first_load else 0))


def stream_read(src: torch.Tensor, sink: torch.Tensor, stream=None) -> None:
    """Diagnostic: read every byte of the CUDA tensor `src` once (the weight-stream
    floor), folding it into the int32 CUDA tensor `sink` (see fp8act_stream_read)."""
    if not src.is_cuda or not src.is_contiguous() or not sink.is_cuda or sink.dtype != torch.int32:
        raise TypeError("src must be a contiguous CUDA tensor and sink an int32 CUDA tensor")
    _check("fp8act_stream_read", load().fp8act_stream_read(src.data_ptr(), src.numel() * src.element_size(),
                                                           sink.data_ptr(), _stream(stream)))
