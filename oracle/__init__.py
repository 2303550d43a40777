"""CPU oracle for the W8A8 block-FP8 linear layer (test infrastructure).

Only the tests, the smoke check and the bench's CPU-baseline leg import this
package. It wraps ``fp8_block_oracle.c`` (plain C, built with gcc) through
ctypes and shares nothing with the CUDA path.

Every function's parity is pinned by ``tests/test_oracle_pins.py``; see the
C file's header for the definition it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_block_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfp8_block_oracle.so")

_lock = threading.Lock()
_lib = None

OK, ERR_SHAPE, ERR_NONFINITE, ERR_NAN_CODE = 0, 1, 2, 3
G = 128


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2 -fopenmp, IEEE arithmetic)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # FP8_ORACLE_LIB names a prebuilt copy; the mutation test uses it to
            # load an oracle with a deliberately planted mistake.
            override = os.environ.get("FP8_ORACLE_LIB")
            lib = ctypes.CDLL(override if override else build())
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.oracle_e4m3_table.argtypes = [p]
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode_array.argtypes = [p, i64, p]
            lib.oracle_act_quant.argtypes = [p, i64, i64, p, p]
            lib.oracle_weight_quant.argtypes = [p, i64, i64, p, p]
            lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
            lib.oracle_bf16_from_double.restype = ctypes.c_uint16
            lib.oracle_block_gemm_rows.argtypes = [p, p, p, p, i64, i64, i64, p, i64, p, p, p]
            lib.oracle_block_gemm_w8a16_rows.argtypes = [p, p, p, i64, i64, i64, p, i64, p, p, p]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _check(status: int, what: str) -> None:
    if status != OK:
        names = {ERR_SHAPE: "bad shape", ERR_NONFINITE: "non-finite input",
                 ERR_NAN_CODE: "E4M3 NaN code in input"}
        raise OracleError(f"{what}: {names.get(status, status)}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def e4m3_table() -> np.ndarray:
    """float32[256]: the value of every E4M3 code (NaN for 0x7F, 0xFF)."""
    out = np.empty(256, np.float32)
    _load().oracle_e4m3_table(_ptr(out))
    return out


def e4m3_encode(f) -> np.ndarray:
    """uint8 codes of fp32 values: nearest even, saturating to +-448."""
    a = np.ascontiguousarray(np.asarray(f, dtype=np.float32))
    out = np.empty(a.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(a), a.size, _ptr(out))
    return out


def act_quant(x_bits: np.ndarray):
    """bf16 bits uint16 [M, K] -> (q uint8 [M, K], sa float32 [M, K/128])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    sa = np.empty((M, K // G), np.float32)
    _check(_load().oracle_act_quant(_ptr(x), M, K, _ptr(q), _ptr(sa)), "act_quant")
    return q, sa


def weight_quant(w_bits: np.ndarray):
    """bf16 bits uint16 [N, K] -> (w uint8 [N, K], sw float32 [ceil(N/128), K/128])."""
    W = np.ascontiguousarray(w_bits, dtype=np.uint16)
    N, K = W.shape
    w = np.empty((N, K), np.uint8)
    sw = np.empty(((N + G - 1) // G, K // G), np.float32)
    _check(_load().oracle_weight_quant(_ptr(W), N, K, _ptr(w), _ptr(sw)), "weight_quant")
    return w, sw


def bf16_from_double(y: float) -> int:
    """bf16 bits of an fp64 value, nearest even, rounded in one step."""
    return int(_load().oracle_bf16_from_double(float(y)))


def block_gemm(q, sa, w, sw, rows=None):
    """Exact block-scaled GEMM.

    Returns (y float64 [R, N], aabs float64 [R, N], out bf16 bits uint16 [R, N]),
    R = M, or len(rows) for a row subset.
    """
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = q.shape
    N = w.shape[0]
    if w.shape[1] != K or sa.shape != (M, K // G) or sw.shape != ((N + G - 1) // G, K // G):
        raise OracleError("block_gemm: inconsistent shapes")
    if rows is None:
        rows_arr, R, rows_p = None, M, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        R, rows_p = rows_arr.size, _ptr(rows_arr)
    y = np.empty((R, N), np.float64)
    aabs = np.empty((R, N), np.float64)
    out = np.empty((R, N), np.uint16)
    _check(_load().oracle_block_gemm_rows(_ptr(q), _ptr(sa), _ptr(w), _ptr(sw), M, N, K,
                                          rows_p, R if rows is not None else 0,
                                          _ptr(y), _ptr(aabs), _ptr(out)), "block_gemm")
    return y, aabs, out


def block_gemm_w8a16(x_bits, w, sw, rows=None):
    """Weight-only block-FP8 GEMM: bf16 activations (raw uint16 bits [M, K])
    times E4M3 weights with 128x128 fp32 block scales, no activation quant.

    Returns (y float64 [R, N], aabs float64 [R, N], out bf16 bits uint16 [R, N]).
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K or sw.shape != ((N + G - 1) // G, K // G):
        raise OracleError("block_gemm_w8a16: inconsistent shapes")
    if rows is None:
        R, rows_p = M, None
    else:
        keep = np.ascontiguousarray(rows, dtype=np.int64)
        R, rows_p = keep.size, _ptr(keep)
    y = np.empty((R, N), np.float64)
    aabs = np.empty((R, N), np.float64)
    out = np.empty((R, N), np.uint16)
    _check(_load().oracle_block_gemm_w8a16_rows(_ptr(x), _ptr(w), _ptr(sw), M, N, K, rows_p,
                                                R if rows is not None else 0, _ptr(y), _ptr(aabs), _ptr(out)),
           "block_gemm_w8a16")
    return y, aabs, out
