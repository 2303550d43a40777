"""The C-ABI library builds for sm_103a, loads, exports every declared symbol and
rejects bad arguments on the host (no kernel runs in these tests)."""
from __future__ import annotations

import ctypes

import pytest

from block_scaled_fp8_act_gb300 import build as fp8build
from block_scaled_fp8_act_gb300 import fp8act

OK, NULL, SHAPE, ALIGN, LAUNCH, TIMEOUT, DEVICE, CUDA = range(8)


@pytest.fixture(scope="module")
def lib():
    fp8build.build()
    return fp8act.load()


def test_library_exports_every_header_symbol(lib):
    names = fp8act.header_symbols()
    assert {"fp8_act_quant", "fp8_weight_quant", "fp8_block_gemm", "fp8_block_gemm_f32",
            "fp8_block_gemm_w8a16", "fp8_block_gemm_w8a16_f32",
            "fp8_act_quant_grouped", "fp8_block_gemm_grouped", "fp8_block_gemm_grouped_f32",
            "fp8_linear", "fp8_linear_f32",
            "fp8act_strerror", "fp8act_check_status", "fp8act_version"} <= set(names)
    raw = ctypes.CDLL(fp8act.lib_path())
    for n in names:
        assert hasattr(raw, n), n


def test_strerror_and_version(lib):
    for s in range(8):
        assert fp8act.strerror(s)
    assert "unknown" in fp8act.strerror(99)
    assert lib.fp8act_version() >= 100


A16 = 0x10000  # a fake 16-byte-aligned address: never dereferenced, the checks run first


def test_act_quant_argument_checks(lib):
    f = lib.fp8_act_quant
    assert f(A16, 1, 100, A16, A16, None) == SHAPE      # K % 128
    assert f(A16, 1, 0, A16, A16, None) == SHAPE        # K == 0
    assert f(A16, -1, 128, A16, A16, None) == SHAPE
    assert f(None, 0, 128, None, None, None) == OK      # empty: no launch, no pointer use
    assert f(None, 1, 128, A16, A16, None) == NULL
    assert f(A16 + 8, 1, 128, A16, A16, None) == ALIGN
    assert f(A16, 1, 128, A16 + 4, A16, None) == ALIGN
    assert f(A16, 1, 128, A16, A16 + 2, None) == ALIGN


def test_weight_quant_argument_checks(lib):
    f = lib.fp8_weight_quant
    assert f(A16, 128, 129, A16, A16, None) == SHAPE
    assert f(A16, -5, 128, A16, A16, None) == SHAPE
    assert f(None, 0, 128, None, None, None) == OK
    assert f(A16, 128, 128, None, A16, None) == NULL
    assert f(A16, 128, 128, A16 + 1, A16, None) == ALIGN


@pytest.mark.parametrize("name", ["fp8_block_gemm", "fp8_block_gemm_f32"])
def test_gemm_argument_checks(lib, name):
    f = getattr(lib, name)
    assert f(A16, A16, A16, A16, 1, 128, 64, A16, None) == SHAPE
    assert f(A16, A16, A16, A16, -1, 128, 128, A16, None) == SHAPE
    assert f(A16, A16, A16, A16, 1, -1, 128, A16, None) == SHAPE
    assert f(None, None, None, None, 0, 128, 128, None, None) == OK
    assert f(None, None, None, None, 4, 0, 128, None, None) == OK
    assert f(A16, None, A16, A16, 1, 128, 128, A16, None) == NULL
    assert f(A16, A16, A16 + 8, A16, 1, 128, 128, A16, None) == ALIGN
    assert f(A16, A16, A16, A16 + 1, 1, 128, 128, A16, None) == ALIGN
    assert f(A16, A16, A16, A16, 1, 128, 128, A16 + 2, None) == ALIGN


def test_valid_call_without_a_gb300_is_refused(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    assert lib.fp8_block_gemm(A16, A16, A16, A16, 1, 128, 128, A16, None) == DEVICE
    assert lib.fp8_act_quant(A16, 1, 128, A16, A16, None) == DEVICE


@pytest.mark.parametrize("name", ["fp8_block_gemm_w8a16", "fp8_block_gemm_w8a16_f32"])
def test_w8a16_argument_checks(lib, name):
    f = getattr(lib, name)
    assert f(A16, A16, A16, 1, 128, 64, A16, None) == SHAPE
    assert f(A16, A16, A16, -1, 128, 128, A16, None) == SHAPE
    assert f(None, None, None, 0, 128, 128, None, None) == OK
    assert f(A16, None, A16, 1, 128, 128, A16, None) == NULL
    assert f(A16 + 8, A16, A16, 1, 128, 128, A16, None) == ALIGN
    assert f(A16, A16, A16 + 2, 1, 128, 128, A16, None) == ALIGN
    assert f(A16, A16, A16, 1, 128, 128, A16 + 4, None) == ALIGN


def test_grouped_structs_match_the_header():
    import re
    import os
    text = open(os.path.join(fp8build.INCLUDE, "fp8act.h"), encoding="utf-8").read()
    for cname, py in (("fp8act_quant_problem", fp8act.QuantProblem), ("fp8act_gemm_problem", fp8act.GemmProblem)):
        body = re.search(r"typedef struct \{([^{}]*)\}\s*" + cname + ";", text).group(1)
        names = re.findall(r"(\w+)(?:,|;)", re.sub(r"/\*.*?\*/", "", body, flags=re.S))
        assert names == [f[0] for f in py._fields_], (cname, names)
    assert ctypes.sizeof(fp8act.QuantProblem) == 32
    assert ctypes.sizeof(fp8act.GemmProblem) == 56


@pytest.mark.parametrize("name", ["fp8_block_gemm_grouped", "fp8_block_gemm_grouped_f32"])
def test_gemm_grouped_argument_checks(lib, name):
    f = getattr(lib, name)
    P = fp8act.GemmProblem
    assert f(None, 0, None) == OK
    assert f(None, 2, None) == NULL
    arr = (P * 17)()
    assert f(ctypes.byref(arr), 17, None) == SHAPE
    assert f(ctypes.byref(arr), -1, None) == SHAPE
    good = P(A16, A16, A16, A16, A16, 1, 128, 128)
    arr = (P * 3)(good, P(A16, A16, A16, A16, A16, 1, 128, 64), good)
    assert f(ctypes.byref(arr), 3, None) == SHAPE       # second entry: K % 128
    arr = (P * 2)(good, P(A16, A16, None, A16, A16, 1, 128, 128))
    assert f(ctypes.byref(arr), 2, None) == NULL
    arr = (P * 2)(good, P(A16, A16, A16 + 8, A16, A16, 1, 128, 128))
    assert f(ctypes.byref(arr), 2, None) == ALIGN
    arr = (P * 2)(P(None, None, None, None, None, 0, 128, 128), P(None, None, None, None, None, 3, 0, 256))
    assert f(ctypes.byref(arr), 2, None) == OK           # only empty problems: nothing to launch


def test_act_quant_grouped_argument_checks(lib):
    f = lib.fp8_act_quant_grouped
    P = fp8act.QuantProblem
    assert f(None, 0, None) == OK
    assert f(None, 1, None) == NULL
    good = P(A16, A16, A16, 1, 128)
    arr = (P * 2)(good, P(A16, A16, A16, 1, 100))
    assert f(ctypes.byref(arr), 2, None) == SHAPE
    arr = (P * 2)(good, P(A16, A16 + 4, A16, 1, 128))
    assert f(ctypes.byref(arr), 2, None) == ALIGN
    arr = (P * 1)(P(None, None, None, 0, 128))
    assert f(ctypes.byref(arr), 1, None) == OK


@pytest.mark.parametrize("name", ["fp8_linear", "fp8_linear_f32"])
def test_linear_argument_checks(lib, name):
    f = getattr(lib, name)
    assert f(A16, A16, A16, 1, 128, 64, A16, None) == SHAPE
    assert f(A16, A16, A16, -1, 128, 128, A16, None) == SHAPE
    assert f(A16, A16, A16, 8, 128, 25 * 1024, A16, None) == SHAPE   # 8 rows of K codes exceed 200 KiB
    assert f(None, None, None, 0, 128, 128, None, None) == OK
    assert f(A16, None, A16, 1, 128, 128, A16, None) == NULL
    assert f(A16 + 8, A16, A16, 1, 128, 128, A16, None) == ALIGN
    assert f(A16, A16, A16 + 2, 1, 128, 128, A16, None) == ALIGN
