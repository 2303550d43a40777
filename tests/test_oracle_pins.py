"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one function of ``oracle/`` against a closed form of the
E4M3 / bf16 formats, an exact rational (Fraction) computation, an
invariant of the definition, or an independent library routine (torch's
float8_e4m3fn and bfloat16 converters, a float64 matmul). Together they are
chosen so that a dropped term, a wrong sign, a wrong scale index or a
transposed operand in the oracle fails at least one of them.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_act_gb300 import inputs

G = 128


# ----------------------------------------------------------------- helpers
def torch_e4m3_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float32).numpy()


def torch_e4m3_encode(vals: np.ndarray) -> np.ndarray:
    """torch's fp32 -> float8_e4m3fn conversion (nearest even; NaN from 464 up)."""
    t = torch.from_numpy(np.ascontiguousarray(vals, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def fp32_rne(x: Fraction) -> np.float32:
    """Exact round-to-nearest-even of a rational to fp32 (no double rounding)."""
    if x == 0:
        return np.float32(0.0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    # 2^e <= a < 2^(e+1); fp32 keeps 24 bits; subnormal quantum 2^-149
    qe = max(e - 23, -149)
    scaled = a / Fraction(2) ** qe
    n = math.floor(scaled)
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return np.float32(sign * math.ldexp(float(n), qe))


def bf16_rne_fraction(x: Fraction) -> int:
    """bf16 bits of the exact rational x, nearest even (8 significant bits)."""
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    qe = max(e - 7, -133)
    scaled = a / Fraction(2) ** qe
    n = math.floor(scaled)
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    f = np.float32(math.ldexp(float(n), qe))
    return sign | int(np.array([f], np.float32).view(np.uint32)[0] >> 16)


def e4m3_spacing(v: float) -> float:
    """Gap between neighbouring E4M3 values around |v| (format definition)."""
    v = abs(v)
    if v < 2.0 ** -6:
        return 2.0 ** -9
    return 2.0 ** (math.floor(math.log2(v)) - 3)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------ E4M3 table
def test_e4m3_format_landmarks():
    t = oracle.e4m3_table()
    assert t[0x00] == 0.0 and not np.signbit(t[0x00])
    assert t[0x80] == 0.0 and np.signbit(t[0x80])
    assert t[0x01] == 2.0 ** -9          # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9      # largest subnormal
    assert t[0x08] == 2.0 ** -6          # smallest normal
    assert t[0x38] == 1.0
    assert t[0x39] == 1.125
    assert t[0x7E] == 448.0              # largest finite
    assert t[0xFE] == -448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isfinite(t).sum() == 254   # no infinities, two NaN codes
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)      # monotone in the code
    assert np.array_equal(t[0x80:0xFF], -pos)
    # every finite value is an integer multiple of 2^-9
    fin = t[np.isfinite(t)].astype(np.float64) * 512
    assert np.array_equal(fin, np.round(fin))


def test_e4m3_table_matches_torch_decoder():
    t = oracle.e4m3_table()
    ref = torch_e4m3_decode(np.arange(256))
    assert np.array_equal(t, ref, equal_nan=True)
    assert np.array_equal(np.signbit(t), np.signbit(ref))


# ----------------------------------------------------------- E4M3 encode
def test_encode_roundtrip_every_finite_code():
    t = oracle.e4m3_table()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(t[codes]), codes)


def test_encode_hand_derived_ties_and_saturation():
    cases = [
        (1.0625, 0x38),            # midpoint 1.0 | 1.125 -> even 1.0
        (1.1875, 0x3A),            # midpoint 1.125 | 1.25 -> even 1.25
        (1.0625 + 2 ** -20, 0x39),  # just above a midpoint rounds up
        (1.0625 - 2 ** -20, 0x38),
        (2.0 ** -10, 0x00),        # midpoint 0 | 2^-9 -> even 0
        (3 * 2.0 ** -10, 0x02),    # midpoint 2^-9 | 2^-8 -> even 2^-8
        (7.5 * 2.0 ** -9, 0x08),   # last subnormal | first normal -> even
        (0.96875, 0x38),           # midpoint 0.9375 (0x37) | 1.0 (0x38) -> even
        (232.0, 0x76),             # midpoint 224 | 240 -> even 224
        (440.0, 0x7E),             # above the 416 | 448 midpoint (432)
        (448.0, 0x7E),
        (448.5, 0x7E),             # above max finite: saturate
        (463.99, 0x7E),
        (464.0, 0x7E),
        (1.0e30, 0x7E),
        (-1.0e30, 0xFE),
        (-0.0, 0x80),              # sign of zero kept
        (-2.0 ** -11, 0x80),       # negative value rounding to zero
        (2.0 ** -149, 0x00),
    ]
    vals = np.array([c[0] for c in cases], np.float32)
    want = np.array([c[1] for c in cases], np.uint8)
    got = oracle.e4m3_encode(vals)
    assert np.array_equal(got, want), list(zip(vals, got, want))


def test_encode_matches_torch_converter():
    rng = np.random.default_rng(7)
    mag = np.exp2(rng.uniform(-14, math.log2(463.9), 200_000)).astype(np.float32)
    vals = mag * np.where(rng.random(mag.size) < 0.5, -1, 1).astype(np.float32)
    # every exact midpoint between neighbouring codes, and one fp32 ulp either side
    t = oracle.e4m3_table()[:0x7F].astype(np.float64)
    mids = ((t[:-1] + t[1:]) / 2).astype(np.float32)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    vals = np.concatenate([vals, mids, up, dn, -mids, -up, -dn]).astype(np.float32)
    vals = vals[np.abs(vals) < 464]
    assert np.array_equal(oracle.e4m3_encode(vals), torch_e4m3_encode(vals))


# ------------------------------------------------------------ bf16 cast
def test_bf16_from_double():
    rng = np.random.default_rng(3)
    f = (rng.standard_normal(50_000) * np.exp2(rng.uniform(-140, 120, 50_000))).astype(np.float32)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_double(float(v)) for v in f], np.uint16)
    assert np.array_equal(got, want)
    # doubles that an fp32 intermediate would round onto a bf16 midpoint
    assert oracle.bf16_from_double(1 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert oracle.bf16_from_double(1 + 2 ** -8 - 2 ** -40) == 0x3F80
    assert oracle.bf16_from_double(1 + 2 ** -8) == 0x3F80          # tie -> even
    assert oracle.bf16_from_double(1 + 3 * 2 ** -8) == 0x3F82      # tie -> even
    assert oracle.bf16_from_double(-(1 + 2 ** -8 + 2 ** -40)) == 0xBF81
    assert oracle.bf16_from_double(2.0 ** -133) == 0x0001          # smallest subnormal
    assert oracle.bf16_from_double(2.0 ** -134) == 0x0000          # tie -> even (zero)
    assert oracle.bf16_from_double(1.5 * 2.0 ** -134) == 0x0001
    assert oracle.bf16_from_double(-0.0) == 0x8000


# ------------------------------------------------------------ quantisers
def _check_group_quant(xg: np.ndarray, codes: np.ndarray, s: np.float32):
    """All the facts one quantised group must satisfy, from exact arithmetic."""
    xf = xg.astype(np.float32).ravel()
    codes = codes.ravel()
    amax = float(np.max(np.abs(xf)))
    if amax == 0.0:
        assert s == np.float32(1.0)
        assert np.array_equal(codes & 0x7F, np.zeros_like(codes))
        assert np.array_equal(codes >> 7, np.signbit(xf).astype(np.uint8))
        return
    # s is the fp32 nearest to amax / 448
    assert s == fp32_rne(Fraction(amax) / 448), (amax, s)
    # each code is the E4M3 rounding (nearest even, saturating) of fp32(x / s)
    t = np.array([fp32_rne(Fraction(float(v)) / Fraction(float(s))) for v in xf], np.float32)
    want = torch_e4m3_encode(np.clip(t, -448, 448))
    want = np.where(t == 0, np.where(np.signbit(t), 0x80, 0x00), want).astype(np.uint8)
    assert np.array_equal(codes, want)
    # round trip: |dq * s - x| <= (half a code spacing at x/s + fp32 division error) * s
    dq = oracle.e4m3_table()[codes].astype(np.float64)
    ratio = xf.astype(np.float64) / float(s)
    bound = np.array([0.5 * e4m3_spacing(min(abs(r), 448.0)) for r in ratio])
    bound += np.abs(ratio) * 2.0 ** -23 + np.maximum(np.abs(ratio) - 448.0, 0)
    assert np.all(np.abs(dq - ratio) <= bound)
    # the largest-magnitude element lands on +-448 when s is a normal fp32
    if s >= np.float32(2.0 ** -126):
        i = int(np.argmax(np.abs(xf)))
        assert codes[i] & 0x7F == 0x7E
    # signs are kept
    nz = xf != 0
    assert np.array_equal((codes[nz] >> 7).astype(bool), xf[nz] < 0)


@pytest.mark.parametrize("M,K,edge", [(3, 384, False), (2, 1152, True), (1, 9 * 128, True)])
def test_act_quant_matches_exact_definition(M, K, edge):
    x = (inputs.edge_activations_bf16(M, K, seed=11 + M) if edge
         else inputs.activations_bf16(M, K, seed=5))
    q, sa = oracle.act_quant(inputs.bf16_bits(x))
    xf = x.float().numpy()
    assert q.shape == (M, K) and sa.shape == (M, K // G)
    for m in range(M):
        for kb in range(K // G):
            g = slice(kb * G, (kb + 1) * G)
            _check_group_quant(xf[m, g], q[m, g], sa[m, kb])


def test_act_quant_scale_invariance():
    x = inputs.activations_bf16(4, 512, seed=21)
    q0, s0 = oracle.act_quant(inputs.bf16_bits(x))
    for j in (-7, 3):
        xj = (x.float() * 2.0 ** j).to(torch.bfloat16)   # exact: power of two
        qj, sj = oracle.act_quant(inputs.bf16_bits(xj))
        assert np.array_equal(qj, q0)
        assert np.array_equal(sj, (s0.astype(np.float64) * 2.0 ** j).astype(np.float32))


def test_act_quant_rejects_bad_input():
    with pytest.raises(oracle.OracleError):
        oracle.act_quant(np.zeros((1, 100), np.uint16))
    bad = np.zeros((1, 128), np.uint16)
    bad[0, 5] = 0x7FC0  # bf16 NaN
    with pytest.raises(oracle.OracleError):
        oracle.act_quant(bad)
    bad[0, 5] = 0x7F80  # bf16 +inf
    with pytest.raises(oracle.OracleError):
        oracle.act_quant(bad)
    q, sa = oracle.act_quant(np.zeros((0, 256), np.uint16))
    assert q.shape == (0, 256) and sa.shape == (0, 2)


@pytest.mark.parametrize("N,K", [(200, 256), (128, 384)])
def test_weight_quant_matches_exact_definition(N, K):
    W = inputs.weights_bf16(N, K, seed=31)
    w, sw = oracle.weight_quant(inputs.bf16_bits(W))
    NB = (N + G - 1) // G
    assert w.shape == (N, K) and sw.shape == (NB, K // G)
    Wf = W.float().numpy()
    for nb in range(NB):
        for kb in range(K // G):
            r = slice(nb * G, min((nb + 1) * G, N))
            c = slice(kb * G, (kb + 1) * G)
            _check_group_quant(Wf[r, c], w[r, c], sw[nb, kb])


# ----------------------------------------------------------------- GEMM
def _quantised_problem(M, N, K, seed):
    x = inputs.activations_bf16(M, K, seed=seed)
    W = inputs.weights_bf16(N, K, seed=seed + 1)
    q, sa = oracle.act_quant(inputs.bf16_bits(x))
    w, sw = oracle.weight_quant(inputs.bf16_bits(W))
    return q, sa, w, sw


def test_gemm_brute_force_fractions():
    """Exact rational y for a tiny problem with 2 scale blocks along N and K."""
    M, N, K = 3, 200, 256
    q, sa, w, sw = _quantised_problem(M, N, K, seed=41)
    y, aabs, out = oracle.block_gemm(q, sa, w, sw)
    dq_q = torch_e4m3_decode(q)   # torch's decoder, not the oracle's table
    dq_w = torch_e4m3_decode(w)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            for k in range(K):
                exact += (Fraction(float(sa[m, k // G])) * Fraction(float(sw[n // G, k // G]))
                          * Fraction(float(dq_q[m, k])) * Fraction(float(dq_w[n, k])))
            assert abs(Fraction(float(y[m, n])) - exact) <= Fraction(2.0 ** -50) * Fraction(float(aabs[m, n]))
            assert out[m, n] == bf16_rne_fraction(exact)
    assert np.all(aabs >= np.abs(y))


def test_gemm_one_hot_activation_reproduces_weight_column():
    N, K = 256, 384
    W = inputs.weights_bf16(N, K, seed=51)
    w, sw = oracle.weight_quant(inputs.bf16_bits(W))
    dq_w = torch_e4m3_decode(w)
    for k, c in ((0, 1.0), (200, -3.0), (383, 0.15625)):
        x = torch.zeros(1, K, dtype=torch.bfloat16)
        x[0, k] = c
        q, sa = oracle.act_quant(inputs.bf16_bits(x))
        assert q[0, k] == (0xFE if c < 0 else 0x7E)
        assert np.count_nonzero(q[0] & 0x7F) == 1
        y, _, _ = oracle.block_gemm(q, sa, w, sw)
        s = sa[0, k // G]
        for n in range(N):
            exact = (Fraction(float(s)) * Fraction(float(sw[n // G, k // G])) * 448
                     * Fraction(float(dq_w[n, k])) * (-1 if c < 0 else 1))
            assert abs(Fraction(float(y[0, n])) - exact) <= abs(exact) * Fraction(2.0 ** -52)


def test_gemm_scale_linearity():
    q, sa, w, sw = _quantised_problem(4, 300, 512, seed=61)
    y0, _, _ = oracle.block_gemm(q, sa, w, sw)
    for j in (-5, 4):
        ya, _, _ = oracle.block_gemm(q, (sa * np.float32(2.0 ** j)).astype(np.float32), w, sw)
        yw, _, _ = oracle.block_gemm(q, sa, w, (sw * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(ya, y0 * 2.0 ** j)
        assert np.array_equal(yw, y0 * 2.0 ** j)
    # one block's scale only moves that block's share of the sum
    sw2 = sw.copy()
    sw2[1, 2] *= 2
    y2, _, _ = oracle.block_gemm(q, sa, w, sw2)
    assert np.array_equal(y2[:, :128], y0[:, :128])
    assert not np.array_equal(y2[:, 128:256], y0[:, 128:256])


def test_gemm_k_permutation_inside_blocks():
    q, sa, w, sw = _quantised_problem(5, 160, 384, seed=71)
    y0, _, o0 = oracle.block_gemm(q, sa, w, sw)
    rng = np.random.default_rng(0)
    perm = np.concatenate([kb * G + rng.permutation(G) for kb in range(384 // G)])
    y1, _, o1 = oracle.block_gemm(q[:, perm], sa, w[:, perm], sw)
    assert np.array_equal(y0, y1) and np.array_equal(o0, o1)
    # permuting across blocks (different scales) must change the result
    cross = np.roll(np.arange(384), 64)
    y2, _, _ = oracle.block_gemm(q[:, cross], sa, w[:, cross], sw)
    assert not np.allclose(y0, y2)


def test_gemm_matches_float64_dequant_matmul():
    M, N, K = 8, 384, 512
    q, sa, w, sw = _quantised_problem(M, N, K, seed=81)
    y, _, _ = oracle.block_gemm(q, sa, w, sw)
    X = torch.from_numpy(torch_e4m3_decode(q)).double()
    Wd = torch.from_numpy(torch_e4m3_decode(w)).double()
    ref = torch.zeros(M, N, dtype=torch.float64)
    for kb in range(K // G):
        part = X[:, kb * G:(kb + 1) * G] @ Wd[:, kb * G:(kb + 1) * G].T
        col_scale = torch.from_numpy(sw[:, kb].astype(np.float64)).repeat_interleave(G)[:N]
        ref += part * torch.from_numpy(sa[:, kb].astype(np.float64))[:, None] * col_scale[None, :]
    assert torch.allclose(torch.from_numpy(y), ref, rtol=1e-12, atol=1e-12)


def test_gemm_row_subset_and_errors():
    q, sa, w, sw = _quantised_problem(6, 130, 256, seed=91)
    y, a, o = oracle.block_gemm(q, sa, w, sw)
    rows = np.array([5, 0, 3])
    ys, as_, os_ = oracle.block_gemm(q, sa, w, sw, rows=rows)
    assert np.array_equal(ys, y[rows]) and np.array_equal(os_, o[rows]) and np.array_equal(as_, a[rows])
    w_bad = w.copy()
    w_bad[3, 7] = 0x7F
    with pytest.raises(oracle.OracleError):
        oracle.block_gemm(q, sa, w_bad, sw)
    with pytest.raises(oracle.OracleError):
        oracle.block_gemm(q, sa, w, sw, rows=[6])


def test_projection_shapes_fixture():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "projection_shapes.txt")
    rows = [tuple(int(v) for v in line.split()) for line in open(path, encoding="utf-8")
            if line.strip() and not line.startswith("#")]
    assert tuple(rows) == inputs.SHAPES
    assert all(K % G == 0 and N % G == 0 for N, K in rows)


# ------------------------------------------------- weight-only GEMM (W8A16)
def _w8a16_problem(M, N, K, seed):
    x = inputs.activations_bf16(M, K, seed=seed)
    W = inputs.weights_bf16(N, K, seed=seed + 1)
    w, sw = oracle.weight_quant(inputs.bf16_bits(W))
    return x, w, sw


def test_w8a16_brute_force_fractions():
    """Exact rational y (bf16 x times torch-decoded weights) on a tiny problem
    with two scale blocks along N and K."""
    M, N, K = 2, 200, 256
    x, w, sw = _w8a16_problem(M, N, K, seed=141)
    y, aabs, out = oracle.block_gemm_w8a16(inputs.bf16_bits(x), w, sw)
    xf = x.float().numpy()          # bf16 -> fp32 is exact
    dq_w = torch_e4m3_decode(w)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            for kb in range(K // G):
                dot = sum(Fraction(float(xf[m, k])) * Fraction(float(dq_w[n, k])) for k in range(kb * G, (kb + 1) * G))
                exact += Fraction(float(sw[n // G, kb])) * dot
            assert abs(Fraction(float(y[m, n])) - exact) <= Fraction(2.0 ** -50) * Fraction(float(aabs[m, n]))
            assert out[m, n] == bf16_rne_fraction(exact)


def test_w8a16_reduces_to_w8a8_on_quantised_activations():
    """When x is itself dq(q) * sa with power-of-two sa (exact in bf16), the
    weight-only product equals the W8A8 block GEMM of (q, sa) exactly."""
    M, N, K = 3, 256, 384
    rng = np.random.default_rng(7)
    q = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3C                      # no NaN codes
    sa = (2.0 ** rng.integers(-6, 4, size=(M, K // G))).astype(np.float32)
    xf = torch_e4m3_decode(q).astype(np.float64) * np.repeat(sa.astype(np.float64), G, axis=1)
    x = torch.from_numpy(xf).to(torch.bfloat16)
    assert np.array_equal(x.double().numpy(), xf)     # the bf16 activations are exact
    W = inputs.weights_bf16(N, K, seed=143)
    w, sw = oracle.weight_quant(inputs.bf16_bits(W))
    y16, a16, o16 = oracle.block_gemm_w8a16(inputs.bf16_bits(x), w, sw)
    y8, a8, o8 = oracle.block_gemm(q, sa, w, sw)
    assert np.array_equal(y16, y8) and np.array_equal(a16, a8) and np.array_equal(o16, o8)


def test_w8a16_matches_float64_dequant_matmul_and_rows():
    M, N, K = 6, 300, 512
    x, w, sw = _w8a16_problem(M, N, K, seed=151)
    y, _, o = oracle.block_gemm_w8a16(inputs.bf16_bits(x), w, sw)
    X = x.double()
    Wd = torch.from_numpy(torch_e4m3_decode(w)).double()
    ref = torch.zeros(M, N, dtype=torch.float64)
    for kb in range(K // G):
        part = X[:, kb * G:(kb + 1) * G] @ Wd[:, kb * G:(kb + 1) * G].T
        ref += part * torch.from_numpy(sw[:, kb].astype(np.float64)).repeat_interleave(G)[:N][None, :]
    assert torch.allclose(torch.from_numpy(y), ref, rtol=1e-12, atol=1e-12)
    rows = np.array([4, 1])
    ys, _, os_ = oracle.block_gemm_w8a16(inputs.bf16_bits(x), w, sw, rows=rows)
    assert np.array_equal(ys, y[rows]) and np.array_equal(os_, o[rows])
    xb = inputs.bf16_bits(x).copy()
    xb[0, 3] = 0x7FC0                                  # a bf16 NaN
    with pytest.raises(oracle.OracleError):
        oracle.block_gemm_w8a16(xb, w, sw)
