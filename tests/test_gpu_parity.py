"""GPU parity: the CUDA path against the CPU oracle on the same seeded inputs.

Covers, through the C ABI (via the ctypes binding):
* activation and weight quantisation, bit-exact, on the five projection
  shapes, every M of the five workloads, edge-case groups and ragged N;
* the GEMM on the five shapes at M = 1, 2..8, 64, 102 (every output) and
  4096 (sampled rows), plus ragged shapes that cross tile and scale-block
  edges, empty problems, determinism, non-default streams, CUDA-graph
  capture and out-of-bounds write canaries.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_act_gb300 import inputs

pytestmark = pytest.mark.gpu

SHAPES = inputs.SHAPES
_problems: dict = {}


@pytest.fixture(scope="module")
def fp8act():
    from block_scaled_fp8_act_gb300 import fp8act as mod
    mod.load(build=True)
    return mod


def problem(si: int):
    from parity_util import Problem
    if si not in _problems:
        N, K = SHAPES[si]
        _problems[si] = Problem(N, K, inputs.weight_seed(si))
    return _problems[si]


# ------------------------------------------------------------ quantisation
@pytest.mark.parametrize("K", sorted({k for _, k in SHAPES}))
@pytest.mark.parametrize("M", [1, 5, 8, 64, 102])
def test_act_quant_bit_exact(fp8act, M, K):
    x = inputs.activations_bf16(M, K, seed=3000 + M)
    q_ref, sa_ref = oracle.act_quant(inputs.bf16_bits(x))
    q, sa = fp8act.fp8_act_quant(x.cuda())
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sa.cpu().numpy(), sa_ref)


@pytest.mark.parametrize("M,K", [(1, 9 * 128), (7, 5120), (33, 3072)])
def test_act_quant_edge_groups_bit_exact(fp8act, M, K):
    x = inputs.edge_activations_bf16(M, K, seed=M)
    q_ref, sa_ref = oracle.act_quant(inputs.bf16_bits(x))
    q, sa = fp8act.fp8_act_quant(x.cuda())
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sa.cpu().numpy(), sa_ref)


def test_act_quant_prefill_size_bit_exact(fp8act):
    x = inputs.activations_bf16(4096, 8704, seed=4096)
    q_ref, sa_ref = oracle.act_quant(inputs.bf16_bits(x))
    q, sa = fp8act.fp8_act_quant(x.cuda())
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sa.cpu().numpy(), sa_ref)


@pytest.mark.parametrize("si", range(len(SHAPES)))
def test_weight_quant_bit_exact_projection_shapes(fp8act, si):
    p = problem(si)
    assert np.array_equal(p.w.cpu().numpy(), p.w_ref)
    assert np.array_equal(p.sw.cpu().numpy(), p.sw_ref)


@pytest.mark.parametrize("N,K", [(200, 256), (1000, 384), (1, 128), (129, 1152)])
def test_weight_quant_bit_exact_ragged(fp8act, N, K):
    W = inputs.weights_bf16(N, K, seed=N)
    w_ref, sw_ref = oracle.weight_quant(inputs.bf16_bits(W))
    w, sw = fp8act.fp8_weight_quant(W.cuda())
    assert np.array_equal(w.cpu().numpy(), w_ref)
    assert np.array_equal(sw.cpu().numpy(), sw_ref)


# ------------------------------------------------------------------- GEMM
@pytest.mark.parametrize("si", range(len(SHAPES)))
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
def test_gemm_decode_and_verify_widths(fp8act, si, M):
    stats = problem(si).run_and_compare(M, inputs.activation_seed(si, M - 1))
    assert stats["max_ulp"] <= 1 or stats["floor_used"] > 0


@pytest.mark.parametrize("si", range(len(SHAPES)))
@pytest.mark.parametrize("M", [64, 102])
def test_gemm_batched_decode(fp8act, si, M):
    problem(si).run_and_compare(M, inputs.activation_seed(si, 8 + (M == 102)))


@pytest.mark.parametrize("si", range(len(SHAPES)))
def test_gemm_prefill_sampled_rows(fp8act, si):
    """M = 4096 on every projection shape, on every output column of about
    640 rows: the first and last 128, one random row in each 32-row lane
    quadrant of each of the 32 token tiles, and 256 random rows."""
    from parity_util import tile_rows
    rows = tile_rows(4096, 256, seed=si)
    assert len(rows) >= 256 + 2 * 128
    problem(si).run_and_compare(4096, inputs.activation_seed(si, 10), rows=rows)


@pytest.mark.parametrize("N,K", [(2600, 1024), (5000, 512)])
def test_gemm_prefill_ragged_n(fp8act, N, K):
    """M = 4096 with N past the last full 256-wide tile: the last tile's rows
    beyond N read as zero, its scale blocks end inside the tile, and nothing
    is stored past N. N = 5000 takes the split tail (a 136-column ragged tail
    of 128-wide tiles, K split over a cluster)."""
    from parity_util import Problem, tile_rows
    rows = tile_rows(4096, 256, seed=N)
    Problem(N, K, seed=N + K).run_and_compare(4096, seed=7, rows=rows)


@pytest.mark.parametrize("N", [2600, 5064])
def test_gemm_prefill_ragged_n_writes_nothing_outside_out(fp8act, N):
    """M = 4096 with a ragged N: 2600 goes through the persistent 256-wide
    store path alone (the last tile ends 40 rows past N); 5064 through the
    split tail (19 column groups of 256 in the persistent launch, the last
    200 columns as 128-wide tiles with K split over a cluster, writing a
    column slice of the output with the full row stride). Canaries on both
    sides of the output stay intact."""
    from parity_util import Problem
    p = Problem(N, 1024, seed=N + 1024)
    M = 4096
    q, sa, _, _ = p.activations(M, seed=5)
    pad = 1 << 16
    for dtype, call in ((torch.bfloat16, fp8act.fp8_block_gemm), (torch.float32, fp8act.fp8_block_gemm_f32)):
        buf = torch.full((M * p.N + 2 * pad,), -7.0, dtype=dtype, device="cuda")
        out = buf[pad:pad + M * p.N].view(M, p.N)
        call(q, sa, p.w, p.sw, out)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == -7.0) and torch.all(buf[pad + M * p.N:] == -7.0), dtype
        assert torch.all(torch.isfinite(out.float()))


# ------------------------------------------- batched decode (16 < M <= 128)
@pytest.mark.parametrize("M", [17, 24, 33, 48, 49, 80, 96, 113, 128])
@pytest.mark.parametrize("N,K", [(1000, 2048), (300, 640), (2176, 1152)])
def test_gemm_midm_widths_and_splits(fp8act, M, N, K):
    """Batched-decode widths on both sides of the kernel boundary (the
    weight-streaming tcgen05 kernel up to 48 tokens, its token tiles 32 and
    48 wide; the token-tiled kernel from 49) against N that ends inside a
    weight tile and K split over clusters of 2 .. 8 CTAs (N = 1000: 8 tiles,
    16 K groups; N = 300: 3 tiles, 5 K groups; N = 2176: 17 tiles, 9 K
    groups)."""
    from parity_util import Problem
    Problem(N, K, seed=N + K + 1).run_and_compare(M, seed=M + 11)


@pytest.mark.parametrize("M", [32, 102])
def test_gemm_midm_many_tiles_per_cta(fp8act, vocab_problem, M):
    """The vocabulary-sized head at batched-decode widths: 1187 weight tiles
    on at most one CTA per SM, so every CTA walks several tiles (the
    persistent path of both tile kernels: the accumulator ring runs on
    across tiles)."""
    vocab_problem.run_and_compare(M, seed=720 + M)


@pytest.mark.parametrize("M,N,K", [(1, 17, 128), (3, 200, 256), (8, 1000, 384), (9, 130, 512),
                                   (16, 4096, 1024), (63, 300, 640), (65, 257, 768),
                                   (127, 129, 256), (129, 520, 1152), (300, 384, 384)])
def test_gemm_ragged_shapes(fp8act, M, N, K):
    from parity_util import Problem
    p = Problem(N, K, seed=N + K)
    p.run_and_compare(M, seed=M + 7)


def test_gemm_edge_activations(fp8act):
    from parity_util import Problem
    p = Problem(640, 9 * 128, seed=5)
    for M in (1, 8, 20):
        p.run_and_compare(M, seed=M, edge=True)


def test_gemm_empty_problems(fp8act):
    q = torch.empty((0, 256), dtype=torch.uint8, device="cuda")
    sa = torch.empty((0, 2), dtype=torch.float32, device="cuda")
    w = torch.zeros((128, 256), dtype=torch.uint8, device="cuda")
    sw = torch.ones((1, 2), dtype=torch.float32, device="cuda")
    assert fp8act.fp8_block_gemm(q, sa, w, sw).shape == (0, 128)


def test_gemm_deterministic_and_stream_safe(fp8act):
    p = problem(1)
    q, sa, _, _ = p.activations(8, seed=1)
    a = fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        b = fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_quant_and_gemm_capture_in_cuda_graph(fp8act):
    p = problem(1)
    x = inputs.activations_bf16(4, p.K, seed=9).cuda()
    q = torch.empty((4, p.K), dtype=torch.uint8, device="cuda")
    sa = torch.empty((4, p.K // 128), dtype=torch.float32, device="cuda")
    out = torch.empty((4, p.N), dtype=torch.bfloat16, device="cuda")
    fp8act.fp8_act_quant(x, q, sa)
    fp8act.fp8_block_gemm(q, sa, p.w, p.sw, out)
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fp8act.fp8_act_quant(x, q, sa, stream=s)
            fp8act.fp8_block_gemm(q, sa, p.w, p.sw, out, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


@pytest.mark.parametrize("si", [0, 1, 2])
@pytest.mark.parametrize("M", [9, 12, 16])
def test_gemm_verify_widths_up_to_16(fp8act, si, M):
    problem(si).run_and_compare(M, inputs.activation_seed(si, 11 + M))


def test_gemm_writes_nothing_outside_out(fp8act):
    p = problem(1)
    for M in (1, 7, 13, 70):
        q, sa, _, _ = p.activations(M, seed=M)
        pad = 4096
        buf = torch.full((M * p.N + 2 * pad,), -7.0, dtype=torch.bfloat16, device="cuda")
        out = buf[pad:pad + M * p.N].view(M, p.N)
        fp8act.fp8_block_gemm(q, sa, p.w, p.sw, out)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == -7.0) and torch.all(buf[pad + M * p.N:] == -7.0)


def test_status_is_clean(fp8act):
    assert fp8act.check_status() == 0


# ------------------------------------------------------- weight-only (W8A16)
def _w8a16_compare(fp8act, p, M, seed, rows=None):
    from parity_util import compare_gemm
    x = inputs.activations_bf16(M, p.K, seed)
    xd = x.cuda()
    out = fp8act.fp8_block_gemm_w8a16(xd, p.w, p.sw)
    out32 = fp8act.fp8_block_gemm_w8a16_f32(xd, p.w, p.sw)
    torch.cuda.synchronize()
    y, aabs, ref = oracle.block_gemm_w8a16(inputs.bf16_bits(x), p.w_ref, p.sw_ref, rows=rows)
    if rows is not None:
        idx = torch.as_tensor(np.asarray(rows), device=out.device)
        out, out32 = out.index_select(0, idx), out32.index_select(0, idx)
    return compare_gemm(out, out32, y, aabs, ref, p.K)


@pytest.mark.parametrize("si", range(len(SHAPES)))
@pytest.mark.parametrize("M", [1, 2, 5, 8, 12, 16])
def test_w8a16_decode_widths(fp8act, si, M):
    _w8a16_compare(fp8act, problem(si), M, seed=500 + M)


@pytest.mark.parametrize("M,N,K", [(1, 17, 128), (5, 200, 256), (12, 1000, 384), (40, 257, 768)])
def test_w8a16_ragged(fp8act, M, N, K):
    from parity_util import Problem
    _w8a16_compare(fp8act, Problem(N, K, seed=N + 3 * K), M, seed=M)


def test_w8a16_edge_activations_and_determinism(fp8act):
    from parity_util import compare_gemm
    p = problem(1)
    x = inputs.edge_activations_bf16(7, p.K, seed=9)
    xd = x.cuda()
    a = fp8act.fp8_block_gemm_w8a16_f32(xd, p.w, p.sw)
    b = fp8act.fp8_block_gemm_w8a16_f32(xd, p.w, p.sw)
    out = fp8act.fp8_block_gemm_w8a16(xd, p.w, p.sw)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    y, aabs, ref = oracle.block_gemm_w8a16(inputs.bf16_bits(x), p.w_ref, p.sw_ref)
    compare_gemm(out, a, y, aabs, ref, p.K)


# ------------------------------------------------- vocabulary-sized head GEMV
@pytest.fixture(scope="module")
def vocab_problem(fp8act):
    from parity_util import Problem
    N, K = inputs.VOCAB_SHAPE
    p = Problem(N, K, inputs.weight_seed(inputs.VOCAB_SEED_INDEX))
    assert np.array_equal(p.w.cpu().numpy(), p.w_ref) and np.array_equal(p.sw.cpu().numpy(), p.sw_ref)
    return p


@pytest.mark.parametrize("M", [1, 8])
def test_vocab_head_gemv(fp8act, vocab_problem, M):
    """N = 151936 gives a grid of 9496 CTAs, far more than one wave: the
    multi-wave launch path of the weight-streaming kernel."""
    vocab_problem.run_and_compare(M, seed=700 + M)


def test_vocab_head_w8a16(fp8act, vocab_problem):
    _w8a16_compare(fp8act, vocab_problem, 1, seed=711)


@pytest.mark.parametrize("M", [1, 8])
def test_vocab_head_fused(fp8act, vocab_problem, M):
    """`fp8_linear` on the vocabulary head: 9496 tiles dealt over one CTA per
    SM, so every warp group walks several rounds of tiles (M = 8 also shares
    the quantisation over 4-CTA clusters). Oracle parity, and the fp32 result
    equals the two-launch path's bit for bit."""
    xd, out32 = _linear_compare(fp8act, vocab_problem, M, seed=720 + M)
    q, sa = fp8act.fp8_act_quant(xd)
    ref32 = fp8act.fp8_block_gemm_f32(q, sa, vocab_problem.w, vocab_problem.sw)
    torch.cuda.synchronize()
    assert torch.equal(out32, ref32)


# ------------------------------------------------------------ grouped calls
def test_act_quant_grouped_bit_exact(fp8act):
    """One launch over the five K's and ragged M's, bit-exact per problem."""
    specs = [(1, 5120), (8, 3072), (3, 8704), (16, 5120), (102, 5120), (0, 256), (5, 128)]
    xs = [inputs.activations_bf16(M, K, seed=40 + i) for i, (M, K) in enumerate(specs)]
    res = fp8act.fp8_act_quant_grouped([x.cuda() for x in xs])
    torch.cuda.synchronize()
    for x, (q, sa) in zip(xs, res):
        q_ref, sa_ref = oracle.act_quant(inputs.bf16_bits(x))
        assert np.array_equal(q.cpu().numpy(), q_ref)
        assert np.array_equal(sa.cpu().numpy(), sa_ref)


def _grouped_compare(fp8act, probs, ms, seed):
    from parity_util import compare_gemm
    acts = [p.activations(M, seed + i) for i, (p, M) in enumerate(zip(probs, ms))]
    args = [(q, sa, p.w, p.sw) for (q, sa, _, _), p in zip(acts, probs)]
    outs = fp8act.fp8_block_gemm_grouped(args)
    outs32 = fp8act.fp8_block_gemm_grouped_f32(args)
    torch.cuda.synchronize()
    for (q, sa, q_ref, sa_ref), p, o, o32 in zip(acts, probs, outs, outs32):
        assert np.array_equal(q.cpu().numpy(), q_ref) and np.array_equal(sa.cpu().numpy(), sa_ref)
        y, aabs, ref = oracle.block_gemm(q_ref, sa_ref, p.w_ref, p.sw_ref)
        compare_gemm(o, o32, y, aabs, ref, p.K)


@pytest.mark.parametrize("M", [1, 8])
def test_gemm_grouped_five_shapes(fp8act, M):
    _grouped_compare(fp8act, [problem(si) for si in range(len(SHAPES))], [M] * len(SHAPES), seed=800 + M)


def test_gemm_grouped_ragged_mix(fp8act):
    """Different M per problem (1..16, and 40 on the tile kernel), N that is
    not a multiple of 16 or 128, K from 1 to 9 groups."""
    from parity_util import Problem
    dims = [(17, 128, 1), (200, 256, 5), (1000, 384, 12), (257, 768, 16), (130, 1152, 3), (300, 512, 40)]
    probs = [Problem(N, K, seed=900 + i) for i, (N, K, _) in enumerate(dims)]
    _grouped_compare(fp8act, probs, [m for _, _, m in dims], seed=910)


@pytest.mark.parametrize("M", [32, 64, 102, 128])
def test_gemm_grouped_batched_five_shapes(fp8act, M):
    """Batched-decode widths over the five projections in one grouped call:
    their 336 weight tiles fill the SMs, so one persistent launch of the
    128 x 128 tile kernel takes them all (the tiles dealt over the CTAs in
    order of falling K, no split K); every output against the oracle."""
    _grouped_compare(fp8act, [problem(si) for si in range(len(SHAPES))], [M] * len(SHAPES), seed=820 + M)


def test_gemm_grouped_batched_ragged(fp8act):
    """The grouped tile launch with ragged problems: N ending inside a weight
    tile and inside a scale block, M from 17 to 128, K from 3 to 16 groups,
    201 tiles in all (past the SM count, so the grouped launch is taken),
    problems given out of K order."""
    from parity_util import Problem
    dims = [(300, 384, 50), (9000, 1024, 100), (1000, 2048, 128), (10000, 640, 17), (5000, 512, 77)]
    assert sum((N + 127) // 128 for N, _, _ in dims) >= 152
    probs = [Problem(N, K, seed=940 + i) for i, (N, K, _) in enumerate(dims)]
    _grouped_compare(fp8act, probs, [m for _, _, m in dims], seed=950)


def test_gemm_grouped_every_route_in_one_call(fp8act):
    """Twelve problems in one grouped call: one at M = 8 (the grouped
    weight-streaming launch), ten at 17 <= M <= 128 (the first eight, 192
    tiles, in one grouped tile launch; the last two, too few tiles to fill
    the SMs, one tile-kernel launch each) and one at M = 200 (its own
    launch); every output against the oracle."""
    from parity_util import Problem
    dims = [(500, 384, 8)] + [(3000, 256, m) for m in (17, 30, 45, 64, 80, 96, 113, 128, 20, 100)] + \
        [(700, 512, 200)]
    assert sum((N + 127) // 128 for N, _, m in dims[1:9]) >= 152
    probs = [Problem(N, K, seed=990 + i) for i, (N, K, _) in enumerate(dims)]
    _grouped_compare(fp8act, probs, [m for _, _, m in dims], seed=995)


def test_gemm_grouped_prefill_five_shapes(fp8act):
    """Prefill width (M = 4096) over the five projections in one grouped call:
    5376 tiles of 128 tokens x 256 weight rows in one persistent launch (the
    token tiles of a column group together, the tiles dealt over the CTAs in
    order of falling K). Every output column of about 640 rows per shape (the
    prefill test's rows: first and last 128, one per token tile and TMEM lane
    quadrant, 256 random) against the oracle; on the three shapes whose own
    call has no split tail, all outputs equal that call's bit for bit."""
    from parity_util import compare_gemm, oracle_gemm, tile_rows
    ps = [problem(si) for si in range(len(SHAPES))]
    acts = [p.activations(4096, 1300 + i) for i, p in enumerate(ps)]
    args = [(q, sa, p.w, p.sw) for (q, sa, _, _), p in zip(acts, ps)]
    outs = fp8act.fp8_block_gemm_grouped(args)
    outs32 = fp8act.fp8_block_gemm_grouped_f32(args)
    torch.cuda.synchronize()
    for si, ((q, sa, q_ref, sa_ref), p, o, o32) in enumerate(zip(acts, ps, outs, outs32)):
        rows = tile_rows(4096, 256, seed=1310 + si)
        y, aabs, ref = oracle_gemm(q_ref, sa_ref, p.w_ref, p.sw_ref, rows=rows)
        idx = torch.as_tensor(np.asarray(rows), device=o.device)
        compare_gemm(o.index_select(0, idx), o32.index_select(0, idx), y, aabs, ref, p.K)
        if p.N != 5120:  # (5120, K) runs a split tail of its own
            single = fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw)
            torch.cuda.synchronize()
            assert torch.equal(o32, single), (p.N, p.K)


def test_gemm_grouped_wide_ragged(fp8act):
    """The grouped 256-wide launch on ragged problems: M from 129 to 1000 (a
    last token tile of 1 .. 127 rows), N ending inside a 256-wide tile and a
    scale block, K from 2 to 8 groups, 323 tiles (past two waves, so the
    grouped launch is taken); every output against the oracle."""
    from parity_util import Problem
    dims = [(5000, 512, 1000), (3000, 640, 300), (9000, 256, 129), (2600, 1024, 600)]
    assert sum(((m + 127) // 128) * ((N + 255) // 256) for N, _, m in dims) >= 304
    probs = [Problem(N, K, seed=1400 + i) for i, (N, K, _) in enumerate(dims)]
    _grouped_compare(fp8act, probs, [m for _, _, m in dims], seed=1410)


def test_gemm_grouped_batched_equals_single_call_without_split(fp8act):
    """(17408, 5120) alone runs 136 unsplit tiles, one K order per tile; in a
    grouped launch with the other projections each of its tiles runs the
    same K order on some CTA, so the fp32 results are equal bit for bit."""
    ps = [problem(si) for si in range(len(SHAPES))]
    acts = [p.activations(102, 970 + i) for i, p in enumerate(ps)]
    outs32 = fp8act.fp8_block_gemm_grouped_f32([(q, sa, p.w, p.sw) for (q, sa, _, _), p in zip(acts, ps)])
    q, sa, _, _ = acts[0]
    single = fp8act.fp8_block_gemm_f32(q, sa, ps[0].w, ps[0].sw)
    torch.cuda.synchronize()
    assert ps[0].N == 17408 and torch.equal(outs32[0], single)


# ------------------------------------------- fused act-quant + GEMM (fp8_linear)
def _linear_compare(fp8act, p, M, seed, edge=False):
    from parity_util import compare_gemm
    x = inputs.edge_activations_bf16(M, p.K, seed) if edge else inputs.activations_bf16(M, p.K, seed)
    xd = x.cuda()
    out = fp8act.fp8_linear(xd, p.w, p.sw)
    out32 = fp8act.fp8_linear_f32(xd, p.w, p.sw)
    torch.cuda.synchronize()
    q_ref, sa_ref = oracle.act_quant(inputs.bf16_bits(x))
    y, aabs, ref = oracle.block_gemm(q_ref, sa_ref, p.w_ref, p.sw_ref)
    compare_gemm(out, out32, y, aabs, ref, p.K)
    return xd, out32


@pytest.mark.parametrize("si", range(len(SHAPES)))
@pytest.mark.parametrize("M", [1, 3, 8, 12, 16])
def test_linear_fused_decode_widths(fp8act, si, M):
    _linear_compare(fp8act, problem(si), M, seed=600 + M)


@pytest.mark.parametrize("si", range(len(SHAPES)))
@pytest.mark.parametrize("M", [1, 2, 5, 8, 12, 16])
def test_linear_fused_equals_two_launches(fp8act, si, M):
    """For M <= 16 the fused kernel runs the two-launch path's warp count per
    tile and its loop, so equal codes and scales give the same fp32 sums bit
    for bit: any code or scale the in-kernel quantisation got wrong would
    show here. M = 1 quantises per SM; M = 2, 5, 8 on these shapes share the
    quantisation over clusters of 2 or 4 CTAs (each CTA writes its share into
    every peer's shared memory); M = 12, 16 add a second 8-token group per
    weight tile."""
    p = problem(si)
    xd, out32 = _linear_compare(fp8act, p, M, seed=650 + 10 * M + si)
    q, sa = fp8act.fp8_act_quant(xd)
    ref32 = fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw)
    torch.cuda.synchronize()
    assert torch.equal(out32, ref32)


@pytest.mark.parametrize("M,N,K", [(1, 17, 128), (5, 200, 256), (12, 1000, 384), (2, 257, 9 * 128)])
def test_linear_fused_ragged(fp8act, M, N, K):
    from parity_util import Problem
    _linear_compare(fp8act, Problem(N, K, seed=N + 5 * K), M, seed=M)


def test_linear_fused_edge_groups(fp8act):
    """Edge-case groups (zeros, -0, single values, 2^-126, bf16 subnormals,
    outliers, E4M3 midpoints, constants). K = 9 groups so that every row
    holds one group of each kind, as in the W8A8 edge test; at M = 1 the
    fused result must equal the two-launch one bit for bit."""
    from parity_util import Problem
    p = Problem(640, 9 * 128, seed=5)
    for M in (1, 8, 13):
        xd, out32 = _linear_compare(fp8act, p, M, seed=M, edge=True)
        if M == 1:
            q, sa = fp8act.fp8_act_quant(xd)
            ref32 = fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw)
            torch.cuda.synchronize()
            assert torch.equal(out32, ref32)


# ------------------------------- the newer entry points: graphs, streams, canaries
def test_new_paths_capture_in_cuda_graph_and_match_eager(fp8act):
    """W8A16, fused and grouped calls captured in one CUDA graph on a
    non-default stream give the same bits as the eager calls."""
    ps = [problem(si) for si in range(len(SHAPES))]
    xs = [inputs.activations_bf16(3, p.K, seed=960 + i).cuda() for i, p in enumerate(ps)]
    eager16 = [fp8act.fp8_block_gemm_w8a16(x, p.w, p.sw) for x, p in zip(xs, ps)]
    eagerf = [fp8act.fp8_linear(x, p.w, p.sw) for x, p in zip(xs, ps)]
    qsa = fp8act.fp8_act_quant_grouped(xs)
    eagerg = fp8act.fp8_block_gemm_grouped([(q, sa, p.w, p.sw) for (q, sa), p in zip(qsa, ps)])
    torch.cuda.synchronize()
    o16 = [torch.empty_like(t) for t in eager16]
    of = [torch.empty_like(t) for t in eagerf]
    og = [torch.empty_like(t) for t in eagerg]
    qsa2 = [(torch.empty_like(q), torch.empty_like(sa)) for q, sa in qsa]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for x, p, o in zip(xs, ps, o16):
                fp8act.fp8_block_gemm_w8a16(x, p.w, p.sw, out=o, stream=s)
            for x, p, o in zip(xs, ps, of):
                fp8act.fp8_linear(x, p.w, p.sw, out=o, stream=s)
            fp8act.fp8_act_quant_grouped(xs, outs=qsa2, stream=s)
            fp8act.fp8_block_gemm_grouped([(q, sa, p.w, p.sw) for (q, sa), p in zip(qsa2, ps)], outs=og, stream=s)
    g.replay()
    torch.cuda.synchronize()
    names = [f"{call} {si}" for call in ("w8a16", "fused", "grouped") for si in range(len(ps))]
    for name, a, b in zip(names, eager16 + eagerf + eagerg, o16 + of + og):
        assert torch.equal(a, b), (name, (a.float() - b.float()).abs().max().item())


def test_new_paths_write_nothing_outside_out(fp8act):
    p = problem(1)
    pad = 4096
    for M in (1, 7, 13):
        x = inputs.activations_bf16(M, p.K, seed=M).cuda()
        q, sa = fp8act.fp8_act_quant(x)
        for call in ("w8a16", "fused", "grouped"):
            buf = torch.full((M * p.N + 2 * pad,), -7.0, dtype=torch.bfloat16, device="cuda")
            out = buf[pad:pad + M * p.N].view(M, p.N)
            if call == "w8a16":
                fp8act.fp8_block_gemm_w8a16(x, p.w, p.sw, out=out)
            elif call == "fused":
                fp8act.fp8_linear(x, p.w, p.sw, out=out)
            else:
                fp8act.fp8_block_gemm_grouped([(q, sa, p.w, p.sw)], outs=[out])
            torch.cuda.synchronize()
            assert torch.all(buf[:pad] == -7.0) and torch.all(buf[pad + M * p.N:] == -7.0), (call, M)


def test_fused_at_its_shared_memory_limit(fp8act):
    """M = 8 and K = 24576: 8 rows of codes and scales take 198 KiB of the
    fused kernel's 200 KiB; one more K group is refused on the host."""
    from parity_util import Problem
    p = Problem(256, 24576, seed=17)
    _linear_compare(fp8act, p, 8, seed=18)
    x = torch.zeros((8, 24576 + 1024), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((256, 24576 + 1024), dtype=torch.uint8, device="cuda")
    sw = torch.ones((2, (24576 + 1024) // 128), dtype=torch.float32, device="cuda")
    with pytest.raises(fp8act.Fp8ActError):
        fp8act.fp8_linear(x, w, sw)


# ------------------------------------------- more shapes and call patterns
EXTRA_SHAPES = [(3, 1000, 10240), (1, 17, 65536), (8, 2056, 5120), (5, 130, 30720)]


@pytest.mark.parametrize("M,N,K", EXTRA_SHAPES)
def test_gemm_long_k_and_ragged_n(fp8act, M, N, K):
    """Few 16-row tiles against long K (N = 17, K = 65536: two tiles of 512
    K blocks each), N not a multiple of 16 or 128; the W8A16 and fused calls
    on the same shapes, and the fused result equal bit for bit to the
    two-launch one."""
    from parity_util import Problem
    p = Problem(N, K, seed=N + K)
    p.run_and_compare(M, seed=M + 3)
    _w8a16_compare(fp8act, p, M, seed=M + 4)
    xd, out32 = _linear_compare(fp8act, p, M, seed=M + 5)
    q, sa = fp8act.fp8_act_quant(xd)
    ref32 = fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw)
    torch.cuda.synchronize()
    assert torch.equal(out32, ref32)


def test_gemm_repeated_and_interleaved_calls(fp8act):
    """The five shapes called in turn, three times over in alternating order
    on one stream (back-to-back launches that overlap through programmatic
    dependent launch), give the same bits every time."""
    ps = [problem(si) for si in range(len(SHAPES))]
    acts = [p.activations(1 + 2 * si, seed=70 + si)[:2] for si, p in enumerate(ps)]
    first = [fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw) for (q, sa), p in zip(acts, ps)]
    later = []
    for r in range(3):
        order = list(range(len(ps)))[::(-1 if r % 2 else 1)]
        res = {i: fp8act.fp8_block_gemm_f32(acts[i][0], acts[i][1], ps[i].w, ps[i].sw) for i in order}
        later.append([res[i] for i in range(len(ps))])
    torch.cuda.synchronize()
    for res in later:
        for a, b in zip(first, res):
            assert torch.equal(a, b)


def test_gemm_concurrent_streams(fp8act):
    """Two streams issuing GEMMs at the same time: every result equals the
    serial one."""
    p0, p2 = problem(0), problem(2)
    q0, sa0 = p0.activations(2, seed=81)[:2]
    q2, sa2 = p2.activations(6, seed=82)[:2]
    r0 = fp8act.fp8_block_gemm_f32(q0, sa0, p0.w, p0.sw)
    r2 = fp8act.fp8_block_gemm_f32(q2, sa2, p2.w, p2.sw)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    o0 = [torch.empty_like(r0) for _ in range(16)]
    o2 = [torch.empty_like(r2) for _ in range(16)]
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    for a, b in zip(o0, o2):
        fp8act.fp8_block_gemm_f32(q0, sa0, p0.w, p0.sw, a, stream=s1)
        fp8act.fp8_block_gemm_f32(q2, sa2, p2.w, p2.sw, b, stream=s2)
    torch.cuda.synchronize()
    assert all(torch.equal(a, r0) for a in o0) and all(torch.equal(b, r2) for b in o2)


def test_first_calls_on_a_stream_inside_capture(fp8act):
    """A stream whose first GEMM and fused calls are inside a graph capture:
    replays match the eager results, and so do eager calls on that stream
    afterwards."""
    p = problem(2)
    q, sa = p.activations(4, seed=91)[:2]
    x = inputs.activations_bf16(4, p.K, seed=92).cuda()
    ref = fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw)
    ref_f = fp8act.fp8_linear_f32(x, p.w, p.sw)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    out = torch.empty_like(ref)
    out_f = torch.empty_like(ref_f)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw, out, stream=s)
            fp8act.fp8_linear_f32(x, p.w, p.sw, out_f, stream=s)
    for _ in range(3):
        out.zero_()
        out_f.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref) and torch.equal(out_f, ref_f)
    with torch.cuda.stream(s):
        e = fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw, stream=s)
    torch.cuda.synchronize()
    assert torch.equal(e, ref)


@pytest.mark.parametrize("si", [1, 0])
def test_gemm_with_only_16_byte_aligned_operands(fp8act, si):
    """Codes and weights that start 16 bytes past a 32-byte boundary (the API
    asks for 16) take the 16-byte-load kernels; the result must still match."""
    from parity_util import compare_gemm
    p = problem(si)
    M = 3
    q, sa, q_ref, sa_ref = p.activations(M, seed=77)
    qb = torch.empty(M * p.K + 16, dtype=torch.uint8, device="cuda")[16:].view(M, p.K)
    qb.copy_(q)
    wb = torch.empty(p.N * p.K + 16, dtype=torch.uint8, device="cuda")[16:].view(p.N, p.K)
    wb.copy_(p.w)
    assert qb.data_ptr() % 32 == 16 and wb.data_ptr() % 32 == 16
    out = fp8act.fp8_block_gemm(qb, sa, wb, p.sw)
    out32 = fp8act.fp8_block_gemm_f32(qb, sa, wb, p.sw)
    torch.cuda.synchronize()
    y, aabs, ref = oracle.block_gemm(q_ref, sa_ref, p.w_ref, p.sw_ref)
    compare_gemm(out, out32, y, aabs, ref, p.K)


def test_act_quant_bit_exact_over_many_scales(fp8act):
    """17.8M activations whose 1x128 groups are scaled by random factors
    2^-30 .. 2^30 (so the group scales, their reciprocals and the quotients
    cover many binades, and some quotients fall within a few fp32 ulps of an
    E4M3 rounding boundary): codes and scales bit-exact."""
    M, K = 2048, 8704
    rng = np.random.default_rng(123)
    x = rng.standard_normal((M, K), dtype=np.float32)
    x *= (2.0 ** rng.uniform(-30, 30, size=(M, K // 128))).astype(np.float32).repeat(128, axis=1)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    q, sa = fp8act.fp8_act_quant(xb.cuda())
    torch.cuda.synchronize()
    q_ref, sa_ref = oracle.act_quant(inputs.bf16_bits(xb))
    assert np.array_equal(sa.cpu().numpy(), sa_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


def _division_domain_groups(ab_lo: int, ab_hi: int) -> np.ndarray:
    """bf16 bit patterns [groups, 128]: for every positive amax pattern ab in
    [ab_lo, ab_hi], groups whose element 0 is amax and whose other 127
    elements run through every bf16 x with |x| <= amax, both signs (zero
    padded), so each group's amax is exactly ab."""
    blocks = []
    for ab in range(ab_lo, ab_hi + 1):
        mags = np.arange(ab + 1, dtype=np.uint16)
        xs = np.concatenate([mags, mags | np.uint16(0x8000)])
        g = -(-xs.size // 127)
        flat = np.zeros(g * 127, np.uint16)
        flat[:xs.size] = xs
        block = np.empty((g, 128), np.uint16)
        block[:, 0] = ab
        block[:, 1:] = flat.reshape(g, 127)
        blocks.append(block)
    return np.concatenate(blocks)


def test_act_quant_bit_exact_over_whole_quotient_domain(fp8act):
    """Every pair (group amax, element x) of bf16 values with |x| <= amax for
    amax from just below 2^-70 to just above 2^70 (~590M values, the range
    where the kernel forms x / s from the reciprocal of s plus one residual
    correction, and a few patterns on each side where it divides): codes and
    scales equal the oracle's IEEE-division quantisation."""
    lo, hi = 0x1C70, 0x6290  # bf16 patterns of 2^-70 - 16 ulps .. 2^70 + 16 ulps
    step = 1024
    for a0 in range(lo, hi + 1, step):
        bits = _division_domain_groups(a0, min(a0 + step - 1, hi))
        xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
        q, sa = fp8act.fp8_act_quant(xb.cuda())
        torch.cuda.synchronize()
        q_ref, sa_ref = oracle.act_quant(bits)
        assert np.array_equal(sa.cpu().numpy(), sa_ref), hex(a0)
        bad = np.nonzero(q.cpu().numpy() != q_ref)
        assert bad[0].size == 0, (hex(a0), bits[bad[0][0]].tolist()[:4], bad[1][:4])


def test_stream_read_folds_every_word(fp8act):
    """The weight-stream floor diagnostic reads every 32-bit word of the
    buffer exactly once: the folded result is the XOR of all of them."""
    g = torch.Generator(device="cpu").manual_seed(5)
    src = torch.randint(0, 256, (3 * 1024 * 1024 + 48,), dtype=torch.uint8, generator=g)
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8act.stream_read(src.cuda(), sink)
    torch.cuda.synchronize()
    want = np.bitwise_xor.reduce(src.numpy().view(np.uint32))
    assert int(sink.cpu().numpy().view(np.uint32)[0]) == int(want)
