"""Benchmark of the W8A8 block-FP8 linear layer on GB300.

Workload (one "step"): a decode pass at M = 1 over the five dense-27B
projection shapes (N, K) = (17408, 5120), (5120, 3072), (5120, 8704),
(7168, 5120), (8192, 5120): for each shape, fp8_act_quant of the token's
bf16 activations and fp8_block_gemm against that shape's E4M3 weights.
Inputs are seeded synthetic tensors (weights N(0, 0.02), activations N(0, 1)
with 0.1% x20 outliers), quantised by the library's own kernels before the
timed region. The weights are kept in three rotating copies (684 MB in
total, over 5x the 129 MB L2), so every step reads its weights from HBM.

Printed JSON line (rank 0):
  value      achieved HBM GB/s of the whole step (algorithmic bytes / time),
             steps replayed as CUDA graphs, inputs resident in HBM
  e2e        the same through the public API with the activations copied in
             from pinned host memory and the outputs copied back every step
             (calls captured once and replayed as a CUDA graph; the eagerly
             issued figure is reported beside it)
  roofline   the block GEMM kernel against the measured HBM copy bandwidth
  cpu_baseline  the CPU oracle on the same workload (host cores)
  sweep      us/call per shape at M = 1..8 (the no-cliff check), 64, 102
             and 4096 (the last as TFLOP/s of FP8 tensor peak)

`--workload verify|batched|prefill` times the same step at M = 8, 102 or
4096; `--workload decode-w8a16` times the weight-only variant at M = 1 (bf16
activations straight into the GEMM, no quantisation launch); `--workload
lmhead` times one vocabulary-sized head (N = 151936, K = 5120) at M = 1.
`--workload decode-fused` runs one fused fp8_linear launch per shape (the
activation quantisation inside the GEMM kernel).
`--workload decode-grouped` runs the five projections as independent problems
of one grouped act-quant launch and one grouped GEMM launch; `--workload
batched-grouped` and `--workload prefill-grouped` do the same at M = 102 and
4096 (the grouped tile kernel).
`--impl reference` times the CPU oracle instead (the reference arm).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_scaled_fp8_act_gb300 import inputs  # noqa: E402

G = 128
METRIC = "us/call and achieved HBM GB/s (% of roofline) for block-FP8 GEMM at M=1-8"
WORKLOADS = {
    # name: (M, description, roofline bound)
    "decode": (1, "decode M=1 over the five dense-27B projection shapes (act quant + block-FP8 GEMM per shape)",
               "hbm"),
    "verify": (8, "speculative verify M={M} (draft k={k}) over the five dense-27B projection shapes "
                  "(act quant + block-FP8 GEMM per shape)", "hbm"),
    "batched": (102, "batched decode M={M} over the five dense-27B projection shapes "
                     "(act quant + block-FP8 GEMM per shape)", "hbm"),
    "prefill": (4096, "prefill chunk M={M} over the five dense-27B projection shapes "
                      "(act quant + block-FP8 GEMM per shape)", "tensor"),
    "decode-w8a16": (1, "weight-only decode M={M} over the five dense-27B projection shapes "
                        "(bf16 activations x block-FP8 weights, one GEMM per shape, no act quant)", "hbm"),
    "lmhead": (1, "vocabulary-sized head M={M}: N=151936, K=5120 (act quant + block-FP8 GEMM)", "hbm"),
    "decode-fused": (1, "fused decode M={M} over the five dense-27B projection shapes "
                        "(one fp8_linear launch per shape: act quant inside the block-FP8 GEMM)", "hbm"),
    "decode-grouped": (1, "grouped decode M={M}: the five dense-27B projection shapes as independent problems, "
                          "one grouped act-quant launch + one grouped block-FP8 GEMM launch", "hbm"),
    "batched-grouped": (102, "grouped batched decode M={M}: the five dense-27B projection shapes as independent "
                             "problems, one grouped act-quant launch + one grouped block-FP8 GEMM launch", "hbm"),
    "prefill-grouped": (4096, "grouped prefill chunk M={M}: the five dense-27B projection shapes as independent "
                              "problems, one grouped act-quant launch + one grouped block-FP8 GEMM launch", "tensor"),
}
GROUPED = {"decode-grouped", "batched-grouped", "prefill-grouped"}
# Workloads on other shapes than the five projections: (shapes, weight seed indices).
WORKLOAD_SHAPES = {"lmhead": ((inputs.VOCAB_SHAPE,), (inputs.VOCAB_SEED_INDEX,))}
WEIGHT_ONLY = {"decode-w8a16"}
FUSED = {"decode-fused"}


def gemm_kernel_name(M: int) -> str:
    return "gemm_skinny_kernel" if M <= 16 else ("gemm_midm_kernel" if M <= 48 else "gemm_tc_kernel")
WEIGHT_COPIES = 3
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense FP8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)
NOMINAL_HBM_GBS = 7900.0     # GB300 HBM3e, nominal
NOMINAL_FP8_TFLOPS = 4500.0  # GB300 dense FP8, nominal


# ------------------------------------------------------------------ helpers
def algorithmic_gemm_bytes(M: int, N: int, K: int) -> int:
    """Bytes the block GEMM must move: weights + their scales, codes +
    scales of the activations, and the bf16 output."""
    KB, NB = K // G, (N + G - 1) // G
    return N * K + 4 * NB * KB + M * K + 4 * M * KB + 2 * M * N


def algorithmic_w8a16_bytes(M: int, N: int, K: int) -> int:
    """Weight-only GEMM: weights + scales, bf16 activations, bf16 output."""
    KB, NB = K // G, (N + G - 1) // G
    return N * K + 4 * NB * KB + 2 * M * K + 2 * M * N


def algorithmic_quant_bytes(M: int, K: int) -> int:
    """bf16 in, E4M3 codes and fp32 scales out."""
    return 2 * M * K + M * K + 4 * M * (K // G)


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {
    "gemm_skinny_kernel": ("gemm_skinny.cu", "act_group.cuh", "common.cuh", "sm100_ptx.cuh"),
    "gemm_skinny_grouped_kernel": ("gemm_skinny.cu", "act_group.cuh", "common.cuh", "sm100_ptx.cuh"),
    "linear_persistent_kernel": ("gemm_skinny.cu", "act_group.cuh", "common.cuh", "sm100_ptx.cuh"),
    "gemm_tc_kernel": ("gemm_tc.cu", "common.cuh", "sm100_ptx.cuh", "tc_ptx.cuh"),
    "gemm_tc_grouped_kernel": ("gemm_tc.cu", "common.cuh", "sm100_ptx.cuh", "tc_ptx.cuh"),
    "gemm_midm_kernel": ("gemm_midm.cu", "common.cuh", "sm100_ptx.cuh", "tc_ptx.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    """Short hash of a kernel's CUDA sources, to tell whether recorded ncu traffic is current."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_scaled_fp8_act_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str) -> float | None:
    """DRAM bytes per launch recorded from an ncu capture for the current
    sources (profiles/ncu_traffic.txt: `kernel workload source_hash bytes`)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(kernel)
    for line in open(path, encoding="utf-8"):
        parts = line.split()
        if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload \
                and parts[2] == want:
            return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during a timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- workload
class Weights:
    """E4M3 weights + scales of the five shapes in `copies` rotating copies
    (quantised on the device by fp8_weight_quant)."""

    def __init__(self, device: torch.device, copies: int = WEIGHT_COPIES, shapes=inputs.SHAPES, seed_index=None):
        from block_scaled_fp8_act_gb300 import fp8act
        self.shapes = list(shapes)
        self.copies = copies
        self.seed_index = list(seed_index) if seed_index is not None else list(range(len(self.shapes)))
        self.w, self.sw = [], []
        for si, (N, K) in enumerate(self.shapes):
            W = inputs.weights_bf16(N, K, inputs.weight_seed(self.seed_index[si])).to(device)
            w0, sw0 = fp8act.fp8_weight_quant(W)
            del W
            self.w.append([w0] + [w0.clone() for _ in range(copies - 1)])
            self.sw.append([sw0] + [sw0.clone() for _ in range(copies - 1)])
        torch.cuda.synchronize()


class Workload:
    """Device-resident activations of one M over the five shapes (plus pinned
    host copies for the end-to-end leg), sharing one Weights set."""

    def __init__(self, M: int, weights: Weights, device: torch.device, weight_only: bool = False,
                 grouped: bool = False, fused: bool = False):
        self.M = M
        self.weight_only = weight_only
        self.grouped = grouped
        self.fused = fused
        self.bf16_in = weight_only or fused  # the GEMM reads the bf16 activations itself
        self.shapes = weights.shapes
        self.copies = weights.copies
        self.w, self.sw = weights.w, weights.sw
        # The activations of all shapes live in one device buffer (and one pinned
        # host buffer), the outputs in another, so that the end-to-end leg moves
        # each direction with a single copy. Every slice starts on a 256-byte
        # boundary (M * K * 2 and M * N * 2 are multiples of 256).
        self.x_all = torch.empty(sum(M * K for _, K in self.shapes), dtype=torch.bfloat16, device=device)
        self.out_all = torch.empty(sum(M * N for N, _ in self.shapes), dtype=torch.bfloat16, device=device)
        self.x_host_all = torch.empty(self.x_all.numel(), dtype=torch.bfloat16).pin_memory()
        self.out_host_all = torch.empty(self.out_all.numel(), dtype=torch.bfloat16).pin_memory()
        self.x, self.q, self.sa, self.out = [], [], [], []
        xo = oo = 0
        for si, (N, K) in enumerate(self.shapes):
            x = inputs.activations_bf16(M, K, inputs.activation_seed(si, 0))
            self.x_host_all[xo:xo + M * K].copy_(x.reshape(-1))
            self.x.append(self.x_all[xo:xo + M * K].view(M, K))
            self.q.append(torch.empty((M, K), dtype=torch.uint8, device=device))
            self.sa.append(torch.empty((M, K // G), dtype=torch.float32, device=device))
            self.out.append(self.out_all[oo:oo + M * N].view(M, N))
            xo += M * K
            oo += M * N
        self.x_all.copy_(self.x_host_all)
        torch.cuda.synchronize()

    def gemm_bytes_of(self, N: int, K: int) -> int:
        return (algorithmic_w8a16_bytes if self.bf16_in else algorithmic_gemm_bytes)(self.M, N, K)

    def step_bytes(self) -> int:
        return sum(self.gemm_bytes_of(N, K) + (0 if self.bf16_in else algorithmic_quant_bytes(self.M, K))
                   for N, K in self.shapes)

    def launches_per_step(self) -> int:
        if self.grouped:
            return 2
        return (1 if self.bf16_in else 2) * len(self.shapes)

    def gemm_units(self) -> list:
        """The GEMM launches of one step: (label, algorithmic bytes, flops, enqueue(copy, stream))."""
        if self.grouped:
            return [("all five, grouped", sum(self.gemm_bytes_of(N, K) for N, K in self.shapes),
                     sum(2.0 * self.M * N * K for N, K in self.shapes), self.gemm_grouped)]
        return [((N, K), self.gemm_bytes_of(N, K), 2.0 * self.M * N * K,
                 lambda c, s, si=si: self.gemm(si, c, s)) for si, (N, K) in enumerate(self.shapes)]

    def gemm_grouped(self, copy: int, stream) -> None:
        from block_scaled_fp8_act_gb300 import fp8act
        fp8act.fp8_block_gemm_grouped([(self.q[si], self.sa[si], self.w[si][copy], self.sw[si][copy])
                                       for si in range(len(self.shapes))], outs=self.out, stream=stream)

    def gemm(self, si: int, copy: int, stream) -> None:
        from block_scaled_fp8_act_gb300 import fp8act
        if self.weight_only:
            fp8act.fp8_block_gemm_w8a16(self.x[si], self.w[si][copy], self.sw[si][copy], self.out[si],
                                        stream=stream)
        elif self.fused:
            fp8act.fp8_linear(self.x[si], self.w[si][copy], self.sw[si][copy], self.out[si], stream=stream)
        else:
            fp8act.fp8_block_gemm(self.q[si], self.sa[si], self.w[si][copy], self.sw[si][copy],
                                  self.out[si], stream=stream)

    def enqueue_step(self, copy: int, stream) -> None:
        from block_scaled_fp8_act_gb300 import fp8act
        if self.grouped:
            fp8act.fp8_act_quant_grouped(self.x, outs=list(zip(self.q, self.sa)), stream=stream)
            self.gemm_grouped(copy, stream)
            return
        for si in range(len(self.shapes)):
            if not self.bf16_in:
                fp8act.fp8_act_quant(self.x[si], self.q[si], self.sa[si], stream=stream)
            self.gemm(si, copy, stream)


def _label(lb) -> dict:
    return {"N": lb[0], "K": lb[1]} if isinstance(lb, tuple) else {"launch": lb}


def capture(fn, stream) -> torch.cuda.CUDAGraph:
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm the code path once outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    return g


def graph_schedule(n: int, steps_per_graph: int, copies: int) -> list[tuple[str, int]]:
    """Replays that run exactly n steps: ("multi", j) replays S-step graph j (its
    steps use weight copies (j S + s) mod copies), then ("single", c) replays
    the one-step graph of copy c for the remainder. Step i always uses weight
    copy i mod copies."""
    S = steps_per_graph
    out = [("multi", j % copies) for j in range(n // S)] if S > 1 else []
    done = n // S * S if S > 1 else 0
    out += [("single", i % copies) for i in range(done, n)]
    return out


def time_graphs(graphs, steps: int, warmup: int, stream) -> float:
    """Seconds per replay, replaying graphs round-robin, CUDA events on `stream`."""
    for i in range(warmup):
        graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(steps):
            graphs[i % len(graphs)].replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3 / steps


def chain_times(fns, stream, launches: int, reps: int) -> list[tuple[float, float, float]]:
    """Per function: (median, p10, p90) seconds per call over `reps` replays of
    a CUDA graph of `launches` back-to-back calls fn(i) (i = call index),
    timed with events on the launching stream."""
    out = []
    for fn in fns:
        def chain(fn=fn):
            for i in range(launches):
                fn(i)
        g = capture(chain, stream)
        ts = [time_graphs([g], 1, 1, stream) / launches for _ in range(reps)]
        out.append((statistics.median(ts), float(np.percentile(ts, 10)), float(np.percentile(ts, 90))))
        del g
    return out


def gemm_kernel_times(wl: Workload, stream, launches: int = 60, reps: int = 7, spread=None) -> list[float]:
    """Average duration (s) of each GEMM launch of a step (one per shape, or
    one grouped launch) over the rotating weight copies: the median of `reps`
    replays (p10 / p90 appended to `spread` when given)."""
    res = chain_times([lambda i, fn=u[3]: fn(i % wl.copies, stream) for u in wl.gemm_units()], stream, launches,
                      reps)
    if spread is not None:
        spread.extend((lo, hi) for _, lo, hi in res)
    return [med for med, _, _ in res]


def floor_times(wl: Workload, stream, launches: int = 60, reps: int = 7) -> list[float]:
    """The streaming-read floor of each shape's weight stream: a chain of plain
    reads of the same (rotating) weight copies, launched like the GEMMs."""
    from block_scaled_fp8_act_gb300 import fp8act
    sink = torch.zeros(1, dtype=torch.int32, device=wl.out_all.device)
    res = chain_times([lambda i, si=si: fp8act.stream_read(wl.w[si][i % wl.copies], sink, stream=stream)
                       for si in range(len(wl.shapes))], stream, launches, reps)
    return [med for med, _, _ in res]


def quant_kernel_times(wl: Workload, stream, launches: int = 60, reps: int = 7) -> list[tuple[float, float, float, int]]:
    """The activation-quantisation launch of each shape, timed like the GEMMs.
    Where one call's tensors exceed 1 MB, the chain rotates over copies of
    its input and outputs that together hold more than twice the L2, so each
    call reads its input from HBM (at decode sizes the activations are L2
    resident in a real step too). Per shape: (median, p10, p90, copies)."""
    from block_scaled_fp8_act_gb300 import fp8act
    l2 = torch.cuda.get_device_properties(wl.out_all.device).L2_cache_size
    fns, copies = [], []
    for si in range(len(wl.shapes)):
        x, q, sa = wl.x[si], wl.q[si], wl.sa[si]
        per = x.numel() * x.element_size() + q.numel() + sa.numel() * 4
        n = 1 if per < (1 << 20) else min(16, -(-2 * l2 // per))
        xs, qs, sas = [x] + [x.clone() for _ in range(n - 1)], [q] + [torch.empty_like(q) for _ in range(n - 1)], \
            [sa] + [torch.empty_like(sa) for _ in range(n - 1)]
        fns.append(lambda i, xs=xs, qs=qs, sas=sas, n=n: fp8act.fp8_act_quant(xs[i % n], qs[i % n], sas[i % n],
                                                                             stream=stream))
        copies.append(n)
    return [(*t, n) for t, n in zip(chain_times(fns, stream, launches, reps), copies)]


# ----------------------------------------------------------- CPU oracle leg
def oracle_step_time(budget_s: float = 12.0) -> dict:
    """The CPU oracle on the same workload: act quant + exact block GEMM per
    shape at M = 1, weights quantised by the oracle beforehand (untimed).
    Repeats whole steps until `budget_s` of work has been timed."""
    import oracle
    prepared = []
    for si, (N, K) in enumerate(inputs.SHAPES):
        W = inputs.weights_bf16(N, K, inputs.weight_seed(si))
        w, sw = oracle.weight_quant(inputs.bf16_bits(W))
        x = inputs.bf16_bits(inputs.activations_bf16(1, K, inputs.activation_seed(si, 0)))
        prepared.append((x, w, sw))
    times = []
    t_total = 0.0
    while t_total < budget_s or not times:
        t0 = time.perf_counter()
        for x, w, sw in prepared:
            q, sa = oracle.act_quant(x)
            oracle.block_gemm(q, sa, w, sw)
        dt = time.perf_counter() - t0
        times.append(dt)
        t_total += dt
    step_bytes = sum(algorithmic_gemm_bytes(1, N, K) + algorithmic_quant_bytes(1, K) for N, K in inputs.SHAPES)
    per_step = statistics.median(times)
    # one more step on a single thread, for the per-core figure
    cores = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        for x, w, sw in prepared:
            q, sa = oracle.act_quant(x)
            oracle.block_gemm(q, sa, w, sw)
        single = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(cores)
    return {"value": step_bytes / per_step / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle", "seconds_per_step": per_step, "steps_timed": len(times),
            "single_thread_value": step_bytes / single / 1e9,
            "sample": f"{len(times)} full decode steps (M=1, all five shapes: act quant + exact int64/fp64 GEMM); "
                      f"weight quantisation untimed; single_thread_value from one more step on one thread"}


# ----------------------------------------------------------------- runner
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world: int, v: float) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


REF_WINDOWS = 10  # a reference step multiplies one tenth of each shape's weight rows


def _oracle_prepared() -> list:
    """Seeded weights quantised by the oracle and the M = 1 activations, per shape (untimed)."""
    import oracle
    prepared = []
    for si, (N, K) in enumerate(inputs.SHAPES):
        W = inputs.weights_bf16(N, K, inputs.weight_seed(si))
        w, sw = oracle.weight_quant(inputs.bf16_bits(W))
        x = inputs.bf16_bits(inputs.activations_bf16(1, K, inputs.activation_seed(si, 0)))
        prepared.append((N, K, x, w, sw))
    return prepared


def _oracle_window_step(prepared: list, i: int) -> int:
    """One bounded reference step: act quant + exact block GEMM of every shape
    on weight-row window i % REF_WINDOWS (whole 128-row blocks; consecutive
    steps walk the windows, so the weights stream from memory, not cache).
    Returns the algorithmic bytes the step covered."""
    import oracle
    nbytes = 0
    for N, K, x, w, sw in prepared:
        nb = (N + G - 1) // G
        j = i % REF_WINDOWS
        b0, b1 = j * nb // REF_WINDOWS, (j + 1) * nb // REF_WINDOWS
        r0, r1 = b0 * G, min(b1 * G, N)
        q, sa = oracle.act_quant(x)
        oracle.block_gemm(q, sa, w[r0:r1], sw[b0:b1])
        nbytes += algorithmic_gemm_bytes(1, r1 - r0, K) + algorithmic_quant_bytes(1, K)
    return nbytes


def run_reference(args, world: int, rank: int) -> None:
    """The reference arm: the CPU oracle on the decode workload, W warm-up and
    K timed steps, each step a tenth of every shape's weight rows."""
    if rank != 0:
        return
    import oracle
    prepared = _oracle_prepared()
    for i in range(args.warmup):
        _oracle_window_step(prepared, i)
    t0 = time.perf_counter()
    nbytes = 0
    for i in range(args.steps):
        nbytes += _oracle_window_step(prepared, args.warmup + i)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    sample = (f"{args.steps} steps, each the act quant + exact int64/fp64 block GEMM of all five shapes at M=1 on "
              f"one of {REF_WINDOWS} weight-row windows (windows walked in turn); weight quantisation untimed")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64+f64",
            "data": "synthetic", "config": {"workload": WORKLOADS["decode"][1], "M": 1, "shapes": inputs.SHAPES},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def sweep(weights, device, stream, peaks) -> dict:
    """us/call of the block GEMM per shape at every workload M (outside the
    timed step), compact: per M the five us/call and the fraction of the
    roofline (HBM up to M = 102, FP8 tensor peak at 4096; burst peaks, each
    GEMM runs alone); and at M = 64, 102 and 4096 the five shapes as one
    grouped call (one launch)."""
    res = {"shapes": [list(sh) for sh in weights.shapes], "us": {}, "frac": {}}
    hbm = peaks["hbm_gbs"]
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    for M in (1, 2, 3, 4, 5, 6, 7, 8, 64, 102, 4096):
        wl = Workload(M, weights, device)
        ts = gemm_kernel_times(wl, stream, launches=30 if M <= 102 else 3, reps=3)
        res["us"][str(M)] = [round(t * 1e6, 2) for t in ts]
        if M <= 102:
            fr = [algorithmic_gemm_bytes(M, N, K) / t / 1e9 / hbm for (N, K), t in zip(wl.shapes, ts)]
        else:
            fr = [2.0 * M * N * K / t / 1e12 / fp8_peak for (N, K), t in zip(wl.shapes, ts)]
        res["frac"][str(M)] = [round(f, 3) for f in fr]
        del wl
        torch.cuda.empty_cache()
    # the five shapes as one grouped call (one launch: us and fraction of the lot)
    res["grouped"] = {}
    for M in (64, 102, 4096):
        wl = Workload(M, weights, device, grouped=True)
        (t,) = gemm_kernel_times(wl, stream, launches=30 if M <= 102 else 3, reps=3)
        if M <= 102:
            fr = sum(algorithmic_gemm_bytes(M, N, K) for N, K in wl.shapes) / t / 1e9 / hbm
        else:
            fr = sum(2.0 * M * N * K for N, K in wl.shapes) / t / 1e12 / fp8_peak
        res["grouped"][str(M)] = {"us": round(t * 1e6, 2), "frac": round(fr, 3)}
        del wl
        torch.cuda.empty_cache()
    return res


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiling runs)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work to time")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode",
                    help="decode (M=1, the headline), verify, batched or prefill")
    ap.add_argument("--m", type=int, default=None, help="token count for the chosen workload")
    ap.add_argument("--floor", action="store_true",
                    help="also time the streaming-read floor of each shape's weights (diagnostic)")
    ap.add_argument("--repeats", type=int, default=5,
                    help="extra timed repetitions of the K steps, reported as min / median / max")
    ap.add_argument("--steps-per-graph", type=int, default=10,
                    help="consecutive steps captured in one CUDA graph (timed steps stay exactly --steps)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    from block_scaled_fp8_act_gb300 import fp8act
    fp8act.load(build=True)
    device = torch.device("cuda", torch.cuda.current_device())
    peaks, peaks_kind = load_peaks()
    stream = torch.cuda.Stream()

    M = args.m if args.m else WORKLOADS[args.workload][0]
    desc = WORKLOADS[args.workload][1].format(M=M, k=M - 1)
    # FP8 ridge point ~560 flop/B (measured tensor / HBM peaks) ~ M = 280 tokens
    bound = "tensor" if M > 280 else "hbm"
    weight_only = args.workload in WEIGHT_ONLY
    grouped = args.workload in GROUPED
    fused = args.workload in FUSED
    if (weight_only or fused) and M > 16:
        ap.error("the weight-only and fused workloads are decode paths (M <= 16)")
    kernel = ("gemm_skinny_grouped_kernel" if M <= 16 else "gemm_tc_grouped_kernel") if grouped \
        else gemm_kernel_name(M)
    if fused and M <= 8:
        kernel = "linear_persistent_kernel"  # the fused call's one-CTA-per-SM kernel
    if args.workload in WORKLOAD_SHAPES:
        shapes, seeds = WORKLOAD_SHAPES[args.workload]
        weights = Weights(device, shapes=shapes, seed_index=seeds)
    else:
        weights = Weights(device)
    wl = Workload(M, weights, device, weight_only=weight_only, grouped=grouped, fused=fused)
    # One graph per step, and graphs of S consecutive steps (step i uses weight copy i mod
    # copies, as in the one-step graphs), the way a serving loop captures a whole forward
    # pass of many layers: programmatic dependent launch overlaps consecutive kernels
    # inside a graph but not across graph launches.
    S = max(1, min(args.steps_per_graph, args.steps))
    graphs = [capture(lambda c=c: wl.enqueue_step(c, stream), stream) for c in range(wl.copies)]
    multi = [capture(lambda j=j: [wl.enqueue_step((j * S + s) % wl.copies, stream) for s in range(S)], stream)
             for j in range(wl.copies)] if S > 1 else graphs
    launches_per_step = wl.launches_per_step()

    def replay_steps(n: int) -> None:
        """Exactly n steps: n // S replays of the S-step graphs, then single steps."""
        for kind, c in graph_schedule(n, S, wl.copies):
            (multi if kind == "multi" else graphs)[c].replay()

    # ---- timed region: K steps of the whole path, graphs replayed back to back
    with torch.cuda.stream(stream):
        replay_steps(args.warmup)
        if S > 1:
            for g in multi:  # first replays (graph upload) stay out of the timed region
                g.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            start.record(stream)
            replay_steps(args.steps)
            end.record(stream)
        end.synchronize()
        torch.cuda.synchronize()
        barrier(world)
        t_step = start.elapsed_time(end) / 1e3 / args.steps
        # the same K steps again, args.repeats times, for the spread
        rep_ms = []
        for _ in range(args.repeats):
            r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                r0.record(stream)
                replay_steps(args.steps)
                r1.record(stream)
            r1.synchronize()
            rep_ms.append(r0.elapsed_time(r1) / args.steps)
        # dominant kernel: the block GEMM, timed per shape on the same stream
        gemm_spread = []
        gemm_ts = gemm_kernel_times(wl, stream, launches=60 if M <= 128 else 8, spread=gemm_spread)
    t_step = max_over_ranks(world, t_step)
    step_bytes = wl.step_bytes()
    step_flops = sum(2.0 * M * N * K for N, K in wl.shapes)
    if bound == "tensor":
        value, unit = world * step_flops / t_step / 1e12, "TFLOP/s"
    else:
        value, unit = world * step_bytes / t_step / 1e9, "GB/s"

    # ---- e2e: public API, activations from pinned host, outputs back, every step
    def e2e_step(c):
        wl.x_all.copy_(wl.x_host_all, non_blocking=True)
        wl.enqueue_step(c, stream)
        wl.out_host_all.copy_(wl.out_all, non_blocking=True)
    e2e_steps = 0 if args.no_e2e else max(50, args.steps // 10)

    def timed_e2e(run) -> float:
        """Seconds per step of `run(i)` over e2e_steps steps: the larger of the
        CUDA-event time on the stream and the host wall time."""
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                run(i)
            torch.cuda.synchronize()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0 = time.perf_counter()
            s0.record(stream)
            for i in range(e2e_steps):
                run(i)
            s1.record(stream)
            s1.synchronize()
            wall = (time.perf_counter() - t0) / max(e2e_steps, 1)
        return max(s0.elapsed_time(s1) / 1e3 / max(e2e_steps, 1), wall)

    def timed_e2e_pipelined() -> tuple[float, int, int]:
        """Seconds per step, steps timed and steps per graph, with every step's host
        copies inside the timed region, overlapped with the neighbouring steps'
        compute (independent batches, as a server streams them). P steps form one
        CUDA graph replay (as in the device-timed leg where a step's host copies
        are at most 2 MB, one step per replay above). Replay r runs
        on buffer-set group r % 2: its P uploads go out on an upload stream once
        replay r - 2 has read that group's activations, the replay waits for them
        and for the group's previous outputs to be back on the host, and its P
        downloads follow on a download stream. The larger of the event time (first
        upload to last download) and the host wall time."""
        per_set = (wl.x_all.numel() + wl.out_all.numel()) * 2
        # Where a step's copies are large the host link sets the pace and finer
        # replays overlap it better (measured at M = 102: 2865 GB/s with one step
        # per replay, 2580 with ten); small copies hide entirely either way and
        # the longer replays save the per-replay boundary (decode: 4093 against 3911).
        P = S if per_set <= (2 << 20) else 1
        groups = [[wl if (g, k) == (0, 0) else
                   Workload(M, weights, device, weight_only=weight_only, grouped=grouped, fused=fused)
                   for k in range(P)] for g in range(2)]
        # replay r: weight copy of its step k is (r P + k) mod copies; the graph depends on
        # r mod 2 (buffer group) and r P mod copies
        n_graphs = 2 * wl.copies
        step_graphs = [capture(lambda j=j: [groups[j % 2][k].enqueue_step((j * P + k) % wl.copies, stream)
                                            for k in range(P)], stream) for j in range(n_graphs)]
        up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)

        def run(reps: int) -> tuple[float, float]:
            ev_in = [torch.cuda.Event() for _ in range(reps)]
            ev_comp = [torch.cuda.Event() for _ in range(reps)]
            ev_out = [torch.cuda.Event() for _ in range(reps)]
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            s0.record(up)
            for r in range(reps):
                sets = groups[r % 2]
                with torch.cuda.stream(up):
                    if r >= 2:
                        up.wait_event(ev_comp[r - 2])  # replay r - 2 has read this group's activations
                    for st in sets:
                        st.x_all.copy_(st.x_host_all, non_blocking=True)
                    ev_in[r].record(up)
                with torch.cuda.stream(stream):
                    stream.wait_event(ev_in[r])
                    if r >= 2:
                        stream.wait_event(ev_out[r - 2])  # this group's outputs are back on the host
                    step_graphs[r % n_graphs].replay()
                    ev_comp[r].record(stream)
                with torch.cuda.stream(down):
                    down.wait_event(ev_comp[r])
                    for st in sets:
                        st.out_host_all.copy_(st.out_all, non_blocking=True)
                    ev_out[r].record(down)
            s1.record(down)
            s1.synchronize()
            wall = time.perf_counter() - t0
            return s0.elapsed_time(s1) / 1e3, wall

        run(max(-(-args.warmup // P), 2))
        reps = max(2, -(-e2e_steps // P))
        ev_t, wall = run(reps)
        del step_graphs, groups
        return max(ev_t, wall) / (reps * P), reps * P, P

    # Eager: every API call issued from Python each step (binding overhead included).
    t_e2e_eager = max_over_ranks(world, timed_e2e(lambda i: e2e_step(i % wl.copies)))
    # Pipelined: copies on their own streams, overlapping the neighbouring steps' compute.
    t_e2e_pipe, e2e_pipe_steps, e2e_pipe_per_graph = timed_e2e_pipelined() if e2e_steps else (float("inf"), 0, 0)
    t_e2e_pipe = max_over_ranks(world, t_e2e_pipe)
    # Graph: the same calls (copies included) captured once and replayed per step.
    e2e_graphs = [capture(lambda c=c: e2e_step(c), stream) for c in range(wl.copies)]
    t_e2e = max_over_ranks(world, timed_e2e(lambda i: e2e_graphs[i % wl.copies].replay()))
    del e2e_graphs
    h2d = wl.x_host_all.numel() * 2
    d2h = wl.out_host_all.numel() * 2
    step_units = step_flops / 1e12 if bound == "tensor" else step_bytes / 1e9

    units = wl.gemm_units()
    gemm_bytes = [u[1] for u in units]
    gemm_flops = [u[2] for u in units]
    labels = [u[0] for u in units]
    traffic = recorded_traffic(kernel, f"{args.workload}_m{M}_" + ("per_launch" if grouped else "mean_of_5"))
    if bound == "tensor":
        achieved = sum(gemm_flops) / sum(gemm_ts) / 1e12
        # a millisecond-long GEMM inside a long step runs under the power cap:
        # the sustained bf16 rate (seconds-long cuBLAS loop) is its reference
        peak = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])) * FP8_OVER_BF16
        peak_kind = (f"{peaks_kind} bf16 dense (cuBLAS, sustained under the power cap) x {FP8_OVER_BF16:g}, "
                     "the nominal FP8/bf16 ratio")
        roof_unit, per_launch = "TFLOP/s", {"flops_per_launch": sum(gemm_flops) / len(gemm_flops)}
        per_shape = [{**_label(lb), "us_per_call": round(t * 1e6, 3), "us_p10": round(lo * 1e6, 3),
                      "us_p90": round(hi * 1e6, 3), "tflops": round(f / t / 1e12, 1),
                      "frac": round(f / t / 1e12 / peak, 4)}
                     for lb, t, f, (lo, hi) in zip(labels, gemm_ts, gemm_flops, gemm_spread)]
    else:
        achieved = sum(gemm_bytes) / sum(gemm_ts) / 1e9
        peak = float(peaks["hbm_gbs"])
        peak_kind = f"{peaks_kind} HBM copy bandwidth"
        roof_unit, per_launch = "GB/s", {"bytes_per_launch": sum(gemm_bytes) / len(gemm_bytes)}
        per_shape = [{**_label(lb), "us_per_call": round(t * 1e6, 3), "us_p10": round(lo * 1e6, 3),
                      "us_p90": round(hi * 1e6, 3), "gbs": round(b / t / 1e9, 1),
                      "frac": round(b / t / 1e9 / peak, 4)}
                     for lb, t, b, (lo, hi) in zip(labels, gemm_ts, gemm_bytes, gemm_spread)]

    floor = None
    if args.floor and not wl.grouped:
        fts = floor_times(wl, stream)
        floor = [{"N": N, "K": K, "floor_us": round(f * 1e6, 3), "floor_gbs": round(N * K / f / 1e9, 1),
                  "gemm_us": round(g * 1e6, 3), "gemm_over_floor": round(g / f, 3)}
                 for (N, K), f, g in zip(wl.shapes, fts, gemm_ts)]
    # the activation quantisation, reported on its own (HBM bound at large M)
    act_quant = None
    if not wl.bf16_in and not wl.grouped:
        act_quant = [{"K": K, "us_per_call": round(med * 1e6, 3), "us_p10": round(lo * 1e6, 3),
                      "us_p90": round(hi * 1e6, 3), "gbs": round(algorithmic_quant_bytes(M, K) / med / 1e9, 1),
                      "frac": round(algorithmic_quant_bytes(M, K) / med / 1e9 / float(peaks["hbm_gbs"]), 4),
                      "input_copies": n}
                     for (_, K), (med, lo, hi, n) in zip(wl.shapes, quant_kernel_times(wl, stream))]
    del graphs, multi
    torch.cuda.synchronize()
    result = {
        "metric": METRIC if args.workload == "decode" else f"block-FP8 linear, {desc}",
        "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 x e4m3 -> f32 acc -> bf16" if weight_only else "e4m3 x e4m3 -> f32 acc -> bf16",
        "data": "synthetic",
        "config": {"workload": desc, "M": M, "shapes": [list(s) for s in wl.shapes],
                   "l2": f"inputs larger than L2: {wl.copies} rotating weight copies "
                         f"({wl.copies * sum(N * K for N, K in wl.shapes) / 1e6:.0f} MB), no flush",
                   "graphs": f"{S} steps per CUDA graph replay ({launches_per_step} kernels per step)",
                   "steps_per_graph": S,
                   "parallelism": f"replicas x{world}"},
        "repeats": {"n": len(rep_ms), "ms_per_step_min": round(min(rep_ms), 5) if rep_ms else None,
                    "ms_per_step_median": round(statistics.median(rep_ms), 5) if rep_ms else None,
                    "ms_per_step_max": round(max(rep_ms), 5) if rep_ms else None},
        "us_per_call": per_shape,
        "act_quant": act_quant,
        "floor": floor,
        "gpu_launches": args.steps * launches_per_step,
        "roofline": {"bound": bound, "kernel": kernel, "achieved": round(achieved, 1),
                     "peak": round(peak, 1), "unit": roof_unit, "frac": round(achieved / peak, 4),
                     "frac_nominal": round(achieved / (NOMINAL_HBM_GBS if bound == "hbm" else NOMINAL_FP8_TFLOPS), 4),
                     "traffic": traffic, "peak_kind": peak_kind, **per_launch,
                     "us_per_launch": round(sum(gemm_ts) / len(gemm_ts) * 1e6, 3)},
        "e2e": {"value": round(world * step_units / t_e2e_pipe, 2),
                "unit": unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(t_e2e_pipe * 1e3, 5),
                "steps": e2e_pipe_steps, "steps_per_graph": e2e_pipe_per_graph,
                "how": "each step: one H2D copy of all its activations from pinned host memory, the step's "
                       "API calls (captured once through the public API), one D2H copy of all its outputs, "
                       "every copy inside the timed region; steps_per_graph consecutive steps per CUDA graph "
                       "replay on their own buffer sets, their uploads and downloads on separate streams "
                       "overlapping the neighbouring replays' compute (independent batches)",
                "serial": {"value": round(world * step_units / t_e2e, 2), "ms_per_step": round(t_e2e * 1e3, 5),
                           "how": "the same per-step copies and graph on one stream, nothing overlapped"},
                "eager": {"value": round(world * step_units / t_e2e_eager, 2),
                          "ms_per_step": round(t_e2e_eager * 1e3, 5),
                          "how": "serial, with the calls issued from Python every step (ctypes binding "
                                 "overhead included)"}},
        "clocks": clk.summary(),
    }
    if not args.no_sweep and rank == 0 and args.workload == "decode":
        del wl
        torch.cuda.empty_cache()
        sw_res = sweep(weights, device, stream, peaks)
        # ahead of the long fields, so that a truncated tail of the line keeps it
        keys = list(result)
        at = keys.index("us_per_call")
        result = {**{k: result[k] for k in keys[:at]}, "sweep": sw_res, **{k: result[k] for k in keys[at:]}}
    if rank == 0 and not args.no_cpu_baseline:
        cb = oracle_step_time(budget_s=args.cpu_budget)
        result["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample", "single_thread_value")}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
