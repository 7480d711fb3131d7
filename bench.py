"""Benchmark of the MXFP8 hot path on GB300.

One step = one pass of the path over one batch of synthetic inputs:
MX-quantise X, W and dY (row and column copies, one fused pass each), then the
fprop, dgrad and wgrad block-scaled GEMMs. Default workload: the dense FFN
up-projection (tokens M=8192, K=2048, N=10944), DeepSeek-V3 16B shaped. The
default line also carries every other workload's own measurement under
"configs" (single Linear, MLA projections, routed experts, quantiser sweep,
blockwise FP8 and current-scaling variants, FP32 weight refresh); --workload
NAME prints one alone.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload dense_ffn]
    python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Timing: CUDA events on the launching stream around exactly K steps, barrier +
synchronize on both sides, max over ranks. Per-kernel CUDA events inside the
timed region give the dominant kernel's average launch time for the roofline.
The inputs and MX copies of a step (~0.7 GB) exceed the 129 MB L2, so no flush
is done between steps. Multi-GPU: independent replicas (no data-path
collective); value = work of all ranks / max time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

PEAK_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s)

# The headline metric: the same string on both arms, so the two lines compare.
METRIC_DENSE = "MXFP8 GEMM TFLOPS (fprop+dgrad+wgrad step incl. MX quantisation, dense FFN up-proj)"
WORKLOAD_DENSE = ("dense_ffn_up_proj M=8192 K=2048 N=10944: quantise X,W,dY (row+col) + fprop + dgrad + wgrad")


def fp8_peaks(peaks, src):
    """FP8 tensor peak (TFLOP/s) as the measured BF16 cuBLAS rate x the nominal
    FP8/BF16 ratio: the burst figure for the bench's timed regions (milliseconds
    to tens of milliseconds, far shorter than the sustained probe's seconds
    under the power cap), and the sustained one, reported beside it."""
    burst = peaks["bf16_tflops"] * FP8_OVER_BF16
    sustained = peaks["bf16_tflops_sustained"] * FP8_OVER_BF16
    label = (f"{src} bf16 burst {peaks['bf16_tflops']} x nominal fp8/bf16 ratio {FP8_OVER_BF16} (timed region "
             f"< 1 s); frac_sustained uses bf16 sustained {peaks['bf16_tflops_sustained']}")
    return burst, sustained, label


def tensor_roofline(kernel, achieved, peaks, src, **extra):
    burst, sustained, label = fp8_peaks(peaks, src)
    d = {"bound": "tensor", "kernel": kernel, "achieved": achieved, "peak": burst, "unit": "TFLOP/s",
         "frac": achieved / burst, "frac_sustained": achieved / sustained, "peak_source": label}
    d.update(extra)
    return d


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAK_FALLBACK), "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (replicas)
# ---------------------------------------------------------------------------

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # raw samples go to the temp directory; the line carries their summary
        self.path = os.path.join(tempfile.gettempdir(), f"mxfp8_bench_clocks_gpu{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx_ = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx_) if mx_ else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

TIMING_NOTE = ("value: the timed region, K steps with no event inside them; per-kernel durations (roofline): "
               "K further steps with a CUDA-event span around each kernel launch or launch group")


class Timers:
    """CUDA events around the launches of one kernel family inside the timed region."""

    def __init__(self):
        self.pairs = {}

    def span(self, name, stream):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        self.pairs.setdefault(name, []).append((s, e))
        return e

    def total_ms(self, name):
        return sum(s.elapsed_time(e) for s, e in self.pairs.get(name, []))

    def count(self, name):
        return len(self.pairs.get(name, []))


class DenseFFN:
    """fprop Y = X W^T, dgrad dX = dY W, wgrad dW = dY^T X with MX copies of X, W, dY."""
    name = "dense_ffn_up_proj"

    def __init__(self, M=8192, K=2048, N=10944, seed=None):
        import mxfp8_block_scaled_gb300 as mx
        self.mx = mx
        self.M, self.K, self.N = M, K, N
        d = dense_host_inputs()
        self.host = {k: d[k].pin_memory() for k in ("X", "W", "dY")}
        # Two slots of device inputs and outputs, so the end-to-end run can copy
        # one step's data while another step computes.
        self.dev_slots = [{k: v.cuda() for k, v in self.host.items()} for _ in range(2)]
        self.dev = self.dev_slots[0]
        self.alloc()

    def alloc(self):
        mx = self.mx
        M, K, N = self.M, self.K, self.N
        u8 = dict(dtype=torch.uint8, device="cuda")

        def copies(R, C):
            return (mx.MXTensor(torch.empty((R, C), **u8), torch.empty(mx.mx_scale_bytes(R, C), **u8), R, C,
                                mx.MX_ROWWISE),
                    mx.MXTensor(torch.empty((C, R), **u8), torch.empty(mx.mx_scale_bytes(C, R), **u8), C, R,
                                mx.MX_COLWISE))
        self.q = {"X": copies(M, K), "W": copies(N, K), "dY": copies(M, N)}
        bf = dict(dtype=torch.bfloat16, device="cuda")
        self.out_slots = [{"Y": torch.empty((M, N), **bf), "dX": torch.empty((M, K), **bf),
                           "dW": torch.empty((N, K), **bf)} for _ in range(2)]
        self.out = self.out_slots[0]
        self.host_out = [{k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in self.out.items()}
                         for _ in range(2)]

    def gemm_flops(self):
        return 2.0 * self.M * self.N * self.K          # identical for the three modes here

    def step_flops(self):
        return 3 * self.gemm_flops()

    def quant_bytes(self):
        # algorithmic bytes of one fused both-axes pass: 2 read + 1 + 1 written + 2 * (1/32) scales per element
        return {k: (2 + 1 + 1 + 2 / 32) * r.rows * r.k for k, (r, _) in self.q.items()}

    def launches_per_step(self):
        # two quantiser launches, fprop, and dgrad + wgrad in one launch
        (xr, xc), (wr, wc) = self.q["X"], self.q["W"]
        return 2 + gemm_launches(self.mx, self.mx.MX_FPROP, xr, wr) + 1

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host.values())

    def d2h_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.out.values())

    def step(self, stream, timers=None, slot=0):
        mx = self.mx
        sp = stream.cuda_stream
        dev, out_t = self.dev_slots[slot], self.out_slots[slot]
        # X and W (what the forward GEMM reads) in one launch; dY, which only
        # exists once the backward pass starts, in a second.
        for names in (("X", "W"), ("dY",)):
            descs = []
            for k in names:
                x = dev[k]
                r, c = self.q[k]
                descs.append(mx.MXQuantTensorC(x.data_ptr(), x.shape[0], x.shape[1], x.stride(0), r.data.data_ptr(),
                                               r.scale.data_ptr(), c.data.data_ptr(), c.scale.data_ptr()))
            e = timers.span(("quant", "+".join(names)), stream) if timers else None
            mx.mx_quantize_multi(descs, mx.MX_BOTH, None, sp)
            if e is not None:
                e.record(stream)
        (xr, xc), (wr, wc), (dr, dc) = self.q["X"], self.q["W"], self.q["dY"]
        # fprop; then the backward pass's dgrad and wgrad, independent of each
        # other, in one launch
        e = timers.span("gemm", stream) if timers else None
        mx.mx_gemm(mx.MX_FPROP, xr.c_operand(), wr.c_operand(), out_t["Y"].data_ptr(), out_t["Y"].stride(0), None,
                   sp)
        mx.mx_gemm_multi([mx.MXGemmProblemC(dr.c_operand(), wc.c_operand(), out_t["dX"].data_ptr(),
                                            out_t["dX"].stride(0), mx.MX_DGRAD, 0),
                          mx.MXGemmProblemC(dc.c_operand(), xc.c_operand(), out_t["dW"].data_ptr(),
                                            out_t["dW"].stride(0), mx.MX_WGRAD, 0)], None, sp)
        if e is not None:
            e.record(stream)

    def run_e2e(self, stream, steps):
        """`steps` end-to-end steps: each copies its inputs from pinned host memory,
        runs the step and copies its three outputs back. Step i's inputs go in on
        one copy stream and step i-1's outputs come out on another while step i-1
        and step i compute, through two slots of device buffers; every copy of
        every step stays inside the caller's timed region."""
        h2d, d2h = self._copy_streams()
        ev = lambda: torch.cuda.Event()
        inputs_free = [None, None]   # slot's inputs consumed by its last step
        outputs_free = [None, None]  # slot's outputs copied out
        start = ev()
        start.record(stream)
        h2d.wait_event(start)
        d2h.wait_event(start)
        for i in range(steps):
            slot = i & 1
            if inputs_free[slot] is not None:
                h2d.wait_event(inputs_free[slot])
            with torch.cuda.stream(h2d):
                for k in self.host:
                    self.dev_slots[slot][k].copy_(self.host[k], non_blocking=True)
            landed = ev()
            landed.record(h2d)
            stream.wait_event(landed)
            if outputs_free[slot] is not None:
                stream.wait_event(outputs_free[slot])
            self.step(stream, slot=slot)
            done = ev()
            done.record(stream)
            inputs_free[slot] = done
            d2h.wait_event(done)
            with torch.cuda.stream(d2h):
                for k, t in self.out_slots[slot].items():
                    self.host_out[slot][k].copy_(t, non_blocking=True)
            out_done = ev()
            out_done.record(d2h)
            outputs_free[slot] = out_done
        stream.wait_stream(h2d)
        stream.wait_stream(d2h)

    def _copy_streams(self):
        if not hasattr(self, "_h2d"):
            self._h2d, self._d2h = torch.cuda.Stream(), torch.cuda.Stream()
        return self._h2d, self._d2h


# ---------------------------------------------------------------------------
# CPU oracle timing
# ---------------------------------------------------------------------------

_DENSE_HOST = {}


def dense_host_inputs():
    if not _DENSE_HOST:
        import workloads
        _DENSE_HOST.update(workloads.dense_ffn(M=8192, K=2048, N=10944))
    return _DENSE_HOST


def _f64(t):
    import oracle
    return oracle.bf16_bits_to_float64(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def oracle_linear_sample(X, W, dY, rows: int, cols: int, seed: int = 7):
    """Time the oracle on a bounded sample of one Linear layer's step (X [M, K],
    W [N, K], dY [M, N]): for each of fprop/dgrad/wgrad, a [rows x cols] block
    of outputs (fewer where the GEMM is narrower), including the oracle
    quantisation of exactly the operand rows/columns that block reads.
    Returns (flops_of_sample, seconds)."""
    import oracle
    M, K = X.shape
    N = W.shape[0]
    g = np.random.Generator(np.random.Philox(seed))
    picks = []
    for (Mg, Ng, Kg) in ((M, N, K), (M, K, N), (N, K, M)):
        picks.append((np.sort(g.choice(Mg, min(rows, Mg), replace=False)),
                      np.sort(g.choice(Ng, min(cols, Ng), replace=False)), Kg))
    # slices of the BF16 sources (host copies, not timed)
    (i0, j0, _), (i1, j1, _), (i2, j2, _) = picks
    srcs = [(_f64(X[torch.from_numpy(i0)]), _f64(W[torch.from_numpy(j0)])),
            (_f64(dY[torch.from_numpy(i1)]), _f64(W[:, torch.from_numpy(j1)])),
            (_f64(dY[:, torch.from_numpy(i2)]), _f64(X[:, torch.from_numpy(j2)]))]
    t0 = time.perf_counter()
    a, b = srcs[0]
    oracle.mx_gemm_ref(*oracle.mx_quantize_rowwise(a), *oracle.mx_quantize_rowwise(b))
    a, b = srcs[1]
    oracle.mx_gemm_ref(*oracle.mx_quantize_rowwise(a), *oracle.mx_quantize_colwise(b))
    a, b = srcs[2]
    oracle.mx_gemm_ref(*oracle.mx_quantize_colwise(a), *oracle.mx_quantize_colwise(b))
    dt = time.perf_counter() - t0
    flops = sum(2.0 * len(i) * len(j) * Kg for (i, j, Kg) in picks)
    return flops, dt


def oracle_dense_sample(rows: int, cols: int, seed: int = 7):
    """The dense FFN up-projection's sample (see oracle_linear_sample)."""
    d = dense_host_inputs()
    return oracle_linear_sample(d["X"], d["W"], d["dY"], rows, cols, seed)


def cpu_threads():
    n = os.cpu_count() or 1
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            n = int(os.environ[v])
    return n


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def profile_traffic(kernel: str, field: str = "bytes_per_step"):
    """DRAM traffic of a roofline entry's launches (bytes per step, or per
    launch, as that entry counts its time) from a committed ncu summary, if it
    was taken from the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(kernel)
    if not ent:
        return None
    src = os.path.join(ROOT, "mxfp8_block_scaled_gb300", "csrc", ent.get("source", ""))
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return ent.get(field) if h == ent.get("source_sha256_16") else None


def run_reference(args, rank, world):
    if rank != 0:
        return
    rows = cols = 64
    for _ in range(args.warmup):
        oracle_dense_sample(rows, cols)
    t_total = 0.0
    flops_total = 0.0
    for s in range(args.steps):
        fl, dt = oracle_dense_sample(rows, cols, seed=100 + s)
        t_total += dt
        flops_total += fl
    v = flops_total / t_total / 1e12
    line = {"impl": "reference", "metric": METRIC_DENSE,
            "value": v, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * t_total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_DENSE,
                       "sample": f"{rows}x{cols} output block per GEMM per step"},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": f"{rows}x{cols} output block of each GEMM per step, with the oracle "
                                       f"quantisation of the operand rows it reads"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


class MoEExperts:
    """Routed-expert step (64 experts, 49152 rows, gate_up N=2816/K=2048 and
    down N=2048/K=1408): quantise the activation and the output gradient of each
    projection (row copy + per-group padded column copy in one pass), then the
    grouped fprop, dgrad and wgrad GEMMs of both projections. The stacked
    weights' row and column copies are refreshed apart (refresh_weights)."""
    name = "moe_routed_experts"

    def __init__(self):
        import mxfp8_block_scaled_gb300 as mx
        self.mx = mx
        d = moe_host_inputs()
        self.offsets = torch.from_numpy(d["offsets"]).cuda()
        self.counts = d["counts"]
        self.M = int(d["offsets"][-1])
        self.cap = mx.mx_grouped_padded_rows(d["offsets"])
        self.proj = []
        for a_key, w_key, dy_key in (("X", "W_gate_up", "dY_gate_up"), ("A_down", "W_down", "dY_down")):
            A = d[a_key].cuda()
            W = d[w_key].cuda()
            dY = d[dy_key].cuda()
            E, N, K = W.shape
            ar, ac = mx.quantize(A, mx.MX_BOTH, group_offsets=self.offsets, col_capacity=self.cap)
            dr, dc = mx.quantize(dY, mx.MX_BOTH, group_offsets=self.offsets, col_capacity=self.cap)
            wr, wc = mx.quantize_stacked(W, mx.MX_BOTH)
            bf = dict(dtype=torch.bfloat16, device="cuda")
            outs = {"Y": torch.empty((self.M, N), **bf), "dX": torch.empty((self.M, K), **bf),
                    "dW": torch.empty((E, N, K), **bf)}
            self.proj.append(dict(A=A, W=W, dY=dY, ar=ar, ac=ac, dr=dr, dc=dc, wr=wr, wc=wc, out=outs, E=E, N=N, K=K))
        del d

    def gemm_flops(self):
        return [2.0 * self.M * pr["N"] * pr["K"] for pr in self.proj for _ in range(3)]

    def step_flops(self):
        return sum(self.gemm_flops())

    def refresh_weights(self, stream, timers=None):
        """The weight refresh after an optimizer step: row and column copies of
        both projections' stacked weights ("DeepSeek-V3 16B FSDP2 MXFP8/HiF8
        训练设计" §8.1: weights are quantised once after each optimizer step and
        reused by the micro-batches and recomputation that follow)."""
        mx = self.mx
        sp = stream.cuda_stream
        for pr in self.proj:
            W, wr, wc = pr["W"], pr["wr"], pr["wc"]
            e = timers.span("wquant", stream) if timers else None
            mx.mx_quantize_batched(W.data_ptr(), pr["E"], pr["N"], pr["K"], pr["K"], pr["N"] * pr["K"], mx.MX_BOTH,
                                   wr.data.data_ptr(), wr.scale.data_ptr(), wc.data.data_ptr(), wc.scale.data_ptr(),
                                   None, sp)
            if e is not None:
                e.record(stream)

    def step(self, stream, timers=None):
        """One micro-batch: the forward chain gate_up -> SwiGLU (fused into
        gate_up's epilogue) -> down, then each projection's dgrad and wgrad, with
        the activations and output gradients quantised (row copy + per-expert
        column copy in one pass each). The output gradients are the synthetic dY
        tensors; the weights' copies come from the last refresh_weights."""
        mx = self.mx
        sp = stream.cuda_stream
        o = self.offsets.data_ptr()
        E = self.offsets.numel() - 1
        for j, pr in enumerate(self.proj):
            for src, r, c in ((pr["A"], pr["ar"], pr["ac"]), (pr["dY"], pr["dr"], pr["dc"])):
                e = timers.span("quant", stream) if timers else None
                mx.mx_quantize(src.data_ptr(), src.shape[0], src.shape[1], src.stride(0), mx.MX_BOTH,
                               r.data.data_ptr(), r.scale.data_ptr(), c.data.data_ptr(), c.scale.data_ptr(), o, E,
                               self.cap, None, sp)
                if e is not None:
                    e.record(stream)
            wr, wc = pr["wr"], pr["wc"]
            for mode, a, b, out in ((mx.MX_FPROP, pr["ar"], wr, pr["out"]["Y"]),
                                    (mx.MX_DGRAD, pr["dr"], wc, pr["out"]["dX"]),
                                    (mx.MX_WGRAD, pr["dc"], pr["ac"], pr["out"]["dW"])):
                e = timers.span("gemm", stream) if timers else None
                if mode == mx.MX_FPROP and j == 0:
                    # gate_up fprop with SwiGLU in the epilogue: writes the down projection's input
                    mx.mx_grouped_gemm_swiglu(a.c_operand(), b.c_operand(), o, E, self.proj[1]["A"].data_ptr(),
                                              self.proj[1]["A"].stride(0), None, sp)
                else:
                    mx.mx_grouped_gemm(mode, a.c_operand(), b.c_operand(), o, E, out.data_ptr(), out.stride(-2),
                                       None, sp)
                if e is not None:
                    e.record(stream)

    def launches_per_step(self):
        return sum(2 + 3 for pr in self.proj)


_MOE_HOST = {}


def moe_host_inputs():
    if not _MOE_HOST:
        import workloads
        _MOE_HOST.update(workloads.moe_experts())
    return _MOE_HOST


def oracle_moe_sample(rows: int, cols: int, seed: int = 11):
    """Time the oracle on a bounded sample of the routed-expert step: for the
    largest expert of each projection, a [rows x cols] block of its fprop,
    dgrad and wgrad outputs, with the oracle quantisation (per-expert column
    blocks for wgrad) of exactly the operand rows/columns that block reads.
    Returns (flops_of_sample, seconds)."""
    import oracle
    d = moe_host_inputs()
    offs = d["offsets"]
    e = int(np.argmax(np.diff(offs)))
    lo, hi = int(offs[e]), int(offs[e + 1])
    g = np.random.Generator(np.random.Philox(seed))
    flops, dt = 0.0, 0.0
    for a_key, w_key, dy_key in (("X", "W_gate_up", "dY_gate_up"), ("A_down", "W_down", "dY_down")):
        A, W, dY = d[a_key][lo:hi], d[w_key][e], d[dy_key][lo:hi]
        m, K = A.shape
        N = W.shape[0]
        i = np.sort(g.choice(m, min(rows, m), replace=False))
        jn = np.sort(g.choice(N, min(cols, N), replace=False))
        jk = np.sort(g.choice(K, min(cols, K), replace=False))
        src = [_f64(A[torch.from_numpy(i)]), _f64(W[torch.from_numpy(jn)]), _f64(dY[torch.from_numpy(i)]),
               _f64(W[:, torch.from_numpy(jk)]), _f64(dY[:, torch.from_numpy(jn[:rows])]),
               _f64(A[:, torch.from_numpy(jk)])]
        seg = np.array([0, m], dtype=np.int64)
        t0 = time.perf_counter()
        oracle.mx_gemm_ref(*oracle.mx_quantize_rowwise(src[0]), *oracle.mx_quantize_rowwise(src[1]))
        oracle.mx_gemm_ref(*oracle.mx_quantize_rowwise(src[2]), *oracle.mx_quantize_colwise(src[3]))
        a, as_, _ = oracle.mx_quantize_colwise_grouped(src[4], seg)
        b, bs, _ = oracle.mx_quantize_colwise_grouped(src[5], seg)
        oracle.mx_gemm_ref(a, as_, b, bs)
        dt += time.perf_counter() - t0
        flops += 2.0 * len(i) * len(jn) * K + 2.0 * len(i) * len(jk) * N + 2.0 * min(rows, len(jn)) * len(jk) * m
    return flops, dt


def timed_cpu_baseline(fn, budget_s: float, unit_scale: float = 1e12):
    """Repeat an oracle sample (seeds 0, 1, ...) until budget_s of oracle time;
    returns (work per second / unit_scale, seconds, repetitions)."""
    work, dt, n = 0.0, 0.0, 0
    while dt < budget_s:
        w, t = fn(n)
        work, dt, n = work + w, dt + t, n + 1
    return work / dt / unit_scale, dt, n


def run_moe(args, rank, world, peaks, peak_src):
    wl = MoEExperts()
    stream = torch.cuda.Stream()
    wl.refresh_weights(stream)
    ms, timers, clk = _measure(lambda t: wl.step(stream, t), args, world, stream)
    value = world * args.steps * wl.step_flops() / (ms / 1e3) / 1e12
    pairs = timers.pairs["gemm"]
    fl = wl.gemm_flops()
    per_gemm = []
    for i, name in enumerate(["gate_up fprop + SwiGLU epilogue", "gate_up dgrad", "gate_up wgrad", "down fprop",
                              "down dgrad", "down wgrad"]):
        t = sum(pairs[j][0].elapsed_time(pairs[j][1]) for j in range(i, len(pairs), 6)) / args.steps
        per_gemm.append({"gemm": name, "ms": t, "tflops": fl[i] / (t / 1e3) / 1e12})
    gemm_ms = timers.total_ms("gemm") / args.steps
    achieved = sum(fl) / (gemm_ms / 1e3) / 1e12
    # the refresh after an optimizer step, timed on its own (K refreshes back to back)
    rms, rtimers, _ = _measure(lambda t: wl.refresh_weights(stream, t), args, world, stream, clocks=False)
    w_elems = sum(pr["E"] * pr["N"] * pr["K"] for pr in wl.proj)
    refresh_ms = rms / args.steps
    line = {"metric": "MXFP8 grouped-GEMM TFLOPS (routed experts, fprop+dgrad+wgrad of gate_up and down incl. "
                      "MX quantisation of activations and gradients)",
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": "moe_routed_experts: 64 experts, 49152 rows (Zipf 1.1, 4 empty), gate_up "
                                   "2048->2816 with SwiGLU fused into its epilogue (writes down's input), "
                                   "down 1408->2048", "parallelism": f"replicas{world}",
                       "weights": "quantised once per optimizer step (refresh_weights, timed apart); a step is "
                                  "one micro-batch",
                       "l2": "no flush: a step moves several GB (> 129 MB L2)"},
            "per_gemm": per_gemm,
            "roofline": tensor_roofline("mx_gemm_pair_kernel (grouped)", achieved, peaks, peak_src, traffic=None,
                                        ms_per_step=gemm_ms,
                                        basis="the six grouped GEMMs' FLOPs (true expert rows, no padding) over "
                                              "their summed launch durations"),
            "quant_ms_per_step": timers.total_ms("quant") / args.steps,
            "weight_refresh": {"ms": refresh_ms, "launches": 2,
                               "gbs": (2 + 1 + 1 + 2 / 32) * w_elems / (refresh_ms / 1e3) / 1e9,
                               "tflops_with_one_refresh_per_step": wl.step_flops() /
                               ((ms / args.steps + refresh_ms) / 1e3) / 1e12},
            "gpu_launches": wl.launches_per_step() * args.steps, "clocks": clk}
    if rank == 0 and not args.no_cpu_baseline:
        v, dt, n = timed_cpu_baseline(lambda i: oracle_moe_sample(256, 256, seed=11 + i), args.cpu_budget)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                                "seconds": dt, "sample": f"{n} x (largest expert of each projection: 256x256 "
                                                         "blocks of fprop, dgrad and wgrad with the oracle "
                                                         "quantisation of the rows they read)"}
    return line


def run_quant_sweep(args, rank, world, peaks, peak_src):
    """Quantiser bandwidth sweep: BF16 [M x 7168], M in {4096 .. 32768}, both
    copies in one fused pass per launch. One step = one launch per M. Each M's
    own figure comes from K launches of that M back to back (no event between
    them), after the timed region of whole steps."""
    import workloads
    import mxfp8_block_scaled_gb300 as mx
    C = 7168
    xs = {M: workloads.quant_sweep(M).cuda() for M in workloads.QUANT_SWEEP_M}
    outs = {M: mx.quantize(x, mx.MX_BOTH) for M, x in xs.items()}
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream

    def launch(M):
        x = xs[M]
        r, c = outs[M]
        mx.mx_quantize(x.data_ptr(), M, C, C, mx.MX_BOTH, r.data.data_ptr(), r.scale.data_ptr(), c.data.data_ptr(),
                       c.scale.data_ptr(), None, 0, 0, None, sp)

    def step(timers=None):
        for M in xs:
            launch(M)

    ms, _, clk = _measure(step, args, world, stream, kernel_pass=False)
    per_elem = 2 + 1 + 1 + 2 / 32
    step_bytes = sum(per_elem * M * C for M in xs)
    value = world * args.steps * step_bytes / (ms / 1e3) / 1e9
    per_m = {}
    for M in xs:
        m_ms, _, _ = _measure(lambda t, M=M: launch(M), args, world, stream, kernel_pass=False, clocks=False)
        gbs = per_elem * M * C / (m_ms / args.steps / 1e3) / 1e9
        per_m[str(M)] = {"gbs": gbs, "us_per_launch": m_ms / args.steps * 1e3, "frac": gbs / peaks["hbm_gbs"],
                         "bytes_per_launch": per_elem * M * C}
    big = max(xs)
    achieved = per_m[str(big)]["gbs"]
    line = {"metric": "MX quantiser GB/s (row + column copies, one fused pass)", "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3",
            "data": "synthetic",
            "config": {"workload": "quant_sweep BF16 [M x 7168], M in 4096/8192/16384/32768, axis both",
                       "parallelism": f"replicas{world}", "l2": "no flush: each step moves ~1.8 GB (> 129 MB L2)"},
            "per_M": per_m,
            "roofline": {"bound": "hbm", "kernel": "mx_quant_kernel", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": profile_traffic("mx_quant_kernel:quant_sweep_M32768", "bytes_per_launch"),
                         "bytes_per_launch": per_elem * big * C,
                         "peak_source": f"{peak_src} hbm_gbs", "launch": f"M={big}"},
            "frac_min_over_M": min(v["frac"] for v in per_m.values()),
            "gpu_launches": len(xs) * args.steps, "clocks": clk}
    if rank == 0 and not args.no_cpu_baseline:
        v, dt, n = timed_cpu_baseline(lambda i: oracle_quant_sample(4096, 1024, seed=i), args.cpu_budget,
                                      unit_scale=1e9)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
                                "seconds": dt, "sample": f"{n} x a [1024 x 7168] row slab of the M=4096 sweep "
                                                         "tensor: oracle row and column quantisation, 4.0625 B per "
                                                         "element"}
    return line


_SWEEP_HOST = {}


def oracle_quant_sample(M: int, rows: int = 1024, seed: int = 0):
    """Time the oracle's row and column quantisation of a slab of `rows`
    consecutive rows (a multiple of 32, so the column blocks stay whole) of the
    [M x 7168] sweep tensor; returns (algorithmic bytes, seconds)."""
    import oracle
    import workloads
    if M not in _SWEEP_HOST:
        _SWEEP_HOST.clear()
        _SWEEP_HOST[M] = workloads.quant_sweep(M)
    x = _SWEEP_HOST[M]
    r0 = (seed * rows) % M
    f = _f64(x[r0:r0 + rows])
    t0 = time.perf_counter()
    oracle.mx_quantize_rowwise(f)
    oracle.mx_quantize_colwise(f)
    dt = time.perf_counter() - t0
    return 4.0625 * f.size, dt


def _linear_set(projs, mx):
    """Device tensors and MX buffers for a list of (name, X, W, dY) Linear layers."""
    layers = []
    for name, X, W, dY in projs:
        X, W, dY = X.cuda(), W.cuda(), dY.cuda()
        xr, xc = mx.quantize(X, mx.MX_BOTH)
        wr, wc = mx.quantize(W, mx.MX_BOTH)
        dr, dc = mx.quantize(dY, mx.MX_BOTH)
        M, K = X.shape
        N = W.shape[0]
        bf = dict(dtype=torch.bfloat16, device="cuda")
        # scratch for fprop, should it split its last round (dgrad + wgrad run as
        # one launch of whole tiles)
        need = mx.mx_gemm_workspace_bytes(mx.MX_FPROP, xr.c_operand(), wr.c_operand())
        layers.append(dict(name=name, M=M, N=N, K=K, src=(X, W, dY), q=((xr, xc), (wr, wc), (dr, dc)),
                           ws=torch.empty(max(need, 16), dtype=torch.uint8, device="cuda"), ws_bytes=need,
                           out=(torch.empty((M, N), **bf), torch.empty((M, K), **bf), torch.empty((N, K), **bf))))
    return layers


def _linear_step(layers, mx, stream, timers=None):
    """Per layer: quantise X and W (one launch) and dY (both copies each); then
    fprop, and the backward pass's dgrad + wgrad in one launch."""
    sp = stream.cuda_stream
    for ly in layers:
        for names in ((0, 1), (2,)):
            descs = []
            for i in names:
                x, (r, c) = ly["src"][i], ly["q"][i]
                descs.append(mx.MXQuantTensorC(x.data_ptr(), x.shape[0], x.shape[1], x.stride(0), r.data.data_ptr(),
                                               r.scale.data_ptr(), c.data.data_ptr(), c.scale.data_ptr()))
            e = timers.span("quant", stream) if timers else None
            mx.mx_quantize_multi(descs, mx.MX_BOTH, None, sp)
            if e is not None:
                e.record(stream)
        (xr, xc), (wr, wc), (dr, dc) = ly["q"]
        y, dx, dw = ly["out"]
        e = timers.span((ly["name"], 0), stream) if timers else None
        mx.mx_gemm_with_workspace(mx.MX_FPROP, xr.c_operand(), wr.c_operand(), y.data_ptr(), y.stride(0),
                                  ly["ws"].data_ptr(), ly["ws_bytes"], None, sp)
        if e is not None:
            e.record(stream)
        e = timers.span((ly["name"], 1), stream) if timers else None
        mx.mx_gemm_multi([mx.MXGemmProblemC(dr.c_operand(), wc.c_operand(), dx.data_ptr(), dx.stride(0),
                                            mx.MX_DGRAD, 0),
                          mx.MXGemmProblemC(dc.c_operand(), xc.c_operand(), dw.data_ptr(), dw.stride(0),
                                            mx.MX_WGRAD, 0)], None, sp)
        if e is not None:
            e.record(stream)


def gemm_launches(mx, mode, a, b, workspace=False):
    """Kernel launches of one dense GEMM call: the GEMM, plus the split-tail
    reduction when a workspace is passed and the GEMM splits its last round."""
    return 1 + (1 if workspace and mx.mx_gemm_workspace_bytes(mode, a.c_operand(), b.c_operand()) > 0 else 0)


def _gemm_shapes(ly):
    """(label, M, N, K) of the three GEMMs of one Linear layer."""
    M, N, K = ly["M"], ly["N"], ly["K"]
    return (("fprop", M, N, K), ("dgrad", M, K, N), ("wgrad", N, K, M))


def _measure(step, args, world, stream, kernel_pass=True, clocks=True):
    """W warm-up steps, the timed region, then the kernel pass.

    The timed region is exactly K steps with no event inside them, bracketed
    by a barrier and a synchronize on both sides; its CUDA-event time gives
    `value` and `ms_per_step`. The kernel pass runs K more steps with a
    CUDA-event span around each kernel launch (or launch group) and gives the
    per-kernel durations of the roofline entries. Each timing event costs the
    stream about 2 us (a dense FFN step took 456 us without its six events and
    469 us with them), which is why the whole-step time comes from the pass
    without them. Clocks are sampled across both passes.
    kernel_pass=False skips the second pass; clocks=False samples no clocks.
    Returns (max-over-ranks ms of the timed region, Timers, clock record)."""
    for _ in range(args.warmup):
        step(None)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device()) if clocks else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step(None)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    timers = Timers()
    if kernel_pass:
        for _ in range(args.steps):
            step(timers)
        torch.cuda.synchronize()
        barrier(world)
    clk = sampler.stop() if sampler else None
    return max_over_ranks(t0.elapsed_time(t1), world), timers, clk


def run_mla(args, rank, world, peaks, peak_src, pages: bool = False):
    """MLA projection set at M = 16384 tokens (q_down 2048->1536, kv_down
    2048->576, kv_up 512->4096, o_proj 2048->2048; with `pages`, the frozen 16B
    configuration's own projections q_proj 2048->2048, kv_a_proj_with_mqa
    2048->3136, kv_b_proj 3072->3072, o_proj 2048->2048): per projection X and
    W quantised in one launch and dY in another, then fprop, then dgrad + wgrad
    in one launch. A GEMM's roofline time is max(FLOPs / FP8 peak, algorithmic
    bytes / HBM bandwidth); the backward launch's is the sum of its two."""
    import workloads
    import mxfp8_block_scaled_gb300 as mx
    projs = []
    table = workloads.MLA_PROJECTIONS_PAGES if pages else workloads.MLA_PROJECTIONS
    for name, _, _ in table:
        d = workloads.mla_projection(name, pages=pages)
        projs.append((name, d["X"], d["W"], d["dY"]))
    layers = _linear_set(projs, mx)
    stream = torch.cuda.Stream()
    ms, timers, clk = _measure(lambda t: _linear_step(layers, mx, stream, t), args, world, stream)
    peak_fp8, _, _ = fp8_peaks(peaks, peak_src)
    per_gemm, flops_total, gemm_ms_total = [], 0.0, 0.0

    def roof(M, N, K):
        fl = 2.0 * M * N * K
        byts = (M * K + N * K) * (1 + 1 / 32) + 2 * M * N
        return fl, max(fl / (peak_fp8 * 1e12), byts / (peaks["hbm_gbs"] * 1e9)) * 1e3, \
            "tensor" if fl / (peak_fp8 * 1e12) >= byts / (peaks["hbm_gbs"] * 1e9) else "hbm"

    for ly in layers:
        (_, M, N, K), dg, wg = _gemm_shapes(ly)
        for j, (label, shapes) in enumerate((("fprop", [(M, N, K)]), ("dgrad + wgrad (one launch)", [dg[1:], wg[1:]]))):
            parts = [roof(*sh) for sh in shapes]
            fl = sum(pt[0] for pt in parts)
            roof_ms = sum(pt[1] for pt in parts)
            g_ms = timers.total_ms((ly["name"], j)) / timers.count((ly["name"], j))
            per_gemm.append({"gemm": f"{ly['name']} {label}", "shapes": [list(sh) for sh in shapes], "ms": g_ms,
                             "tflops": fl / (g_ms / 1e3) / 1e12, "roofline_ms": roof_ms,
                             "bound": "+".join(pt[2] for pt in parts), "frac": roof_ms / g_ms})
            flops_total += fl
            gemm_ms_total += g_ms
    value = world * args.steps * flops_total / (ms / 1e3) / 1e12
    achieved = flops_total / (gemm_ms_total / 1e3) / 1e12
    line = {"metric": "MXFP8 GEMM TFLOPS (MLA projections, fprop+dgrad+wgrad incl. MX quantisation)",
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": ("mla_projections_pages_shapes M=16384: q_proj 2048->2048, kv_a_proj_with_mqa "
                                    "2048->3136, kv_b_proj 3072->3072, o_proj 2048->2048" if pages else
                                    "mla_projections M=16384: q_down 2048->1536, kv_down 2048->576, "
                                    "kv_up 512->4096, o_proj 2048->2048"), "parallelism": f"replicas{world}",
                       "l2": "no flush: a step moves ~1.5 GB (> 129 MB L2)"},
            "per_gemm": per_gemm,
            "roofline": tensor_roofline("mx_gemm_pair_kernel / mx_gemm_kernel", achieved, peaks, peak_src,
                                        traffic=None, ms_per_step=gemm_ms_total,
                                        roofline_time_frac=sum(g["roofline_ms"] for g in per_gemm) / gemm_ms_total,
                                        basis="per GEMM launch max(FLOPs / FP8 peak, algorithmic bytes / HBM); "
                                              "frac = the GEMMs' FLOPs over their summed launch durations"),
            # per layer: two quantiser launches, fprop (+ its split-tail reduction), dgrad + wgrad
            "gpu_launches": sum(2 + gemm_launches(mx, mx.MX_FPROP, ly["q"][0][0], ly["q"][1][0], workspace=True) + 1
                                for ly in layers) * args.steps,
            "clocks": clk}
    if rank == 0 and not args.no_cpu_baseline:
        def sample(i):
            fl, dt = 0.0, 0.0
            for _, X, W, dY in projs:
                f_, d_ = oracle_linear_sample(X, W, dY, 128, 128, seed=21 + i)
                fl, dt = fl + f_, dt + d_
            return fl, dt
        v, dt, n = timed_cpu_baseline(sample, args.cpu_budget)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                                "seconds": dt, "sample": f"{n} x (each projection: a 128x128 output block of its "
                                                         "fprop, dgrad and wgrad with the oracle quantisation of "
                                                         "the rows they read)"}
    return line


def run_single(args, rank, world, peaks, peak_src):
    """Single MXFP8 Linear fprop (X[256, 512], W[256, 512]): X and W quantised
    1x32 along K in one launch, then the GEMM. Launch-latency bound, so the
    line reports time per step. `value` replays the step from a CUDA graph
    (its two launches recorded once, as a serving loop would); the same step
    issued call by call through the C ABI is reported as `eager_us`."""
    import workloads
    import mxfp8_block_scaled_gb300 as mx
    d = workloads.single_linear()
    X, W = d["X"].cuda(), d["W"].cuda()
    xr, _ = mx.quantize(X, mx.MX_ROWWISE)
    wr, _ = mx.quantize(W, mx.MX_ROWWISE)
    out = torch.empty((X.shape[0], W.shape[0]), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    descs = [mx.MXQuantTensorC(x.data_ptr(), x.shape[0], x.shape[1], x.stride(0), r.data.data_ptr(),
                               r.scale.data_ptr(), None, None) for x, r in ((X, xr), (W, wr))]

    def step(timers):
        e = timers.span("quant", stream) if timers else None
        mx.mx_quantize_multi(descs, mx.MX_ROWWISE, None, sp)
        if e is not None:
            e.record(stream)
        e = timers.span("gemm", stream) if timers else None
        mx.mx_gemm(mx.MX_FPROP, xr.c_operand(), wr.c_operand(), out.data_ptr(), out.stride(0), None, sp)
        if e is not None:
            e.record(stream)

    # eager: every call through the C ABI (K steps without events, then K
    # with per-kernel spans)
    eager_ms, timers, _ = _measure(step, args, world, stream)
    eager_us = eager_ms / args.steps * 1e3
    eager_out = out.clone()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()

    # the same step recorded once into a CUDA graph and replayed; its output
    # must equal the eager step's bit for bit
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        step(None)
    with torch.cuda.stream(stream):
        out.zero_()
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager_out.view(torch.int16), out.view(torch.int16)), "graph replay differs from eager"
    barrier(world)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        g1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = max_over_ranks(g0.elapsed_time(g1), world)
    us = ms / args.steps * 1e3
    line = {"metric": "single MXFP8 Linear fprop latency (quantise X and W, GEMM)", "value": us, "unit": "us",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": "single_linear M=256 N=256 K=512, X and W quantised 1x32 along K",
                       "launch": "CUDA graph of the step's two launches, replayed; eager_us = the same step "
                                 "issued call by call", "parallelism": f"replicas{world}",
                       "l2": "inputs stay in L2 (launch-latency bound; no roofline fraction)"},
            "eager_us": eager_us,
            "per_kernel_us": {"quant_x_and_w": timers.total_ms("quant") / timers.count("quant") * 1e3,
                              "gemm": timers.total_ms("gemm") / timers.count("gemm") * 1e3},
            "gpu_launches": (1 + gemm_launches(mx, mx.MX_FPROP, xr, wr)) * args.steps, "clocks": clk}
    gemm_us = line["per_kernel_us"]["gemm"]
    fl = 2.0 * X.shape[0] * W.shape[0] * X.shape[1]
    line["roofline"] = tensor_roofline("mx_gemm_kernel", fl / (gemm_us / 1e6) / 1e12, peaks, peak_src,
                                       traffic=None, note="launch-latency bound: 6.7e7 FLOP take ~0.02 us at the "
                                                          "tensor peak, so the fraction says nothing about the "
                                                          "kernel; the time per step is the figure")
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        fx, fw = _f64(d["X"]), _f64(d["W"])

        def sample(i):
            t0 = time.perf_counter()
            oracle.mx_gemm_ref(*oracle.mx_quantize_rowwise(fx), *oracle.mx_quantize_rowwise(fw))
            return 1.0, time.perf_counter() - t0
        n_per_s, dt, n = timed_cpu_baseline(sample, min(args.cpu_budget, 3.0), unit_scale=1.0)
        line["cpu_baseline"] = {"value": 1e6 / n_per_s, "unit": "us", "cores": cpu_threads(), "kind": "oracle",
                                "seconds": dt, "sample": f"{n} x the whole step: oracle 1x32 quantisation of X "
                                                         "and W and the full 256x256x512 GEMM"}
    return line


def run_wrefresh(args, rank, world, peaks, peak_src):
    """Weight refresh after an optimizer step: the routed experts' FP32 masters
    (gate_up [64, 2816, 2048] and down [64, 2048, 1408]) quantised into row and
    column copies, one launch per projection."""
    import workloads
    import mxfp8_block_scaled_gb300 as mx
    masters = [workloads.fp32_master(s, seed=workloads.SEED_BASE + 6 + i).cuda()
               for i, s in enumerate(((64, 2816, 2048), (64, 2048, 1408)))]
    outs = [mx.quantize_stacked(w, mx.MX_BOTH) for w in masters]
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream

    def step(timers):
        for i, (w, (r, c)) in enumerate(zip(masters, outs)):
            E, N, K = w.shape
            e = timers.span(i, stream) if timers else None
            mx.mx_quantize_f32(w.data_ptr(), E, N, K, K, N * K, mx.MX_BOTH, r.data.data_ptr(), r.scale.data_ptr(),
                               c.data.data_ptr(), c.scale.data_ptr(), None, sp)
            if e is not None:
                e.record(stream)

    ms, timers, clk = _measure(step, args, world, stream)
    per_elem = 4 + 1 + 1 + 2 / 32
    nbytes = [per_elem * w.numel() for w in masters]
    value = world * args.steps * sum(nbytes) / (ms / 1e3) / 1e9
    per = {f"{tuple(w.shape)}": nb / (timers.total_ms(i) / timers.count(i) / 1e3) / 1e9
           for i, (w, nb) in enumerate(zip(masters, nbytes))}
    achieved = max(per.values())
    line = {"metric": "MX weight refresh GB/s (FP32 master -> row + column copies, one fused pass)", "value": value,
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32->e4m3",
            "data": "synthetic",
            "config": {"workload": "expert weight refresh: FP32 [64,2816,2048] + [64,2048,1408], axis both",
                       "parallelism": f"replicas{world}", "l2": "no flush: a step moves ~3.8 GB (> 129 MB L2)"},
            "per_projection_gbs": per,
            "roofline": {"bound": "hbm", "kernel": "mx_quant_f32_kernel", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": profile_traffic("mx_quant_f32_kernel:gate_up", "bytes_per_launch"),
                         "bytes_per_launch": max(nbytes), "peak_source": f"{peak_src} hbm_gbs"},
            "gpu_launches": 2 * args.steps, "clocks": clk}
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        w0 = masters[1][0].cpu().numpy().astype(np.float64)   # one down expert [2048, 1408], exact FP32 values

        def sample(i):
            t0 = time.perf_counter()
            oracle.mx_quantize_rowwise(w0)
            oracle.mx_quantize_colwise(w0)
            return per_elem * w0.size, time.perf_counter() - t0
        v, dt, n = timed_cpu_baseline(sample, args.cpu_budget, unit_scale=1e9)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
                                "seconds": dt, "sample": f"{n} x one expert's FP32 master [2048 x 1408]: oracle row "
                                                         "and column quantisation, 6.0625 B per element"}
    return line


def run_blockwise(args, rank, world, peaks, peak_src):
    """Variant recipe: the dense FFN up-projection fprop (8192 x 10944 x 2048)
    with DeepSeek-V3 blockwise FP8 (1 x 128 activation blocks, 128 x 128 weight
    blocks, FP32 multipliers); a step quantises X and W and runs the GEMM."""
    import mxfp8_block_scaled_gb300 as mx
    d = dense_host_inputs()
    X, W = d["X"].cuda(), d["W"].cuda()
    M, K = X.shape
    N = W.shape[0]
    qa, qb = mx.quantize_fp8_blockwise(X, 1), mx.quantize_fp8_blockwise(W, 128)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream

    def step(timers):
        for x, q, blk in ((X, qa, 1), (W, qb, 128)):
            e = timers.span("quant", stream) if timers else None
            mx.mx_quantize_fp8_blockwise(x.data_ptr(), x.shape[0], x.shape[1], x.stride(0), blk, q.data.data_ptr(),
                                         q.scale.data_ptr(), None, sp)
            if e is not None:
                e.record(stream)
        e = timers.span("gemm", stream) if timers else None
        mx.mx_gemm_fp8_blockwise(qa.data.data_ptr(), qa.scale.data_ptr(), M, qb.data.data_ptr(), qb.scale.data_ptr(),
                                 N, K, out.data_ptr(), out.stride(0), None, sp)
        if e is not None:
            e.record(stream)

    ms, timers, clk = _measure(step, args, world, stream)
    fl = 2.0 * M * N * K
    gemm_ms = timers.total_ms("gemm") / timers.count("gemm")
    achieved = fl / (gemm_ms / 1e3) / 1e12
    line = {"metric": "FP8 blockwise GEMM TFLOPS (DeepSeek-V3 1x128 / 128x128 recipe, fprop incl. quantisation)",
            "value": world * args.steps * fl / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": "dense_ffn_up_proj fprop M=8192 K=2048 N=10944, blockwise FP8 variant",
                       "parallelism": f"replicas{world}", "l2": "no flush: a step moves ~0.3 GB (> 129 MB L2)"},
            "roofline": tensor_roofline("mx_gemm_blockwise_kernel", achieved, peaks, peak_src,
                                        traffic=profile_traffic("mx_gemm_blockwise_kernel"), avg_launch_ms=gemm_ms),
            "quant_ms_per_launch": timers.total_ms("quant") / timers.count("quant"),
            "gpu_launches": 3 * args.steps, "clocks": clk}
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        xs, ws = _f64(d["X"][:256]), _f64(d["W"][:256])

        def sample(i):
            t0 = time.perf_counter()
            qa_, sa_ = oracle.quantize_1x128(xs)
            qb_, sb_ = oracle.quantize_128x128(ws)
            oracle.gemm_blockwise_ref(qa_, sa_, qb_, sb_)
            return 2.0 * 256 * 256 * K, time.perf_counter() - t0
        v, dt, n = timed_cpu_baseline(sample, args.cpu_budget)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                                "seconds": dt, "sample": f"{n} x (256 rows of X quantised 1x128, the first 256 rows "
                                                         "of W in 128x128 blocks, their 256x256x2048 blockwise GEMM)"}
    return line


def run_current(args, rank, world, peaks, peak_src):
    """Variant recipe: the dense FFN up-projection step with current scaling
    (one FP32 scale per tensor from its amax, E4M3 data): per tensor an amax
    launch and a quantisation launch (row + transposed copy), then fprop, and
    dgrad + wgrad in one launch, on the 256 x 256 pair kernel with two
    accumulators and the two scales applied in the epilogue."""
    import mxfp8_block_scaled_gb300 as mx
    d = dense_host_inputs()
    src = {k: d[k].cuda() for k in ("X", "W", "dY")}
    M, K = src["X"].shape
    N = src["W"].shape[0]
    amax = {k: torch.empty(1, dtype=torch.float32, device="cuda") for k in src}
    q = {k: mx.quantize_current(v, mx.MX_BOTH, amax=mx.current_amax(v)) for k, v in src.items()}
    outs = [torch.empty(sh, dtype=torch.bfloat16, device="cuda") for sh in ((M, N), (M, K), (N, K))]
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream

    def step(timers):
        for k, x in src.items():
            r, c = q[k]
            e = timers.span("quant", stream) if timers else None
            mx.mx_current_amax(x.data_ptr(), 1, x.shape[0], x.shape[1], x.stride(0), 0, amax[k].data_ptr(), None, sp)
            mx.mx_quantize_current(x.data_ptr(), 1, x.shape[0], x.shape[1], x.stride(0), 0, mx.MX_BOTH,
                                   amax[k].data_ptr(), mx.CURRENT_FORMAT_MAX, r.data.data_ptr(), c.data.data_ptr(),
                                   r.scale.data_ptr(), None, 0, 0, None, sp)
            if e is not None:
                e.record(stream)
        (xr, xc), (wr, wc), (dr, dc) = q["X"], q["W"], q["dY"]
        e = timers.span("gemm", stream) if timers else None
        mx.mx_gemm_current(mx.MX_FPROP, xr.c_operand(), wr.c_operand(), outs[0].data_ptr(), outs[0].stride(0),
                           None, sp)
        if e is not None:
            e.record(stream)
        e = timers.span("gemm", stream) if timers else None
        mx.mx_gemm_current_multi([mx.MXGemmProblemC(dr.c_operand(), wc.c_operand(), outs[1].data_ptr(),
                                                    outs[1].stride(0), mx.MX_DGRAD, 0),
                                  mx.MXGemmProblemC(dc.c_operand(), xc.c_operand(), outs[2].data_ptr(),
                                                    outs[2].stride(0), mx.MX_WGRAD, 0)], None, sp)
        if e is not None:
            e.record(stream)

    ms, timers, clk = _measure(step, args, world, stream)
    fl = 3 * 2.0 * M * N * K
    gemm_ms = timers.total_ms("gemm") / args.steps
    quant_ms = timers.total_ms("quant") / args.steps
    # amax pass: 2 B read per element; quantisation: 2 B read + 2 x 1 B written
    qbytes = sum((2 + 2 + 1 + 1) * x.numel() for x in src.values())
    line = {"metric": "MXFP8-path GEMM TFLOPS with current scaling (one FP32 scale per tensor; fprop+dgrad+wgrad "
                      "step incl. amax and quantisation, dense FFN up-proj)",
            "value": world * args.steps * fl / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": "dense_ffn_up_proj M=8192 K=2048 N=10944, current-scaling variant",
                       "parallelism": f"replicas{world}", "l2": "no flush: a step moves ~1 GB (> 129 MB L2)"},
            "roofline": tensor_roofline("mx_gemm_pair_kernel (tensor-scaled)", fl / (gemm_ms / 1e3) / 1e12, peaks,
                                        peak_src, traffic=None, ms_per_step=gemm_ms),
            "quant_roofline": {"bound": "hbm", "kernel": "cur_amax_kernel + mx_quant_kernel (current)",
                               "achieved": qbytes / (quant_ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": qbytes / (quant_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                               "bytes_per_step": qbytes, "ms_per_step": quant_ms,
                               "basis": "amax pass 2 B/element + quantisation 4 B/element over the six launches"},
            "gpu_launches": 8 * args.steps, "clocks": clk}
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        g = np.random.Generator(np.random.Philox(5))
        rows = {k: np.sort(g.choice(v.shape[0], 256, replace=False)) for k, v in d.items() if k in ("X", "W")}

        def sample(i):
            fx, fw = _f64(d["X"][torch.from_numpy(rows["X"])]), _f64(d["W"][torch.from_numpy(rows["W"])])
            t0 = time.perf_counter()
            cx, sx, _ = oracle.current_quantize(fx)
            cw, sw, _ = oracle.current_quantize(fw)
            oracle.current_gemm_ref(cx, sx, cw, sw)
            return 2.0 * 256 * 256 * K, time.perf_counter() - t0
        v, dt, n = timed_cpu_baseline(sample, args.cpu_budget)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                                "seconds": dt, "sample": f"{n} x (256 rows of X and of W quantised with their own "
                                                         "current scale, their 256x256x2048 GEMM)"}
    return line


def run_dense(args, rank, world, peaks, peak_src):
    """The headline: the dense FFN up-projection step (quantise X + W, dY;
    fprop; dgrad + wgrad in one launch), plus its end-to-end run from pinned
    host buffers."""
    wl = DenseFFN()
    stream = torch.cuda.Stream()

    # --- timed region: exactly K steps (then K more with per-kernel spans) ---
    ms_max, timers, clk = _measure(lambda t: wl.step(stream, t), args, world, stream)
    value = world * args.steps * wl.step_flops() / (ms_max / 1e3) / 1e12

    gemm_ms = timers.total_ms("gemm") / args.steps            # fprop + the fused dgrad/wgrad launch
    achieved = wl.step_flops() / (gemm_ms / 1e3) / 1e12
    qb = wl.quant_bytes()
    q_launch = {}                                              # each quantiser launch of a step on its own
    for names in (("X", "W"), ("dY",)):
        key = "+".join(names)
        l_ms = timers.total_ms(("quant", key)) / args.steps
        l_bytes = sum(qb[k] for k in names)
        q_launch[key] = {"ms": l_ms, "bytes": l_bytes, "gbs": l_bytes / (l_ms / 1e3) / 1e9,
                         "frac": l_bytes / (l_ms / 1e3) / 1e9 / peaks["hbm_gbs"]}
    quant_ms = sum(v["ms"] for v in q_launch.values())        # both quantiser launches of a step
    qbytes = sum(qb.values())                                  # X, W and dY per step
    q_gbs = qbytes / (quant_ms / 1e3) / 1e9

    # --- end to end: pinned host inputs -> device -> step -> host outputs ---
    e2e_value = None
    if args.e2e_steps > 0:
        wl.run_e2e(stream, 3)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        wl.run_e2e(stream, args.e2e_steps)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
        e2e_value = world * args.e2e_steps * wl.step_flops() / (e2e_ms / 1e3) / 1e12

    line = {
        "metric": METRIC_DENSE,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": WORKLOAD_DENSE, "M": wl.M, "K": wl.K, "N": wl.N,
                   "parallelism": f"replicas{world}",
                   "l2": "no flush: a step reads/writes ~0.7 GB (> 129 MB L2)"},
        "roofline": tensor_roofline("mx_gemm_pair_kernel", achieved, peaks, peak_src,
                                    traffic=profile_traffic("mx_gemm_pair_kernel"),
                                    flops_per_step=wl.step_flops(), ms_per_step=gemm_ms, launches_per_step=2,
                                    basis="fprop, dgrad and wgrad FLOPs (2MNK each) over the summed duration of "
                                          "the step's two GEMM launches (fprop; dgrad + wgrad in one launch)"),
        "quant_roofline": {"bound": "hbm", "kernel": "mx_quant_kernel", "achieved": q_gbs,
                           "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": q_gbs / peaks["hbm_gbs"],
                           "traffic": profile_traffic("mx_quant_kernel"), "bytes_per_step": qbytes,
                           "ms_per_step": quant_ms, "launches_per_step": 2, "per_launch": q_launch,
                           "basis": "algorithmic bytes of X, W and dY over the summed duration of the step's two "
                                    "quantiser launches (X+W in one, dY in the other; each apart in per_launch)",
                           "peak_source": f"{peak_src} hbm_gbs"},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": wl.h2d_bytes(),
                "d2h_bytes_per_step": wl.d2h_bytes(), "steps": args.e2e_steps,
                "overlap": "step i+1's inputs copy in and step i-1's outputs copy out while step i computes "
                           "(two copy streams, two device buffer slots)"},
        "gpu_launches": wl.launches_per_step() * args.steps,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        v, dt, n = timed_cpu_baseline(lambda i: oracle_dense_sample(1024, 1024, seed=7 + i), args.cpu_budget)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cpu_threads(),
                                "kind": "oracle", "seconds": dt,
                                "sample": f"{n} x (1024x1024 output block of fprop, dgrad and wgrad of the dense FFN "
                                          "up-proj, with the oracle quantisation of the operand rows it reads)"}
    del wl
    return line


def run_mla_pages(args, rank, world, peaks, peak_src):
    return run_mla(args, rank, world, peaks, peak_src, pages=True)


RUNS = {"dense_ffn": run_dense, "single": run_single, "mla": run_mla, "mla_pages": run_mla_pages, "moe": run_moe,
        "quant": run_quant_sweep, "wrefresh": run_wrefresh, "blockwise": run_blockwise, "current": run_current}
# Sub-results of the default line, keyed by the workload they measure.
SUB_CONFIGS = (("config1_single_linear", "single"), ("config3_mla_projections", "mla"),
               ("config3b_mla_projections_pages_shapes", "mla_pages"),
               ("config4_moe_routed_experts", "moe"), ("config5_quant_sweep", "quant"),
               ("variant_blockwise_fp8", "blockwise"), ("variant_current_scaling", "current"),
               ("weight_refresh_fp32_master", "wrefresh"))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all", choices=["all"] + list(RUNS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=5.0,
                    help="seconds of oracle work behind each cpu_baseline")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import mxfp8_block_scaled_gb300 as mx
    mx.lib()
    peaks, peak_src = load_peaks()
    if args.workload != "all":
        line = RUNS[args.workload](args, rank, world, peaks, peak_src)
    else:
        # the headline (dense FFN step, BASELINE's metric and config) carrying
        # every other configuration's own measurement as a sub-result
        line = run_dense(args, rank, world, peaks, peak_src)
        line["configs"] = {}
        for key, wl_name in SUB_CONFIGS:
            torch.cuda.empty_cache()
            sub = RUNS[wl_name](args, rank, world, peaks, peak_src)
            for k in ("n_gpus", "steps", "warmup", "scaling", "vs_baseline", "data"):
                sub.pop(k, None)
            line["configs"][key] = sub
    if rank == 0:
        line["timing"] = TIMING_NOTE
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
