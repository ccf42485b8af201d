"""Benchmark of the Q4_0 quantized linear layer on GB300.

Headline workload: the decode GEMV of a 4B-class FFN up-projection,
m = 1 token, n = 9728 output rows, k = 2560 inputs, W in Q4_0 (14,008,320
bytes of blocks). One step is one q4_0_matmul call on fresh weights: the
step cycles through enough distinct packed copies of W that their total is
more than twice the 129 MB L2, so every step reads its weights from HBM.
Steps run as CUDA-graph replays; the timed region is bracketed by CUDA
events on the launching stream with a synchronize on both sides.

Printed: one JSON line (rank 0). `value` is weight GB/s over all ranks;
`roofline` compares the decode kernel with the measured HBM copy bandwidth;
`e2e` is the same metric through the public API with pinned host buffers
and the per-step host<->device copies inside the timed region;
`cpu_baseline` times the CPU oracle on the host cores on a bounded sample;
`sweep` reports the other workload shapes (parity-tested elsewhere).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                  [--no-sweep] [--no-cpu]

With --gpus N > 1 (torchrun) every rank runs an independent replica of the
workload on its own GPU (the layer has no exchange step); the time is the
maximum over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Q4_0 weight GB/s (% HBM peak) at m=1..16; prefill TFLOP/s (% bf16 peak)"
L2_BYTES = 129 * 1024 * 1024
SLEEP_CYCLES = 200_000          # about 0.1 ms of device time before a timed region
NOMINAL_HBM_GBS = 7900.0        # GB300 spec sheet: HBM3e bandwidth
NOMINAL_BF16_TFLOPS = 2250.0    # GB300 spec sheet: dense bf16 tensor-core peak
HEADLINE = dict(name="decode GEMV, FFN up-projection", m=1, n=9728, k=2560)
WORKLOADS = {
    "decode": HEADLINE,
    "gemv1k": dict(name="single GEMV", m=1, n=1024, k=1024),
    "slots4-up": dict(name="4 slots, up-projection", m=4, n=9728, k=2560),
    "slots4-down": dict(name="4 slots, down-projection", m=4, n=2560, k=9728),
    **{f"sweep-m{m}": dict(name="slot sweep 14336x4096", m=m, n=14336, k=4096) for m in (1, 2, 4, 8, 16)},
    "logit": dict(name="logit head", m=4, n=151936, k=2560),
    "prefill": dict(name="prefill", m=540, n=9728, k=2560),
    # the variants (for profiles): integer-dot X, per-channel int8 weights
    "w4a8-decode": dict(name="W4A8 decode up-projection", m=1, n=9728, k=2560, w4a8=True),
    "w8-decode": dict(name="int8-weight decode up-projection", m=1, n=9728, k=2560, w8=True),
}
SWEEP = [
    dict(name="single GEMV", m=1, n=1024, k=1024),
    dict(name="decode up-projection", m=1, n=9728, k=2560),
    dict(name="4 slots, up-projection", m=4, n=9728, k=2560),
    dict(name="4 slots, down-projection", m=4, n=2560, k=9728),
    dict(name="slot sweep 14336x4096", m=1, n=14336, k=4096),
    dict(name="slot sweep 14336x4096", m=2, n=14336, k=4096),
    dict(name="slot sweep 14336x4096", m=4, n=14336, k=4096),
    dict(name="slot sweep 14336x4096", m=8, n=14336, k=4096),
    dict(name="slot sweep 14336x4096", m=16, n=14336, k=4096),
    dict(name="logit head", m=4, n=151936, k=2560),
    dict(name="prefill", m=540, n=9728, k=2560),
    # prefill of a down-projection: 20 row groups, K split across clusters
    dict(name="prefill, down-projection (K split)", m=540, n=2560, k=9728),
    # the integer-dot variant (q4_0_matmul_w4a8): X coded to int8 per block
    dict(name="W4A8 decode up-projection", m=1, n=9728, k=2560, w4a8=True),
    dict(name="W4A8 slot sweep 14336x4096", m=8, n=14336, k=4096, w4a8=True),
    dict(name="W4A8 slot sweep 14336x4096", m=16, n=14336, k=4096, w4a8=True),
    # per-output-channel int8 weights (q4_w8_matmul): n x k int8 codes plus
    # n fp32 scales per call
    dict(name="int8-weight decode up-projection", m=1, n=9728, k=2560, w8=True),
    dict(name="int8-weight 4 slots, up-projection", m=4, n=9728, k=2560, w8=True),
    dict(name="int8-weight slot sweep 14336x4096", m=16, n=14336, k=4096, w8=True),
    # a mixture layer (q4_0_matmul_experts): 8 experts of 9728 x 2560 with
    # 1..16 token rows each, one launch; weight bytes of all 8 experts
    dict(name="8 experts x 9728x2560, mixed group sizes", m=40, n=9728, k=2560,
         experts=[1, 3, 2, 5, 1, 4, 8, 16]),
]

# Token rows at which one expert's layer is better served by the tensor-core
# GEMM than by the mat-vec (in calls of at most 16 rows): both timed at each m.
CROSSOVER = dict(n=9728, k=2560, ms=[8, 16, 17, 24, 32, 48, 64, 96])


def weight_bytes(n, k):
    return n * (k // 32) * 18


def w8_weight_bytes(n, k):
    """Bytes a call on per-output-channel int8 weights reads: codes and scales."""
    return n * k + 4 * n


def sweep_weight_bytes(cfg):
    n, k = cfg["n"], cfg["k"]
    if cfg.get("w8"):
        return w8_weight_bytes(n, k)
    if cfg.get("experts"):
        return len(cfg["experts"]) * weight_bytes(n, k)
    return weight_bytes(n, k)


def decode_kernel_name(m, n=0, sm_count=152):
    """The kernel the library's automatic dispatch runs for m token rows."""
    if m > 16:
        return "gemm_kernel (q4mm_prefill.cu, after xcast_kernel)"
    if m <= 4:
        return "matvec_kernel (q4mm_matvec.cu, whole records per warp, exact block sums on the warp-level MMA)"
    return "matvec_kernel (q4mm_matvec.cu, half records per warp, X as one fp16 term per element)"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


_COMMENT = re.compile(r"/\*.*?\*/|//[^\n]*", re.S)


def source_code_hash(texts):
    """Hash of (file name, code) pairs with comments and blank space removed,
    so that a profile taken on the same code stays valid across comment
    edits."""
    h = hashlib.sha256()
    for name, text in sorted(texts):
        code = " ".join(_COMMENT.sub(" ", text).split())
        h.update(name.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


# host-only sources (no kernels, no plans): excluded from the kernel hash
HOST_ONLY_SOURCES = {"q4mm_gguf.cu", "q4mm_experts.cu"}


def kernel_source_hash():
    csrc = os.path.join(ROOT, "q4_quantized_linear_gb300", "csrc")
    texts = []
    for name in os.listdir(csrc):
        if name in HOST_ONLY_SOURCES:
            continue
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            texts.append((name, f.read()))
    return source_code_hash(texts)


def profiled_traffic(kind):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kind}.md")
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    mh = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    mt = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not mh or not mt or mh.group(1) != kernel_source_hash():
        return None
    return float(mt.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ GPU --

class Workload:
    """Packed weight copies, X and Y resident on the GPU for one shape."""

    def __init__(self, q4lib, m, n, k, min_copies=1, w4a8=False, w8=False, experts=None, chunk=0):
        """w4a8: the integer-dot call; w8: per-output-channel int8 weights
        (fp32 N(0, 1) * 0.02 weights quantised on the GPU); experts: token
        rows per expert (one weight set per expert, rows in expert order);
        chunk: run the m rows as calls of at most `chunk` rows."""
        import torch
        from q4_quantized_linear_gb300 import synth
        self.m, self.n, self.k = m, n, k
        self.w4a8, self.w8, self.chunk = w4a8, w8, chunk
        self.experts = list(experts) if experts else None
        self.blocks = synth.q4_0_blocks(n, k, seed=0)
        self.X = synth.activations(m, k, seed=0)
        per_set = len(self.experts) if self.experts else 1
        wb = (w8_weight_bytes(n, k) if w8 else weight_bytes(n, k)) * per_set
        self.copies = max(min_copies, -(-2 * L2_BYTES // wb) + 1)
        if w8:
            Wf = torch.from_numpy(synth.activations(n, k, seed=5)).cuda() * 0.02
            base = torch.empty(q4lib.q4_w8_packed_size(n, k), dtype=torch.uint8, device="cuda")
            q4lib.q4_w8_quantize(base, Wf, n, k)
            del Wf
        else:
            dev_blocks = torch.from_numpy(self.blocks.reshape(-1)).cuda()
            base = torch.empty(q4lib.q4_0_packed_size(n, k), dtype=torch.uint8, device="cuda")
            q4lib.q4_0_pack(base, dev_blocks, n, k)
            del dev_blocks
        self.W = [base] + [base.clone() for _ in range(self.copies * per_set - 1)]
        if self.experts:
            self.offsets = [0]
            for c in self.experts:
                self.offsets.append(self.offsets[-1] + c)
            assert self.offsets[-1] == m
        self.Xd = torch.from_numpy(self.X).cuda()
        self.Yd = torch.empty((m, n), dtype=torch.float32, device="cuda")
        self.ws, self.wsb = q4lib.workspace_for(m, k, n)
        torch.cuda.synchronize()

    def step(self, q4lib, i, stream):
        c = i % self.copies
        if self.experts:
            E = len(self.experts)
            q4lib.q4_0_matmul_experts(self.W[c * E:(c + 1) * E], self.offsets, self.Xd, self.Yd, self.k, self.n,
                                      stream)
        elif self.w8:
            q4lib.q4_w8_matmul(self.W[c], self.Xd, self.Yd, self.m, self.k, self.n, stream)
        elif self.w4a8:
            q4lib.q4_0_matmul_w4a8(self.W[c], self.Xd, self.Yd, self.m, self.k, self.n, stream)
        elif self.chunk:
            for r0 in range(0, self.m, self.chunk):
                r = min(self.chunk, self.m - r0)
                q4lib.q4_0_matmul_ws(self.W[c], self.Xd[r0:], self.Yd[r0:], r, self.k, self.n,
                                     self.ws, self.wsb, stream)
        else:
            q4lib.q4_0_matmul_ws(self.W[c], self.Xd, self.Yd, self.m, self.k, self.n,
                                 self.ws, self.wsb, stream)


def reduce_max(value):
    """Max of a float over the ranks of the default process group (NCCL on
    the GPU, gloo on the host); the value itself without one."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, steps, units_per_step, slowest_sec):
    """Units all ranks processed, divided by the slowest rank's time."""
    return world * steps * units_per_step / slowest_sec


def time_graph(q4lib, wl, steps, warmup, stream, per_graph=1000, sampler=None, barrier=None):
    """Run `warmup` then time exactly `steps` steps as CUDA-graph replays,
    bracketed by `barrier` (all ranks) and a device synchronize on both
    sides. Returns elapsed seconds of the timed steps."""
    import torch
    per_graph = max(1, min(per_graph, steps))
    per_graph -= per_graph % wl.copies if per_graph >= wl.copies else 0
    per_graph = max(per_graph, 1)

    def capture(count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(count):
                    wl.step(q4lib, i, stream.cuda_stream)
        return g

    with torch.cuda.stream(stream):
        for i in range(max(warmup, 1)):
            wl.step(q4lib, i, stream.cuda_stream)
    torch.cuda.synchronize()
    g_full = capture(per_graph)
    rest = steps % per_graph
    g_rest = capture(rest) if rest else None
    with torch.cuda.stream(stream):
        g_full.replay()
    torch.cuda.synchronize()

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.start()
        time.sleep(0.3)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        # a device-side pause first, so that the graphs are queued before the
        # start event runs: the timed region holds the steps, not the host's
        # launch of the first graph
        torch.cuda._sleep(SLEEP_CYCLES)
        start.record(stream)
        for _ in range(steps // per_graph):
            g_full.replay()
        if g_rest is not None:
            g_rest.replay()
        end.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    clocks = sampler.stop() if sampler else None
    return start.elapsed_time(end) / 1e3, clocks


def time_e2e(q4lib, wl, steps, stream, per_graph=200):
    """Public API with pinned host buffers: every step copies its X host ->
    device, calls the layer and copies its Y device -> host, all inside the
    timed region (captured as CUDA graphs of up to per_graph steps, like the
    device-side timing). Consecutive steps use two device buffer pairs and
    overlap: step i's input copy runs on a copy-in stream while step i - 1
    computes, its output copy on a copy-out stream while step i + 1 computes
    (events order each buffer's writer after its last reader)."""
    import torch
    Xh = [torch.from_numpy(wl.X).pin_memory() for _ in range(2)]
    Yh = [torch.empty((wl.m, wl.n), dtype=torch.float32).pin_memory() for _ in range(2)]
    Xd = [wl.Xd, wl.Xd.clone()]
    Yd = [wl.Yd, torch.empty_like(wl.Yd)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    saved = (wl.Xd, wl.Yd)

    def steps_on(count):
        ev_in = [torch.cuda.Event() for _ in range(count)]
        ev_k = [torch.cuda.Event() for _ in range(count)]
        ev_out = [torch.cuda.Event() for _ in range(count)]
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(count):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_k[i - 2])          # step i - 2's kernel has read Xd[b]
                Xd[b].copy_(Xh[b], non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])          # step i - 2's Y has left Yd[b]
            wl.Xd, wl.Yd = Xd[b], Yd[b]
            wl.step(q4lib, i, stream.cuda_stream)
            ev_k[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_k[i])
                Yh[b].copy_(Yd[b], non_blocking=True)
                ev_out[i].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    per_graph = max(1, min(per_graph, steps))
    try:
        with torch.cuda.stream(stream):
            steps_on(3)
        torch.cuda.synchronize()
        graphs = {}

        def graph(count):
            if count not in graphs:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.stream(stream):
                    with torch.cuda.graph(g, stream=stream):
                        steps_on(count)
                graphs[count] = g
            return graphs[count]

        g_full = graph(per_graph)
        rest = steps % per_graph
        g_rest = graph(rest) if rest else None
        with torch.cuda.stream(stream):
            g_full.replay()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(SLEEP_CYCLES)
            start.record(stream)
            for _ in range(steps // per_graph):
                g_full.replay()
            if g_rest is not None:
                g_rest.replay()
            end.record(stream)
        torch.cuda.synchronize()
    finally:
        wl.Xd, wl.Yd = saved
    return start.elapsed_time(end) / 1e3, Xh[0].numel() * 4, Yh[0].numel() * 4


def time_single(q4lib, wl, stream, trials=50):
    """Device-side latency of one isolated call: no kernel of the library
    before or after it, CUDA events around it on its stream, the call
    queued behind a device-side pause so that the host's launch is not
    timed; the median over trials."""
    import torch
    out = []
    for i in range(trials + 3):
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(SLEEP_CYCLES)
            start.record(stream)
            wl.step(q4lib, i, stream.cuda_stream)
            end.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            out.append(start.elapsed_time(end) * 1e3)
    return statistics.median(out)


def run_sweep(q4lib, stream, peaks):
    import torch
    out = []
    for cfg in SWEEP:
        m, n, k = cfg["m"], cfg["n"], cfg["k"]
        wl = Workload(q4lib, m, n, k, w4a8=cfg.get("w4a8", False), w8=cfg.get("w8", False),
                      experts=cfg.get("experts"))
        wb = sweep_weight_bytes(cfg)
        decode = m <= 16 or bool(cfg.get("experts"))
        est = wb / (peaks["hbm_gbs"] * 1e9) if decode else 2.0 * m * n * k / (peaks["bf16_tflops"] * 1e12)
        steps = int(min(20000, max(200, 0.25 / max(est, 1e-7))))
        steps -= steps % wl.copies
        steps = max(steps, wl.copies)
        sec, _ = time_graph(q4lib, wl, steps, 20, stream)
        t = sec / steps
        rec = dict(cfg, steps=steps, weight_copies=wl.copies, us_per_call=t * 1e6,
                   weight_gbs=wb / t / 1e9, tokens_per_s=m / t)
        if n * k <= 1 << 20:
            # a layer this small is a latency case: one isolated call as well
            rec["single_call_latency_us"] = time_single(q4lib, wl, stream)
        if decode:
            rec["frac_hbm"] = rec["weight_gbs"] / peaks["hbm_gbs"]
            rec["frac_hbm_nominal"] = rec["weight_gbs"] / NOMINAL_HBM_GBS
        else:
            rec["tflops"] = 2.0 * m * n * k / t / 1e12
            rec["frac_bf16"] = rec["tflops"] / peaks["bf16_tflops"]
            rec["frac_bf16_nominal"] = rec["tflops"] / NOMINAL_BF16_TFLOPS
        out.append(rec)
        del wl
        torch.cuda.empty_cache()
    return out


def run_crossover(q4lib, stream):
    """One expert's layer at m token rows: the library's own dispatch (the
    mat-vec up to 16 rows, the tensor-core GEMM above) against the mat-vec
    in calls of at most 16 rows. Microseconds per layer."""
    import torch
    n, k = CROSSOVER["n"], CROSSOVER["k"]
    out = []
    for m in CROSSOVER["ms"]:
        rec = dict(m=m, n=n, k=k)
        for key, chunk in (("dispatch_us", 0), ("matvec_chunks_us", 16)):
            if chunk and m <= 16:
                continue
            wl = Workload(q4lib, m, n, k, chunk=chunk)
            steps = 2000 - 2000 % wl.copies
            sec, _ = time_graph(q4lib, wl, steps, 20, stream)
            rec[key] = sec / steps * 1e6
            del wl
            torch.cuda.empty_cache()
        out.append(rec)
    return out


def cpu_baseline(cfg, gpu_Y=None, tensor=False, run_seconds=1.5):
    """The oracle (fp64, fixed order) timed on the host cores: single-threaded
    and on every thread it may use, the median of three runs each, each run a
    bounded sample (repeated calls on the leading rows of W for about
    run_seconds). With the GPU result given, also its max error over
    tolerance against the oracle on the rows the oracle computed."""
    import oracle
    from q4_quantized_linear_gb300 import synth
    m, n, k = cfg["m"], cfg["n"], cfg["k"]
    oracle.build()
    blocks = synth.q4_0_blocks(n, k, seed=0)
    X = synth.activations(m, k, seed=0)

    def rate(rows, reps, el):
        if tensor:
            return reps * 2.0 * m * rows * k / el / 1e12
        return reps * weight_bytes(rows, k) / el / 1e9

    def runs(rows, nthreads):
        vals, last = [], None
        for _ in range(3):
            reps, t0 = 0, time.perf_counter()
            while True:
                last = oracle.matmul(blocks[:rows], X, rows, k, nthreads=nthreads)
                reps += 1
                el = time.perf_counter() - t0
                if el >= run_seconds:
                    break
            vals.append(rate(rows, reps, el))
        return statistics.median(vals), last

    # the sample: leading rows of W, at most what one run covers in a second
    # (all threads) or a tenth of that (one thread)
    rows_all = n if m * n * k <= 2e9 else max(64, int(2e9 / (m * k)) // 64 * 64)
    rows_one = max(64, min(rows_all, int(2e8 / (m * k)) // 64 * 64))
    v_all, (Yr, B) = runs(rows_all, 0)
    v_one, _ = runs(rows_one, 1)
    unit = "TFLOP/s" if tensor else "GB/s"
    try:
        affinity = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        affinity = None
    res = {"value": v_all, "unit": unit, "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"median of 3 runs of about {run_seconds} s each: repeated oracle calls (fp64, fixed order) "
                     f"on m={m} x rows 0..{rows_all - 1} of n={n}, k={k}, all threads",
           "single_thread": {"value": v_one, "unit": unit, "cores": 1,
                             "sample": f"median of 3 runs: rows 0..{rows_one - 1}, one thread"},
           "nproc": os.cpu_count(), "sched_getaffinity": affinity}
    if gpu_Y is not None:
        rtol, atol = (1e-3, 1e-5) if m <= 16 else (1e-2, 1e-4)
        ratio = float((np.abs(gpu_Y[:, :rows_all].astype(np.float64) - Yr) / (rtol * B + atol)).max())
        res["parity_max_err_over_tol"] = ratio
    return res


def native(args):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from q4_quantized_linear_gb300 import build
    build.build()
    from q4_quantized_linear_gb300 import binding as q4lib

    # the packed weights are written once, before any timing, and then only
    # read: declare them read-only so consecutive calls overlap their weight
    # streams (programmatic dependent launch)
    q4lib.q4_set_weight_prefetch(True)
    peaks = load_peaks()
    cfg = WORKLOADS[args.workload]
    m, n, k = cfg["m"], cfg["n"], cfg["k"]
    wb = sweep_weight_bytes(cfg)
    flops = 2.0 * m * n * k
    tensor = m > 16
    stream = torch.cuda.Stream()
    wl = Workload(q4lib, m, n, k, w4a8=cfg.get("w4a8", False), w8=cfg.get("w8", False))

    sampler = ClockSampler(local) if rank == 0 else None
    barrier = dist.barrier if world > 1 else None
    sec, clocks = time_graph(q4lib, wl, args.steps, args.warmup, stream, sampler=sampler, barrier=barrier)
    sec = reduce_max(sec)
    unit = "TFLOP/s" if tensor else "GB/s"
    per_step_units = flops / 1e12 if tensor else wb / 1e9
    value = whole_job_rate(world, args.steps, per_step_units, sec)
    per_launch = sec / args.steps

    e2e_steps = min(args.steps, 5000)
    if barrier:
        barrier()
    esec, h2d, d2h = time_e2e(q4lib, wl, e2e_steps, stream)
    esec = reduce_max(esec)
    e2e_value = whole_job_rate(world, e2e_steps, per_step_units, esec)

    gpu_Y = wl.Yd.cpu().numpy()
    sweep = run_sweep(q4lib, stream, peaks) if (rank == 0 and not args.no_sweep) else None
    crossover = run_crossover(q4lib, stream) if (rank == 0 and not args.no_sweep) else None
    if world > 1:
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    cpu = None if args.no_cpu else cpu_baseline(cfg, gpu_Y, tensor)
    achieved = per_step_units / per_launch
    traffic = profiled_traffic(f"{args.workload}_m{m}_n{n}_k{k}")
    # a kernel of tens of microseconds runs at the burst rate
    peak, peak_key = (peaks["bf16_tflops"], "bf16_tflops") if tensor else (peaks["hbm_gbs"], "hbm_gbs")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": sec / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        # the operands the tensor cores take, fp32 accumulation throughout:
        # prefill bf16; decode m <= 4 fp16 weights (exact) against X as two
        # fp16 fixed-point terms per block; m >= 8 X as one fp16 term
        "dtype": "bf16" if tensor else ("f16x2" if m <= 4 else "f16"),
        "data": "synthetic",
        "config": {
            "workload": f"{cfg['name']}: Q4_0 W n={n} x k={k}, m={m}",
            "m": m, "n": n, "k": k,
            "weight_bytes_per_step": wb,
            "flop_per_step": flops,
            "l2": f"inputs larger than L2: {wl.copies} distinct packed weight copies "
                  f"({wl.copies * wb / 1e6:.0f} MB) cycled step by step",
            "launch": "CUDA graph replays of q4_0_matmul_ws, programmatic dependent launch, "
                      "weights declared read-only (q4_set_weight_prefetch)",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "bound": "tensor" if tensor else "hbm",
            "kernel": decode_kernel_name(m, n, torch.cuda.get_device_properties(local).multi_processor_count),
            "achieved": achieved,
            "peak": peak,
            "unit": unit,
            "frac": achieved / peak,
            "traffic": traffic,
            "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json {peak_key})" if peaks["source"] == "measured"
            else "fallback",
            # the spec sheet's dense figures, as a second reference beside the
            # measured denominator above (which the fraction uses)
            "nominal_peak": NOMINAL_BF16_TFLOPS if tensor else NOMINAL_HBM_GBS,
            "frac_nominal": achieved / (NOMINAL_BF16_TFLOPS if tensor else NOMINAL_HBM_GBS),
            "units": ("algorithmic FLOP = 2*m*n*k per step (cast + GEMM launches)" if tensor
                      else "algorithmic bytes = n*k + 4n int8 codes and scales per launch" if cfg.get("w8")
                      else "algorithmic bytes = n*k/32*18 Q4_0 weight bytes per launch"),
        },
        "e2e": {"value": e2e_value, "unit": unit, "steps": e2e_steps,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * (2 if tensor else 1),
        "clocks": clocks,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if sweep is not None:
        line["sweep"] = sweep
    if crossover is not None:
        line["expert_crossover"] = crossover
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def reference_sample_rows(n, steps, warmup, t_2048, budget_s=120.0):
    """Rows of W per reference step so that warmup + steps oracle calls take
    about budget_s, given t_2048 seconds for a 2048-row call: the whole layer
    when it fits (64-row units, at least 64, at most n)."""
    rows = int(2048 * budget_s / max((steps + warmup) * t_2048, 1e-9))
    return max(min(64, n), min(n, rows // 64 * 64))


def reference(args):
    """The oracle (CPU, as it stands) on the same config and metric."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return
    import oracle
    from q4_quantized_linear_gb300 import synth
    oracle.build()
    cfg = HEADLINE
    m, n, k = cfg["m"], cfg["n"], cfg["k"]
    wb = weight_bytes(n, k)
    blocks = synth.q4_0_blocks(n, k, seed=0)
    X = synth.activations(m, k, seed=0)
    # Each step covers the leading rows of W, as many as keep the whole
    # --warmup + --steps run near two minutes (the whole layer when it fits;
    # calibrated on 2048 rows).
    cal = min(n, 2048)
    oracle.matmul(blocks[:cal], X, cal, k)
    t0 = time.perf_counter()
    oracle.matmul(blocks[:cal], X, cal, k)
    t_full = (time.perf_counter() - t0) * 2048 / cal
    rows = reference_sample_rows(n, args.steps, args.warmup, t_full)
    sample_bytes = weight_bytes(rows, k)
    for _ in range(args.warmup):
        oracle.matmul(blocks[:rows], X, rows, k)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.matmul(blocks[:rows], X, rows, k)
    el = time.perf_counter() - t0
    value = args.steps * sample_bytes / el / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{cfg['name']}: Q4_0 W n={n} x k={k}, m={m}", "m": m, "n": n, "k": k},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"each step: rows 0..{rows - 1} of W ({sample_bytes} weight bytes), m={m}"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300000)
    ap.add_argument("--warmup", type=int, default=1000)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        if args.steps == 300000:
            args.steps = 20
        if args.warmup == 1000:
            args.warmup = 3
        reference(args)
    else:
        native(args)


if __name__ == "__main__":
    main()
