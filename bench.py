"""Benchmark of the routed NVFP4/INT8 linear layer + Temporal Delta Cache on GB300.

Workload (default): CogVideoX-5B-shaped DiT block linears, bf16, hidden 3072, 17776 tokens
(13x30x45 video + 226 text), QKV 3072->9216, out 3072->3072, FFN 3072->12288->3072 (GELU),
Hadamard block 64, Laplace(0,1) activations with 0.5% outlier channels x100, 42 blocks whose
Gamma ~ U(0, 0.2) routes each block to INT8 (Gamma > 0.05) or NVFP4.  Synthetic, seeded
inputs (no trained weights exist); weights N(0, 0.02), resident in both formats.

One step = one pass over the 42 blocks: for each block its four routed linears (online
block Hadamard + activation quantisation + quantised GEMM; GELU (erf form) fused into the
FFN-up epilogue, whose output is the FFN-down input; when both FFN linears route NVFP4 the
FFN-up epilogue also yields its output's NVFP4 tensor scale, so FFN-down's quantisation is
one pass) and the delta-cache commit of the block's own input/output pair (residual delta,
Gamma_t for the next step's routing, similarity of the last two deltas); block b + 1's input
is block b's output, as in the DiT's residual stream.
value = algorithmic GEMM FLOPs of the step / step time (TFLOP/s).

Further keys of the JSON line: the CogVideoX-2B step (hidden 1920, 30 blocks), the whole
1080p-shaped path (104746 tokens: Gamma, both quantisers, both FFN GEMMs per route, delta
commit and skip), the NVFP4-only-weights variant, the full TDC/PDR loop (50 steps x 30 2B
blocks, its decisions replayed by the CPU oracle) and the CPU oracle baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own replica (independent problems, no data-path
collective: weak scaling); value = FLOPs of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-linear TFLOPS (NVFP4 / INT8) & HBM GB/s of quant+TDC, 1 GB300"
UNIT = "TFLOP/s"
HBLOCK = 64
THR, ALPHA, BETA = 0.05, 1.0, 0.0
TOKENS = 13 * 30 * 45 + 226
TOKENS_1080P = 13 * 67 * 120 + 226

WORKLOADS = {
    "cogvideox_5b_block_linears": {"tokens": TOKENS, "hidden": 3072, "ffn": 12288, "blocks": 42,
                                   "dist": "laplace", "outlier_frac": 0.005, "outlier_mult": 100.0,
                                   "activations": "Laplace(0,1), 0.5% outlier channels x100"},
    "cogvideox_2b_block_linears": {"tokens": TOKENS, "hidden": 1920, "ffn": 7680, "blocks": 30,
                                   "dist": "normal", "outlier_frac": 0.01, "outlier_mult": 50.0,
                                   "activations": "N(0,1), 1% outlier channels x50"},
}
DEFAULT_WORKLOAD = "cogvideox_5b_block_linears"
KINDS = ("gemm_int8", "gemm_nvfp4", "quant_int8", "quant_nvfp4", "tdc_commit")


def linears(spec):
    h, f = spec["hidden"], spec["ffn"]
    return [("qkv", h, 3 * h), ("out", h, h), ("ffn_up", h, f), ("ffn_down", f, h)]


# Algorithmic bytes of the streaming kernels (bf16 input), per call
def bytes_quant_int8(m, k):       # 2 in + 1 out per element + one fp32 scale per row
    return m * k * 3 + 4 * m


def bytes_quant_nvfp4(m, k):      # 2 in + 0.5 codes + 1/16 block scales per element
    return m * k * 2 + m * k // 2 + m * k // 16


# The sources each kernel type is built from (its own file, the shared device helpers and the
# host-side launch glue); a measured DRAM figure stands while these are unchanged.
KERNEL_SOURCES = {
    "gemm_int8": ["gemm_int8_tc.cu", "gemm_int8.cu"],
    "gemm_nvfp4": ["gemm_nvfp4.cu"],
    "quant_int8": ["quant.cu"],
    "quant_nvfp4": ["quant.cu"],
    "tdc_commit": ["reduce.cu"],
}
SHARED_SOURCES = ["common.cuh", "api.cu"]
TRAFFIC_PROFILE = os.path.join("profiles", "dram_traffic_cogvideox5b_layers.md")


def kernel_sources_hash(kind: str) -> str:
    """sha256 over the kernel type's source files and the shared ones, names and bytes."""
    import hashlib
    csrc = os.path.join(ROOT, "int8_mixed_precision_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in sorted(KERNEL_SOURCES[kind] + SHARED_SOURCES)]
    files.append(os.path.join(ROOT, "include", "dit6.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(kind: str):
    """DRAM bytes per launch of a kernel type in the default step, from the committed ncu
    summary: the mean of the per-shape captures listed for that type (every block that routes
    a kernel type runs it once per listed layer shape), or None when the type has no capture or
    its sources have changed since (their hash, listed per type, differs)."""
    import re
    try:
        text = open(os.path.join(ROOT, TRAFFIC_PROFILE)).read()
    except OSError:
        return None
    if kind not in KERNEL_SOURCES:
        return None
    m = re.search(r"^\| " + re.escape(kind) + r" sources \| ([0-9a-f]{64}) \|", text, re.M)
    if not m or m.group(1) != kernel_sources_hash(kind):
        return None
    rows = re.findall(r"^\| " + re.escape(kind) + r" \| [^|]+ \| \d+ \| [\d.]+ \| [\d.]+ \| (\d+) \|", text, re.M)
    return int(round(sum(int(r) for r in rows) / len(rows))) if rows else None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class Clocks:
    """nvidia-smi sampling (every 100 ms) around the timed region: the sampler starts half a
    second early, mark() brackets the timed region, and the summary keeps the samples whose
    timestamps fall inside it (all samples if none does)."""

    def __init__(self, index: int):
        self.proc = None
        self.index = index
        self.window = None

    def __enter__(self):
        q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)
        except OSError:
            self.proc = None
        return self

    def mark(self, start: float, end: float):
        self.window = (start, end)

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            time.sleep(0.15)   # one more sample period after the timed region
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    @staticmethod
    def parse(lines, window=None):
        """Samples (time, sm MHz, max MHz, set of active throttle reasons) from nvidia-smi csv
        lines, restricted to the wall-clock window when one is given and holds any; the flag
        says whether the restriction applied."""
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]),
                             {n for n, v in zip(names, f[6:10]) if v.lower() == "active"}))
            except (ValueError, IndexError):
                continue
        if window:
            inside = [r for r in rows if window[0] - 0.05 <= r[0] <= window[1] + 0.05]
            if inside:
                return inside, True
        return rows, False

    def summary(self):
        rows, inside = self.parse(getattr(self, "lines", []), self.window)
        reasons = set().union(*[r[3] for r in rows]) if rows else set()
        return {"sm_mhz": statistics.median([r[1] for r in rows]) if rows else None,
                "sm_max_mhz": rows[-1][2] if rows else None, "reasons": sorted(reasons),
                "samples": len(rows), "in_timed_region": inside}


# ----------------------------------------------------------------------------------------
# our implementation
# ----------------------------------------------------------------------------------------


def device_activations(torch, g, dev, m, k, spec, seed):
    """[m x k] bf16 activations of the workload's law on the device (seeded torch generator):
    N(0,1) or Laplace(0,1) (inverse CDF of a uniform draw), floor(frac * k) outlier channels
    scaled by the multiplier."""
    g.manual_seed(seed)
    if spec["dist"] == "laplace":
        u = torch.rand(m, k, device=dev, generator=g).clamp_(min=2.0 ** -24) - 0.5
        x = -torch.sign(u) * torch.log1p(-2.0 * u.abs())
        del u
    else:
        x = torch.randn(m, k, device=dev, generator=g)
    ch = torch.randperm(k, device=dev, generator=g)[: max(1, int(k * spec["outlier_frac"]))]
    x[:, ch] *= spec["outlier_mult"]
    return x.to(torch.bfloat16)


class Workload:
    """Device-resident synthetic workload: the blocks of routed linears + delta-cache state."""

    def __init__(self, dev, seed: int, name: str = DEFAULT_WORKLOAD):
        import torch
        import int8_mixed_precision_gb300 as dit
        self.dit, self.torch, self.dev = dit, torch, dev
        self.name, self.spec = name, WORKLOADS[name]
        self.lin_shapes = linears(self.spec)
        self.nblocks = self.spec["blocks"]
        g = torch.Generator(device=dev)
        self.ws = dit.workspace(dev)
        M, H = self.spec["tokens"], self.spec["hidden"]
        act = lambda k, s: device_activations(torch, g, dev, M, k, self.spec, seed * 1000 + s)
        # two alternating sets of linear inputs (consecutive blocks never share an input
        # tensor); the FFN-down input is GELU(FFN-up output), produced in the step
        self.inputs = [{name: act(k, 10 * s + i) for i, (name, k, _) in enumerate(self.lin_shapes)
                        if name != "ffn_down"} for s in range(2)]
        # per-block Gamma pairs: X_out = X_in + gamma_b * S * X_in, gamma_b ~ U(0, 0.2); every
        # block commits its own pair.  The blocks form a residual stream: block b + 1's input is
        # block b's output (the same tensor), as in the DiT, so a step holds nblocks + 1 of them
        g.manual_seed(seed + 7)
        self.gammas_true = (torch.rand(self.nblocks, generator=g, device=dev) * 0.2).tolist()
        # quantised-activation buffers shared by all blocks (one stream orders their uses)
        self.act_bufs = {}
        for _, k, _ in self.lin_shapes:
            if k not in self.act_bufs:
                self.act_bufs[k] = (dit.alloc_nvfp4(M, k, dev), dit.alloc_int8(M, k, dev))
        self.x_in, self.x_out, self.blocks = [], [], []
        for b in range(self.nblocks):
            xi = act(H, 500) if b == 0 else self.x_out[b - 1]
            g.manual_seed(seed * 31 + b)
            sgn = torch.randint(0, 2, xi.shape, generator=g, device=dev).to(torch.float32) * 2 - 1
            self.x_in.append(xi)
            self.x_out.append((xi.float() * (1 + self.gammas_true[b] * sgn)).to(torch.bfloat16))
            del sgn
            lins = {}
            for name, k, n in self.lin_shapes:
                g.manual_seed(seed * 7919 + b * 17 + n + k)
                w = torch.randn(n, k, device=dev, generator=g) * 0.02
                lins[name] = dit.RoutedLinear(dit.QuantizedWeight(w, HBLOCK, self.ws), M, self.ws, dev,
                                              act_buffers=self.act_bufs[k])
                del w
            self.blocks.append({"lin": lins, "d": [torch.empty_like(xi), torch.empty_like(xi)],
                                "has_delta": False})
        self.y = {name: torch.empty(M, n, dtype=torch.bfloat16, device=dev) for name, _, n in self.lin_shapes}
        self.gamma = torch.empty(self.nblocks, dtype=torch.float32, device=dev)
        self.up_scale = torch.empty(1, dtype=torch.float32, device=dev)   # FFN-up output's NVFP4 tensor scale
        self.sim = torch.empty(self.nblocks, dtype=torch.float32, device=dev)
        # routing from the predictor (one Gamma per block; the commit of every step
        # recomputes it, and with fixed pairs the routes stay the same)
        r = torch.empty(4, dtype=torch.int32, device=dev)
        self.routes = []
        for b in range(self.nblocks):
            dit.gamma_route(self.x_in[b], self.x_out[b], [ALPHA] * 4, [BETA] * 4, [THR] * 4,
                            self.gamma[b:b + 1], r, self.ws)
            self.routes.append(r.tolist())
        torch.cuda.synchronize()
        self.flops_step = self.nblocks * sum(2 * M * n * k for _, k, n in self.lin_shapes)
        self.int8_code_bytes = self.act_bufs[H][1]["q"].element_size()
        self.timers = None   # {kernel type: [event pairs]} when per-kernel timing is on

    def free(self):
        self.inputs = self.x_in = self.x_out = self.blocks = self.y = self.act_bufs = None
        self.torch.cuda.empty_cache()

    def chained(self, b):
        nv = self.dit.ROUTE_NVFP4
        return self.routes[b][2] == nv and self.routes[b][3] == nv

    def launches_per_step(self):
        n = 0
        for b in range(self.nblocks):
            for li, r in enumerate(self.routes[b]):
                n += 2 if r == self.dit.ROUTE_INT8 or (self.chained(b) and li == 3) else 3
            n += 1
        return n

    def _timed(self, kind, fn):
        if self.timers is None or kind not in self.timers:
            return fn()
        a = self.torch.cuda.Event(enable_timing=True)
        z = self.torch.cuda.Event(enable_timing=True)
        a.record()
        r = fn()
        z.record()
        self.timers[kind].append((a, z))
        return r

    def step(self, before_block=None):
        """One pass over the blocks; before_block(b), if given, runs on the host before block b's
        launches are enqueued (the end-to-end leg makes the stream wait there for block b's
        host-to-device copies)."""
        dit = self.dit
        for b, blk in enumerate(self.blocks):
            if before_block is not None:
                before_block(b)
            xs = self.inputs[b % 2]
            chained = self.chained(b)
            for li, (name, k, n) in enumerate(self.lin_shapes):
                lin = blk["lin"][name]
                route = self.routes[b][li]
                x = self.y["ffn_up"] if name == "ffn_down" else xs[name]
                y = self.y[name]
                act = dit.ACT_GELU_ERF if name == "ffn_up" else dit.ACT_NONE
                if route == dit.ROUTE_INT8:
                    self._timed("quant_int8", lambda: dit.hadamard_quant_int8(x, HBLOCK, lin.a8["q"], lin.a8["scale"]))
                    w8 = lin.w.int8
                    if w8 is None:  # NVFP4-only weights: derive the INT8 weights for this call
                        w8 = self._timed("w_nvfp4_to_int8", lambda: lin.w.int8_into(lin.w8_scratch))
                    self._timed("gemm_int8", lambda: dit.qgemm_int8(lin.a8["q"], lin.a8["scale"], w8["q"],
                                                                    w8["scale"], y, self.ws, act=act))
                else:
                    # FFN-up -> FFN-down both on NVFP4: the FFN-up GEMM's epilogue also yields its
                    # output's tensor scale, and FFN-down's quantisation is then one pass
                    ts_in = self.up_scale if (chained and name == "ffn_down") else None
                    self._timed("quant_nvfp4", lambda: dit.hadamard_quant_nvfp4(
                        x, HBLOCK, lin.a4["codes"], lin.a4["sf"], lin.a4["gs"], self.ws, tensor_scale_in=ts_in))
                    if chained and name == "ffn_up":
                        self._timed("gemm_nvfp4", lambda: dit.qgemm_nvfp4_amax(
                            lin.a4["codes"], lin.a4["sf"], lin.a4["gs"], lin.w.nvfp4["codes"], lin.w.nvfp4["sf"],
                            lin.w.nvfp4["gs"], y, self.ws, HBLOCK, self.up_scale, act=act))
                    else:
                        self._timed("gemm_nvfp4", lambda: dit.qgemm_nvfp4(
                            lin.a4["codes"], lin.a4["sf"], lin.a4["gs"], lin.w.nvfp4["codes"], lin.w.nvfp4["sf"],
                            lin.w.nvfp4["gs"], y, self.ws, act=act))
            d_new, d_old = blk["d"][0], blk["d"][1]
            self._timed("tdc_commit", lambda: dit.tdc_step(
                dit.TDC_COMMIT, self.x_in[b], self.ws, x_out=self.x_out[b], d1=d_old if blk["has_delta"] else None,
                d_new=d_new, gamma=self.gamma[b:b + 1], sim=self.sim[b:b + 1]))
            blk["d"].reverse()
            blk["has_delta"] = True

    def kernel_units(self):
        """Algorithmic units per kernel type and step: FLOPs (2 M N K) for the GEMMs, the bytes of
        the survey's per-element accounting otherwise (INT8 quantiser 3 B/elem + 4 B/row, NVFP4
        quantiser 2.5625 B/elem, delta commit 8 B/elem).  The second dict holds the bytes the
        quantisers really move (bf16-held INT8 codes, the NVFP4 amax pass)."""
        M, H = self.spec["tokens"], self.spec["hidden"]
        u = {k: 0 for k in KINDS}
        moved = {"quant_int8": 0, "quant_nvfp4": 0}
        for b in range(self.nblocks):
            for li, (name, k, n) in enumerate(self.lin_shapes):
                if self.routes[b][li] == self.dit.ROUTE_INT8:
                    u["gemm_int8"] += 2 * M * n * k
                    u["quant_int8"] += bytes_quant_int8(M, k)
                    moved["quant_int8"] += M * k * (2 + self.int8_code_bytes) + 4 * M
                else:
                    u["gemm_nvfp4"] += 2 * M * n * k
                    u["quant_nvfp4"] += bytes_quant_nvfp4(M, k)
                    one_pass = self.chained(b) and name == "ffn_down"
                    moved["quant_nvfp4"] += bytes_quant_nvfp4(M, k) + (0 if one_pass else 2 * M * k)
            u["tdc_commit"] += M * H * 8
        return u, moved


def _median_us(torch, fn, reps, flush):
    fn()
    times = []
    for _ in range(reps):
        if flush is not None:
            flush.max()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(times)


def run_long_1080p(dev, reps: int = 5):
    """The whole hot path on the 1080p-shaped long sequence (104746 tokens, hidden 3072, FFN
    3072 -> 12288 -> 3072, Laplace activations with 0.5 % outlier channels x100): Gamma and
    routing, both quantisers on the FFN-up input (3072) and the FFN-down input (12288), the FFN
    GEMMs on both routes (GELU in the FFN-up epilogue; on the NVFP4 route it also yields the
    FFN-down input's tensor scale, so that quantisation is one pass), the delta-cache commit and
    skip.  Each kernel: median CUDA-event time of `reps` launches, L2 flushed before each (a
    640 MB read), against the measured burst peaks (kernels timed alone).  The per-route path
    adds the kernels one FFN pass of that route runs."""
    import torch
    import int8_mixed_precision_gb300 as dit
    pk, src = peaks()
    spec = WORKLOADS["cogvideox_5b_block_linears"]
    m, h, f = TOKENS_1080P, 3072, 12288
    g = torch.Generator(device=dev)
    ws = dit.workspace(dev)
    flush = torch.ones(640 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    x = device_activations(torch, g, dev, m, h, spec, 9001)
    g.manual_seed(9002)
    sgn = torch.randint(0, 2, x.shape, generator=g, device=dev).to(torch.float32) * 2 - 1
    x_out = (x.float() * (1 + 0.1 * sgn)).to(torch.bfloat16)
    del sgn
    d1 = (x_out.float() - x.float()).mul_(1.01).to(torch.bfloat16)
    d_new, skip_out = torch.empty_like(x), torch.empty_like(x)
    g.manual_seed(9003)
    w_up = torch.randn(f, h, device=dev, generator=g) * 0.02
    w_dn = torch.randn(h, f, device=dev, generator=g) * 0.02
    up = dit.RoutedLinear(dit.QuantizedWeight(w_up, HBLOCK, ws), m, ws, dev)
    dn = dit.RoutedLinear(dit.QuantizedWeight(w_dn, HBLOCK, ws), m, ws, dev)
    del w_up, w_dn
    y_up = torch.empty(m, f, dtype=torch.bfloat16, device=dev)
    y_dn = torch.empty(m, h, dtype=torch.bfloat16, device=dev)
    gam = torch.empty(1, device=dev)
    sim = torch.empty(1, device=dev)
    routes = torch.empty(4, dtype=torch.int32, device=dev)
    up_scale = torch.empty(1, device=dev)
    up(x, dit.ROUTE_NVFP4, y_up, act=dit.ACT_GELU_ERF)      # a GELU output as the FFN-down input
    A, W = up.a4, up.w.nvfp4
    calls = {
        "gamma_route": (lambda: dit.gamma_route(x, x_out, [ALPHA] * 4, [BETA] * 4, [THR] * 4, gam, routes, ws),
                        "hbm", 4 * m * h),
        "quant_nvfp4_k3072": (lambda: dit.hadamard_quant_nvfp4(x, HBLOCK, up.a4["codes"], up.a4["sf"], up.a4["gs"],
                                                               ws), "hbm", bytes_quant_nvfp4(m, h)),
        "quant_int8_k3072": (lambda: dit.hadamard_quant_int8(x, HBLOCK, up.a8["q"], up.a8["scale"]), "hbm",
                             bytes_quant_int8(m, h)),
        "gemm_nvfp4_ffn_up_gelu_amax": (lambda: dit.qgemm_nvfp4_amax(A["codes"], A["sf"], A["gs"], W["codes"],
                                                                     W["sf"], W["gs"], y_up, ws, HBLOCK, up_scale,
                                                                     act=dit.ACT_GELU_ERF), "tensor_fp4", 2 * m * f * h),
        "gemm_int8_ffn_up_gelu": (lambda: dit.qgemm_int8(up.a8["q"], up.a8["scale"], up.w.int8["q"],
                                                         up.w.int8["scale"], y_up, ws, act=dit.ACT_GELU_ERF),
                                  "tensor_bf16", 2 * m * f * h),
        "quant_nvfp4_k12288_one_pass": (lambda: dit.hadamard_quant_nvfp4(y_up, HBLOCK, dn.a4["codes"], dn.a4["sf"],
                                                                         dn.a4["gs"], ws, tensor_scale_in=up_scale),
                                        "hbm", bytes_quant_nvfp4(m, f)),
        "quant_nvfp4_k12288_two_pass": (lambda: dit.hadamard_quant_nvfp4(y_up, HBLOCK, dn.a4["codes"], dn.a4["sf"],
                                                                         dn.a4["gs"], ws), "hbm", bytes_quant_nvfp4(m, f)),
        "quant_int8_k12288": (lambda: dit.hadamard_quant_int8(y_up, HBLOCK, dn.a8["q"], dn.a8["scale"]), "hbm",
                              bytes_quant_int8(m, f)),
        "gemm_nvfp4_ffn_down": (lambda: dit.qgemm_nvfp4(dn.a4["codes"], dn.a4["sf"], dn.a4["gs"], dn.w.nvfp4["codes"],
                                                        dn.w.nvfp4["sf"], dn.w.nvfp4["gs"], y_dn, ws),
                                "tensor_fp4", 2 * m * h * f),
        "gemm_int8_ffn_down": (lambda: dit.qgemm_int8(dn.a8["q"], dn.a8["scale"], dn.w.int8["q"], dn.w.int8["scale"],
                                                      y_dn, ws), "tensor_bf16", 2 * m * h * f),
        "tdc_commit": (lambda: dit.tdc_step(dit.TDC_COMMIT, x, ws, x_out=x_out, d1=d1, d_new=d_new, gamma=gam,
                                            sim=sim), "hbm", 8 * m * h),
        "tdc_skip": (lambda: dit.tdc_step(dit.TDC_SKIP, x, ws, x_out_skip=skip_out, d1=d1), "hbm", 6 * m * h),
    }
    out = {}
    for name, (fn, bound, units) in calls.items():
        us = _median_us(torch, fn, reps, flush)
        if bound == "hbm":
            a = units / (us * 1e-6) / 1e9
            out[name] = {"us": round(us, 1), "achieved": round(a, 1), "unit": "GB/s", "peak": pk["hbm_gbs"],
                         "frac": round(a / pk["hbm_gbs"], 4)}
        else:
            a = units / (us * 1e-6) / 1e12
            p = pk["bf16_tflops"] * (6.0 if bound == "tensor_fp4" else 1.0)
            out[name] = {"us": round(us, 1), "achieved": round(a, 1), "unit": "TFLOP/s", "peak": round(p, 1),
                         "frac": round(a / p, 4)}
    torch.cuda.synchronize()
    assert dit.device_status(ws) == 0
    flops = 2 * 2 * m * h * f
    paths = {"nvfp4": ["gamma_route", "quant_nvfp4_k3072", "gemm_nvfp4_ffn_up_gelu_amax",
                       "quant_nvfp4_k12288_one_pass", "gemm_nvfp4_ffn_down", "tdc_commit"],
             "int8": ["gamma_route", "quant_int8_k3072", "gemm_int8_ffn_up_gelu", "quant_int8_k12288",
                      "gemm_int8_ffn_down", "tdc_commit"]}
    for route, names in paths.items():
        us = sum(out[n]["us"] for n in names)
        out[f"path_{route}"] = {"us": round(us, 1), "tflops": round(flops / (us * 1e-6) / 1e12, 1),
                                "kernels": names}
    out["workload"] = {"tokens": m, "hidden": h, "ffn": f, "activations": spec["activations"],
                       "peak_source": f"{src} HBM copy; bf16 burst (INT8 codes on the bf16 tensor pipe); "
                                      "bf16 burst x 6 (NVFP4, nominal dense fp4/bf16 ratio)"}
    del up, dn, x, x_out, d1, d_new, skip_out, y_up, y_dn, flush
    torch.cuda.empty_cache()
    return out


def run_int8_requant(dev, reps: int = 5):
    """The INT8 leg of fusing the next layer's quantisation, at the CogVideoX-5B FFN-up shape
    (17776 tokens, 3072 -> 12288, GELU): the GEMM writing bf16 followed by FFN-down's INT8
    quantiser, against the GEMM whose epilogue quantises with given per-token scales (here the
    exact ones of the unfused run, so the codes must agree bit for bit; in a denoising loop they
    would be the previous step's).  Not part of the step: the method's scales are dynamic."""
    import numpy as np
    import torch
    import int8_mixed_precision_gb300 as dit
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    m, k, n = 17776, 3072, 12288
    ws = dit.workspace(dev)
    a = torch.randint(-127, 128, (m, k), generator=g, device=dev).to(torch.bfloat16)
    w = torch.randint(-127, 128, (n, k), generator=g, device=dev).to(torch.bfloat16)
    sa = torch.rand(m, generator=g, device=dev) * 2e-4 + 1e-5
    sw = torch.rand(n, generator=g, device=dev) * 2e-4 + 1e-5
    y = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
    q_ref = torch.empty_like(y)
    s_ref = torch.empty(m, dtype=torch.float32, device=dev)
    q = torch.empty_like(y)
    amax = torch.zeros(m, dtype=torch.float32, device=dev)
    flush = torch.empty(640 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def unfused():
        dit.qgemm_int8(a, sa, w, sw, y, ws, act=dit.ACT_GELU_ERF)
        dit.hadamard_quant_int8(y, 64, q_ref, s_ref)

    def fused():
        dit.qgemm_int8_requant(a, sa, w, sw, s_ref, q, amax, ws, act=dit.ACT_GELU_ERF)

    t_gemm = _median_us(torch, lambda: dit.qgemm_int8(a, sa, w, sw, y, ws, act=dit.ACT_GELU_ERF), reps, flush)
    t_unfused = _median_us(torch, unfused, reps, flush)
    t_fused = _median_us(torch, fused, reps, flush)
    amax.zero_()
    fused()
    torch.cuda.synchronize()
    same = bool(torch.equal(q.view(torch.int16), q_ref.view(torch.int16)))
    s_from_amax = (amax.cpu().numpy() / np.float32(127.0)).astype(np.float32)   # IEEE division, as the quantiser
    same_scale = bool(np.array_equal(s_from_amax.view(np.uint32), s_ref.cpu().numpy().view(np.uint32)))
    status = dit.device_status(ws)
    del a, w, y, q_ref, q, flush
    torch.cuda.empty_cache()
    flops = 2 * m * n * k
    return {"shape": "17776 x 3072 -> 12288, GELU", "gemm_us": round(t_gemm, 1),
            "gemm_then_quantiser_us": round(t_unfused, 1), "fused_requant_us": round(t_fused, 1),
            "saved_us": round(t_unfused - t_fused, 1), "fused_tflops": round(flops / (t_fused * 1e-6) / 1e12, 1),
            "codes_equal_unfused": same, "row_maxima_give_the_same_scales": same_scale, "status": status,
            "note": "per-token scales given (exact ones here); the method's scales are dynamic, so the step "
                    "keeps the unfused pair"}


def run_nvfp4_only_weights(wl, steps: int = 3):
    """The same step with every weight resident in NVFP4 only ([ZH] 2.A weight handling): each
    INT8-routed layer derives its INT8 weights per call into one scratch buffer per K."""
    import torch
    import int8_mixed_precision_gb300 as dit
    dev = wl.dev
    scratch = {k: dit.alloc_int8(max(n for _, kk, n in wl.lin_shapes if kk == k), k, dev) for _, k, _ in wl.lin_shapes}
    saved = []
    for blk in wl.blocks:
        for name, k, n in wl.lin_shapes:
            lin = blk["lin"][name]
            saved.append((lin, lin.w, lin.w8_scratch))
            lin.w = lin.w.without_int8()
            lin.w8_scratch = scratch[k]
    both = sum(w.resident_bytes() for _, w, _ in saved)
    only = sum(lin.w.resident_bytes() for lin, _, _ in saved)
    wl.step()
    wl.timers = {"w_nvfp4_to_int8": []}
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        wl.step()
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    conv_ms = sum(a.elapsed_time(z) for a, z in wl.timers["w_nvfp4_to_int8"]) / steps
    wl.timers = None
    for lin, w, sc in saved:
        lin.w, lin.w8_scratch = w, sc
    return {"workload": wl.name, "ms_per_step": round(ms, 3), "value": round(wl.flops_step / (ms * 1e-3) / 1e12, 3),
            "unit": UNIT, "weight_conversion_ms_per_step": round(conv_ms, 3),
            "resident_weight_bytes": int(only), "resident_weight_bytes_nvfp4_and_int8": int(both),
            "note": "weights resident in NVFP4 only; INT8-routed layers convert theirs per call (dit_nvfp4_to_int8)"}


def run_tdc_loop(wl, steps: int = 50, tau: float = 0.05, seed: int = 77, replay_blocks: int = 2):
    """The full TDC/PDR loop on CogVideoX-2B blocks: per denoising step and block, skip (X_out =
    X_in + cached delta) or compute (four routed linears + delta commit), with the block chain
    X_in(b+1) = X_out(b).  The synthetic "true" block delta follows Delta_t = Delta_{t-1}
    (1 + eps), eps ~ N(0, 0.01) elementwise, N(0, 0.5) on jump steps (Bernoulli(1/8) per
    block-step), Delta_0 ~ N(0, sigma_b), sigma_b ~ U(0.02, 0.15), held in bf16; it is generated
    on the device between our kernels and is not part of the timed segments.  The first
    `replay_blocks` blocks of the chain are replayed by the CPU oracle step by step on host
    copies of their inputs and true deltas: skip decisions and routes must be identical (a
    decision or route within 1e-5 relative of its threshold is counted, not compared)."""
    import torch
    import int8_mixed_precision_gb300 as dit
    from oracle import dmpq as D
    from oracle import tdc as T
    dev, M, H = wl.dev, wl.spec["tokens"], wl.spec["hidden"]
    nb = wl.nblocks
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    gam = torch.zeros(nb, dtype=torch.float32, device=dev)
    sim = torch.zeros(nb, dtype=torch.float32, device=dev)
    blocks = [dit.DeltaCachedBlock(M * H, torch.bfloat16, tau, [ALPHA] * 4, [BETA] * 4, [THR] * 4, wl.ws,
                                   gam[b:b + 1], sim[b:b + 1], dev) for b in range(nb)]
    sig = (torch.rand(nb, generator=g, device=dev) * 0.13 + 0.02).tolist()
    deltas = [(torch.randn(M, H, generator=g, device=dev) * sig[b]).to(torch.bfloat16) for b in range(nb)]
    x0 = wl.x_in[0]
    xb = [torch.empty_like(x0), torch.empty_like(x0)]
    y = wl.y
    oracle = [T.BlockLoop(tau, [ALPHA] * 4, [BETA] * 4, [THR] * 4, "bf16") for _ in range(replay_blocks)]
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view("uint16")
    mismatch, borderline, compared = 0, 0, 0
    segs, n_skip, n_comp, route_count, launches = [], 0, 0, [0, 0], 0
    ev = lambda: torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    oracle_s = 0.0
    for t in range(steps):
        x = x0
        for b, blk in enumerate(blocks):
            if t > 0:  # advance the true trajectory
                jump = bool(torch.rand(1, generator=g, device=dev).item() < 1.0 / 8.0)
                eps = torch.randn(M, H, generator=g, device=dev) * (0.5 if jump else 0.01)
                deltas[b] = (deltas[b].float() * (1.0 + eps)).to(torch.bfloat16)
                del eps
            x_next = xb[1] if x is xb[0] else xb[0]
            mode = blk.decide()
            routes = None
            a, z = ev(), ev()
            if mode == dit.TDC_SKIP:
                a.record()
                blk.skip(x, x_next)
                z.record()
                segs.append(("skip", a, z))
                n_skip += 1
                launches += 1
            else:
                routes = blk.routes()
                lins = wl.blocks[b]["lin"]
                a.record()
                for li, (name, k, n) in enumerate(wl.lin_shapes):
                    xin = y["ffn_up"] if name == "ffn_down" else x
                    lins[name](xin, routes[li], y[name],
                               act=dit.ACT_GELU_ERF if name == "ffn_up" else dit.ACT_NONE)
                    launches += 2 if routes[li] == dit.ROUTE_INT8 else 3
                    route_count[routes[li]] += 1
                z.record()
                segs.append(("linears", a, z))
                x_next.copy_((x.float() + deltas[b].float()).to(torch.bfloat16))
                a2, z2 = ev(), ev()
                a2.record()
                blk.commit(x, x_next)
                z2.record()
                segs.append(("commit", a2, z2))
                n_comp += 1
                launches += 1
            if b < replay_blocks:   # the oracle takes the same step on host copies
                t0 = time.perf_counter()
                r = oracle[b].step(bits(x).reshape(M, H), bits(deltas[b]).reshape(M, H), want_skip_output=False)
                got = "skip" if mode == dit.TDC_SKIP else "compute"
                if r["margin"] <= 1e-5:
                    borderline += 1
                else:
                    compared += 1
                    if r["decision"] != got:
                        mismatch += 1
                    elif routes is not None:
                        g_ref = r["gamma"]
                        if g_ref is not None and D.route_margin(g_ref, ALPHA, BETA, THR) <= 1e-5:
                            borderline += 1
                        elif routes != r["routes"]:
                            mismatch += 1
                oracle_s += time.perf_counter() - t0
            x = x_next
        h = torch.stack([gam, sim]).cpu()      # one device-to-host copy per denoising step
        for b, blk in enumerate(blocks):
            blk.absorb(float(h[0, b]), float(h[1, b]))
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    tot = {"skip": 0.0, "linears": 0.0, "commit": 0.0}
    for kind, a, z in segs:
        tot[kind] += a.elapsed_time(z)
    kernel_ms = sum(tot.values())
    n_elem = M * H
    total_bits = route_count[1] * 8 + route_count[0] * 4.5
    del deltas, xb
    torch.cuda.empty_cache()
    return {
        "workload": "cogvideox_2b_tdc_loop", "denoising_steps": steps, "blocks": nb, "tau": tau,
        "skip_fraction": round(n_skip / (n_skip + n_comp), 4), "computed_block_steps": n_comp,
        "skipped_block_steps": n_skip, "routes": {"int8": route_count[1], "nvfp4": route_count[0]},
        "avg_activation_bits": round(total_bits / max(1, sum(route_count)), 3),
        "kernel_ms_total": round(kernel_ms, 2), "kernel_ms_per_denoising_step": round(kernel_ms / steps, 3),
        "wall_s_incl_synthetic_delta_generation_and_oracle_replay": round(wall, 2),
        "tdc_skip_gbs": round(n_skip * n_elem * 6 / (tot["skip"] * 1e-3) / 1e9, 1) if n_skip else None,
        "tdc_commit_gbs": round(n_comp * n_elem * 8 / (tot["commit"] * 1e-3) / 1e9, 1) if n_comp else None,
        "gpu_launches": launches,
        "oracle_replay": {"blocks": replay_blocks, "block_steps_compared": compared, "borderline": borderline,
                          "mismatches": mismatch, "decisions_match_oracle": mismatch == 0,
                          "cpu_seconds": round(oracle_s, 1)},
    }


def max_over_ranks(value: float, world: int, device="cpu") -> float:
    """Largest value over all ranks (the step time the job reports); identity at world 1."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as tdist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / (ms_max * 1e-3) / 1e12


def instrumented_kernels(wl, pk):
    """One step with every launch event-timed: total ms per kernel type and each type against
    its own bound (GEMMs: bf16 sustained, x 6 for NVFP4; streaming kernels: the HBM copy rate
    at the algorithmic bytes, with the bytes the quantisers really move beside them)."""
    torch = wl.torch
    wl.timers = {k: [] for k in KINDS}
    wl.step()
    torch.cuda.synchronize()
    tot = {k: sum(a.elapsed_time(z) for a, z in v) for k, v in wl.timers.items()}
    n = {k: len(v) for k, v in wl.timers.items()}
    wl.timers = None
    units, moved = wl.kernel_units()
    roof = {}
    for k, t in tot.items():
        if not t:
            continue
        if k.startswith("gemm"):
            a = units[k] / (t * 1e-3) / 1e12
            p = pk["bf16_tflops_sustained"] * (6.0 if k == "gemm_nvfp4" else 1.0)
            roof[k] = {"bound": "tensor", "achieved": round(a, 1), "peak": round(p, 1), "unit": "TFLOP/s",
                       "frac": round(a / p, 4), "launches": n[k], "ms": round(t, 3)}
        else:
            a = units[k] / (t * 1e-3) / 1e9
            roof[k] = {"bound": "hbm", "achieved": round(a, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                       "frac": round(a / pk["hbm_gbs"], 4), "launches": n[k], "ms": round(t, 3)}
            if k in moved:
                roof[k]["moved_gbs"] = round(moved[k] / (t * 1e-3) / 1e9, 1)
    return tot, roof


def time_steps(wl, steps, warmup, world, barrier, dominant=None, clocks=None):
    """Device-timed region (inputs resident in HBM): `steps` steps after `warmup` untimed ones,
    CUDA events on the launching stream, max over ranks.  With `dominant`, that kernel type's
    launches are event-timed inside the region as well."""
    torch = wl.torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        wl.step()
    wl.timers = {dominant: []} if dominant else None
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")
    w0 = time.time()
    e0.record(stream)
    for _ in range(steps):
        wl.step()
    e1.record(stream)
    torch.cuda.nvtx.range_pop()
    e1.synchronize()
    if clocks is not None:
        clocks.mark(w0, time.time())
    barrier()
    ms = e0.elapsed_time(e1) / steps
    dom_ms = [a.elapsed_time(z) for a, z in wl.timers[dominant]] if dominant else []
    wl.timers = None
    return max_over_ranks(ms, world, wl.dev), dom_ms


def e2e_leg(wl, steps, world, barrier):
    """The same metric end to end through the public API: every step copies its inputs from
    pinned host memory (the linear inputs, the first block's input and every block's output,
    the next block's input) and reads its result (the last FFN-down output, Gamma and the
    similarity of every block) back.  The copies run on a second stream into one of two device
    buffer sets (ping-pong by step), in block order with one event per block: block b waits only
    for its own inputs, so the copies of later blocks (and of the next step) overlap the kernels
    of earlier ones."""
    torch = wl.torch
    dev = wl.dev
    stream = torch.cuda.current_stream()
    nb = wl.nblocks
    host_in = {(s, name): t.cpu().pin_memory() for s in range(2) for name, t in wl.inputs[s].items()}
    host_x0 = wl.x_in[0].cpu().pin_memory()
    host_xo = [t.cpu().pin_memory() for t in wl.x_out]
    h2d = sum(t.numel() * t.element_size() for t in list(host_in.values()) + [host_x0] + host_xo)
    out_host = torch.empty_like(wl.y["ffn_down"], device="cpu").pin_memory()
    g_host = torch.empty(2 * nb, dtype=torch.float32).pin_memory()
    d2h = out_host.numel() * out_host.element_size() + g_host.numel() * 4
    orig = {"inputs": wl.inputs, "x_out": wl.x_out, "x_in": wl.x_in}
    x_out1 = [torch.empty_like(t) for t in wl.x_out]
    slots = [orig,
             {"inputs": [{k: torch.empty_like(v) for k, v in st.items()} for st in wl.inputs],
              "x_out": x_out1, "x_in": [torch.empty_like(wl.x_in[0])] + x_out1[:-1]}]
    copy_stream = torch.cuda.Stream(device=dev)
    ready = [[torch.cuda.Event() for _ in range(nb)] for _ in range(2)]
    slot_free = [torch.cuda.Event() for _ in range(2)]
    for ev in slot_free:
        ev.record(stream)
    step_no = [0]

    def e2e_step():
        k = step_no[0] % 2
        sl = slots[k]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(slot_free[k])      # the step that last read this slot is done
            for b in range(nb):
                if b < 2:
                    for name, t in sl["inputs"][b].items():
                        t.copy_(host_in[(b, name)], non_blocking=True)
                if b == 0:
                    sl["x_in"][0].copy_(host_x0, non_blocking=True)
                sl["x_out"][b].copy_(host_xo[b], non_blocking=True)
                ready[k][b].record(copy_stream)
        wl.inputs, wl.x_out, wl.x_in = sl["inputs"], sl["x_out"], sl["x_in"]
        wl.step(before_block=lambda b: stream.wait_event(ready[k][b]))
        slot_free[k].record(stream)
        out_host.copy_(wl.y["ffn_down"], non_blocking=True)
        g_host[:nb].copy_(wl.gamma, non_blocking=True)
        g_host[nb:].copy_(wl.sim, non_blocking=True)
        step_no[0] += 1

    e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    ms = (time.perf_counter() - t0) * 1e3 / steps
    wl.inputs, wl.x_out, wl.x_in = orig["inputs"], orig["x_out"], orig["x_in"]
    del slots, x_out1, host_in, host_x0, host_xo
    torch.cuda.empty_cache()
    return max_over_ranks(ms, world, dev), int(h2d), int(d2h)


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as tdist
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pk, src = peaks()

    def barrier():
        if world > 1:
            tdist.barrier()
        torch.cuda.synchronize()

    wl = Workload(dev, seed=1234 + rank, name=args.workload)
    wl.step()                                   # first warm-up step
    tot, kern_roof = instrumented_kernels(wl, pk)   # second warm-up step, every launch timed
    dominant = max(tot, key=tot.get)
    with Clocks(local_rank) as clk:
        ms, dom_ms = time_steps(wl, args.steps, max(0, args.warmup - 2), world, barrier, dominant, clk)
    e2e_ms, h2d, d2h = e2e_leg(wl, max(1, min(args.steps, 3)), world, barrier)

    extras = {}
    if not args.no_nvfp4_only and rank == 0:
        extras["nvfp4_only_weights"] = run_nvfp4_only_weights(wl)
    if rank != 0:
        return
    units, moved = wl.kernel_units()
    avg_ms = sum(dom_ms) / len(dom_ms)
    n_launch_step = len(dom_ms) / args.steps
    unit_per_launch = units[dominant] / n_launch_step
    if dominant.startswith("gemm"):
        achieved = unit_per_launch / (avg_ms * 1e-3) / 1e12
        if dominant == "gemm_int8":
            peak = pk["bf16_tflops_sustained"]
            peak_note = (f"{src} bf16 sustained: the INT8 codes run exactly on the bf16 tensor pipe "
                         "(sm_103a has no tcgen05 integer MMA)")
        else:
            peak = pk["bf16_tflops_sustained"] * 6.0
            peak_note = f"{src} bf16 sustained x 6 (nominal dense fp4/bf16 ratio)"
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 2), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": measured_traffic(dominant), "kernel": dominant,
                "peak_source": peak_note}
    else:
        achieved = unit_per_launch / (avg_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": measured_traffic(dominant),
                "kernel": dominant, "peak_source": f"{src} HBM copy"}
    value = aggregate_value(wl.flops_step, world, ms)
    e2e_val = aggregate_value(wl.flops_step, world, e2e_ms)
    routes_flat = [r for rr in wl.routes for r in rr]
    spec = wl.spec
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 (e2m1+e4m3) and int8 codes (int32-exact on the bf16 tensor pipe), bf16 activations",
        "data": "synthetic (seeded; CogVideoX-shaped activations with outlier channels, N(0,0.02) weights)",
        "config": {"workload": wl.name, "tokens": spec["tokens"], "hidden": spec["hidden"], "ffn": spec["ffn"],
                   "blocks": wl.nblocks, "activations": spec["activations"], "hadamard_block": HBLOCK,
                   "gamma": "U(0,0.2)", "thr": THR, "int8_layers": routes_flat.count(1),
                   "nvfp4_layers": routes_flat.count(0),
                   "l2": ("inputs larger than L2 in aggregate: each block reads its input (the previous block's "
                          "output), its own output and one of two alternating input sets; a step streams tens of GB, "
                          "so nothing of the previous step is L2-resident when the next starts (no flush)"),
                   "parallelism": f"replicas{world}"},
        "roofline": roof,
        "kernel_ms_per_step": {k: round(v, 3) for k, v in tot.items()},
        "kernel_roofline": kern_roof,
        "e2e": {"value": round(e2e_val, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 3),
                "copies": "pinned host -> device on a copy stream into ping-pong device buffers, one event per "
                          "block; results read back after each step"},
        "gpu_launches": int(wl.launches_per_step() * args.steps),
        "clocks": clk.summary(),
    }
    line.update(extras)
    wl.free()
    del wl
    if not args.no_2b:
        w2 = Workload(dev, seed=4321, name="cogvideox_2b_block_linears")
        w2.step()
        tot2, roof2 = instrumented_kernels(w2, pk)
        ms2, _ = time_steps(w2, max(3, args.steps // 2), 1, 1, lambda: torch.cuda.synchronize())
        line["cogvideox_2b_step"] = {"value": round(w2.flops_step / (ms2 * 1e-3) / 1e12, 3), "unit": UNIT,
                                     "ms_per_step": round(ms2, 3), "blocks": w2.nblocks,
                                     "int8_layers": sum(r.count(1) for r in w2.routes),
                                     "nvfp4_layers": sum(r.count(0) for r in w2.routes),
                                     "kernel_roofline": roof2}
        if not args.no_tdc_loop:
            line["tdc_loop"] = run_tdc_loop(w2, steps=args.tdc_steps, replay_blocks=args.tdc_replay_blocks)
        w2.free()
        del w2
    if not args.no_long:
        line["long_1080p"] = run_long_1080p(dev)
        line["int8_requant_ffn_up"] = run_int8_requant(dev)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------
# CPU oracle baselines (the one place besides the tests that runs the oracle)
# ----------------------------------------------------------------------------------------


_PREP = {}


def _oracle_weights(spec):
    """Both routes' weights of one block, prepared once by the oracle (untimed)."""
    key = spec["hidden"]
    if key not in _PREP:
        import synth
        from oracle import dmpq as D
        _PREP[key] = {name: D.prepare_weight(synth.weights(n, k, seed=5000 + n + k), HBLOCK)
                      for name, k, n in linears(spec)}
    return _PREP[key]


def oracle_sample(tokens: int, seed: int, workload: str = DEFAULT_WORKLOAD):
    """The oracle on a token sample of one block: the four routed linears (alternating
    routes; the FFN-down input is the bf16 GELU of the FFN-up output) + the delta commit.
    Returns (seconds, flops)."""
    import numpy as np
    import synth
    from oracle import dmpq as D
    from oracle import formats as F
    from oracle import tdc as T
    spec = WORKLOADS[workload]
    preps = _oracle_weights(spec)
    act = lambda k, s, dtype: synth.activations(tokens, k, dist=spec["dist"], outlier_frac=spec["outlier_frac"],
                                                outlier_mult=spec["outlier_mult"], seed=s, dtype=dtype)
    xs = {name: act(k, seed + i, "f32") for i, (name, k, _) in enumerate(linears(spec)) if name != "ffn_down"}
    xi = act(spec["hidden"], seed + 9, "bf16")
    xo = synth.gamma_pair(xi, 0.1, seed + 10)
    flops = 0
    t0 = time.perf_counter()
    for i, (name, k, n) in enumerate(linears(spec)):
        route = D.ROUTE_INT8 if i % 2 == 0 else D.ROUTE_NVFP4
        y = D.routed_linear(xs[name], preps[name], HBLOCK, route)
        if name == "ffn_up":
            xs["ffn_down"] = F.bf16_bits_to_f32(F.f32_to_bf16_bits(D.gelu_erf(y).astype(np.float32)))
        flops += 2 * tokens * n * k
    T.tdc_commit(xi, xo, None, "bf16")
    return time.perf_counter() - t0, flops


def cpu_baseline(seconds_budget: float = 15.0, workload: str = DEFAULT_WORKLOAD):
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    tokens, total_t, total_f, reps = 32, 0.0, 0, 0
    while total_t < seconds_budget and reps < 50:
        t, f = oracle_sample(tokens, seed=reps, workload=workload)
        total_t += t
        total_f += f
        reps += 1
        if t < 1.0 and tokens < 2048:
            tokens *= 2
    return {"value": round(total_f / total_t / 1e12, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} oracle passes over one {workload} block (4 routed linears, both routes, GELU "
                      f"+ delta commit) on token samples up to {tokens} tokens; weight preparation untimed; "
                      f"{total_t:.1f} s of CPU work (numpy float64 BLAS on all cores)"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    workload = getattr(args, "workload", DEFAULT_WORKLOAD)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    tokens = 64
    for _ in range(max(0, args.warmup)):
        oracle_sample(16, seed=1, workload=workload)
    total_t, total_f = 0.0, 0
    for s in range(args.steps):
        t, f = oracle_sample(tokens, seed=100 + s, workload=workload)
        total_t += t
        total_f += f
    v = total_f / total_t / 1e12
    sample = (f"each step: the oracle over one {workload} block (4 routed linears, both routes, GELU, + delta "
              f"commit) on a {tokens}-token sample; weight preparation untimed")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_t * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64/int64 (CPU oracle)",
        "data": "synthetic (seeded)", "config": {"workload": workload, "tokens_sample": tokens},
        "cpu_baseline": {"value": round(v, 6), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-2b", action="store_true", help="skip the CogVideoX-2B step (and with it the TDC loop)")
    ap.add_argument("--no-tdc-loop", action="store_true")
    ap.add_argument("--tdc-steps", type=int, default=50)
    ap.add_argument("--tdc-replay-blocks", type=int, default=2)
    ap.add_argument("--no-nvfp4-only", action="store_true", help="skip the NVFP4-only-weights variant")
    ap.add_argument("--no-long", action="store_true", help="skip the 1080p-shaped path")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as tdist
            tdist.destroy_process_group()


if __name__ == "__main__":
    main()
