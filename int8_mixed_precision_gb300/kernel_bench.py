"""Time one libdit6 kernel on one shape (CUDA events, L2 cleaned between repetitions).

  python -m int8_mixed_precision_gb300.kernel_bench --case gemm_nvfp4 --m 17776 --n 5760 --k 1920

Cases: quant_int8, quant_nvfp4 (two passes), quant_nvfp4_given (one pass, tensor scale
given), gamma, tdc_commit, tdc_skip, gemm_int8, gemm_int8_requant, gemm_nvfp4, gemm_nvfp4_amax (the GEMM that
also returns its output's NVFP4 tensor scale), outlier_ratio and gemm_bf16 (the PDR
full-precision route).  Inputs are synthetic bf16 activations (N(0,1), 1% outlier channels
x50) and N(0,0.02) weights.  Prints one JSON line with the median time and the algorithmic
rate (GB/s for streaming kernels at the algorithmic bytes per element -- quantisers: 2 in
+ 1 out + 4 per row for INT8, 2 + 0.5 + 1/16 for NVFP4 -- and TFLOP/s for GEMMs); "moved"
gives the bytes the kernel really reads and writes when they differ (bf16-held INT8 codes,
the NVFP4 amax pass).  Also the small cases used for ncu captures.
"""
from __future__ import annotations

import argparse
import json
import statistics


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", required=True)
    ap.add_argument("--m", type=int, default=17776)
    ap.add_argument("--n", type=int, default=5760)
    ap.add_argument("--k", type=int, default=1920)
    ap.add_argument("--hblock", type=int, default=64)
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--no-flush", action="store_true")
    ap.add_argument("--int8-container", choices=["bf16", "int8"], default="bf16")
    ap.add_argument("--act", choices=["none", "gelu"], default="none", help="GEMM epilogue activation")
    a = ap.parse_args(argv)

    import torch

    import int8_mixed_precision_gb300 as dit
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    ws = dit.workspace(dev)
    m, n, k = a.m, a.n, a.k

    def act(rows, cols):
        x = torch.randn(rows, cols, device=dev, generator=g)
        x[:, torch.randperm(cols, device=dev, generator=g)[: max(1, cols // 100)]] *= 50.0
        return x.to(torch.bfloat16)

    case = a.case
    moved = None
    if case in ("quant_int8", "quant_nvfp4", "quant_nvfp4_given"):
        x = act(m, k)
        if case == "quant_int8":
            q = torch.empty(m, k, dtype=torch.int8 if a.int8_container == "int8" else torch.bfloat16, device=dev)
            s = torch.empty(m, device=dev)
            fn = lambda: dit.hadamard_quant_int8(x, a.hblock, q, s)
            units, unit = m * k * 3 + 4 * m, "GB/s"
            moved = m * k * (2 + q.element_size()) + 4 * m
        else:
            b = dit.alloc_nvfp4(m, k, dev)
            dit.hadamard_quant_nvfp4(x, a.hblock, b["codes"], b["sf"], b["gs"], ws)
            sg = b["gs"].clone() if case == "quant_nvfp4_given" else None
            fn = lambda: dit.hadamard_quant_nvfp4(x, a.hblock, b["codes"], b["sf"], b["gs"], ws, tensor_scale_in=sg)
            units, unit = m * k * 2 + m * k // 2 + m * k // 16, "GB/s"
            moved = units + (0 if sg is not None else m * k * 2)
    elif case in ("gamma", "tdc_commit", "tdc_skip"):
        xi = act(m, k)
        xo = (xi.float() * 1.05).to(torch.bfloat16)
        gam = torch.empty(1, device=dev)
        sim = torch.empty(1, device=dev)
        if case == "gamma":
            r = torch.empty(4, dtype=torch.int32, device=dev)
            fn = lambda: dit.gamma_route(xi, xo, [1.0] * 4, [0.0] * 4, [0.05] * 4, gam, r, ws)
            units = m * k * 4
        elif case == "tdc_commit":
            d1, d2 = torch.zeros_like(xi), torch.empty_like(xi)
            fn = lambda: dit.tdc_step(dit.TDC_COMMIT, xi, ws, x_out=xo, d1=d1, d_new=d2, gamma=gam, sim=sim)
            units = m * k * 8
        else:
            d1, out = torch.zeros_like(xi), torch.empty_like(xi)
            fn = lambda: dit.tdc_step(dit.TDC_SKIP, xi, ws, x_out_skip=out, d1=d1)
            units = m * k * 6
        unit = "GB/s"
    elif case == "gemm_nvfp4_amax":
        # FFN up with GELU whose output feeds an NVFP4 layer: the epilogue also reduces the
        # output's NVFP4 tensor scale (the next quantisation is then one pass)
        x = act(m, k)
        w = torch.randn(n, k, device=dev, generator=g) * 0.02
        lin = dit.RoutedLinear(dit.QuantizedWeight(w, a.hblock, ws), m, ws, dev)
        y = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
        lin(x, dit.ROUTE_NVFP4, y, act=dit.ACT_GELU_ERF)
        nxt = torch.empty(1, dtype=torch.float32, device=dev)
        A, W = lin.a4, lin.w.nvfp4
        fn = lambda: dit.qgemm_nvfp4_amax(A["codes"], A["sf"], A["gs"], W["codes"], W["sf"], W["gs"], y, ws,
                                          a.hblock, nxt, act=dit.ACT_GELU_ERF)
        units, unit = 2 * m * n * k, "TFLOP/s"
    elif case == "gemm_int8_requant":
        # FFN up with GELU whose output feeds an INT8 layer: the epilogue quantises the output
        # with per-token scales supplied (here: the exact ones of an unfused run)
        x = act(m, k)
        w = torch.randn(n, k, device=dev, generator=g) * 0.02
        lin = dit.RoutedLinear(dit.QuantizedWeight(w, a.hblock, ws), m, ws, dev)
        y = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
        lin(x, dit.ROUTE_INT8, y, act=dit.ACT_GELU_ERF)
        s_next = torch.empty(m, dtype=torch.float32, device=dev)
        q_next = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
        dit.hadamard_quant_int8(y, 64, q_next, s_next)
        amax = torch.zeros(m, dtype=torch.float32, device=dev)
        W8 = lin.w.int8
        fn = lambda: dit.qgemm_int8_requant(lin.a8["q"], lin.a8["scale"], W8["q"], W8["scale"], s_next, q_next, amax,
                                            ws, act=dit.ACT_GELU_ERF)
        units, unit = 2 * m * n * k, "TFLOP/s"
    elif case == "outlier_ratio":
        x = act(m, k)
        r = torch.empty(1, dtype=torch.float32, device=dev)
        fn = lambda: dit.outlier_ratio(x, ws, r)
        units, unit = m * k * 2, "GB/s"     # one algorithmic read of the activation (the kernel reads it twice)
    elif case == "gemm_bf16":
        x = act(m, k)
        w = (torch.randn(n, k, device=dev, generator=g) * 0.02).to(torch.bfloat16)
        y = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
        act_code = dit.ACT_GELU_ERF if a.act == "gelu" else dit.ACT_NONE
        fn = lambda: dit.gemm_bf16(x, w, y, ws, act=act_code)
        units, unit = 2 * m * n * k, "TFLOP/s"
    elif case in ("gemm_int8", "gemm_nvfp4"):
        x = act(m, k)
        w = torch.randn(n, k, device=dev, generator=g) * 0.02
        lin = dit.RoutedLinear(dit.QuantizedWeight(w, a.hblock, ws, int8_container=a.int8_container), m, ws, dev)
        y = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
        act_code = dit.ACT_GELU_ERF if a.act == "gelu" else dit.ACT_NONE
        if case == "gemm_int8":
            lin(x, dit.ROUTE_INT8, y)
            fn = lambda: dit.qgemm_int8(lin.a8["q"], lin.a8["scale"], lin.w.int8["q"], lin.w.int8["scale"], y, ws,
                                        act=act_code)
        else:
            lin(x, dit.ROUTE_NVFP4, y)
            fn = lambda: dit.qgemm_nvfp4(lin.a4["codes"], lin.a4["sf"], lin.a4["gs"], lin.w.nvfp4["codes"],
                                         lin.w.nvfp4["sf"], lin.w.nvfp4["gs"], y, ws, act=act_code)
        units, unit = 2 * m * n * k, "TFLOP/s"
    else:
        raise SystemExit(f"unknown case {case}")

    # L2 flush between repetitions: a read sweep over a buffer larger than L2, so that the
    # timed kernel starts with neither its inputs nor dirty lines (whose write-back would
    # otherwise be charged to it) in L2
    flush = None if a.no_flush else torch.ones(640 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for _ in range(a.warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(a.reps):
        if flush is not None:
            flush.max()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    assert dit.device_status(ws) == 0, "device status raised"
    t = statistics.median(times)
    rate = units / (t * 1e-3) / (1e9 if unit == "GB/s" else 1e12)
    out = {"case": case, "m": m, "n": n, "k": k, "median_us": round(t * 1e3, 2),
           "min_us": round(min(times) * 1e3, 2), "rate": round(rate, 2), "unit": unit}
    if moved is not None and moved != units:
        out["moved_gbs"] = round(moved / (t * 1e-3) / 1e9, 2)
    print(json.dumps(out))


if __name__ == "__main__":
    main()
