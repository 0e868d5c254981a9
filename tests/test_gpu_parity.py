"""GPU parity: every kernel of libdit6 against the CPU oracle on the same seeded inputs.

Stage-wise: each oracle stage consumes the GPU's own input to that stage.  Codes, scales,
int32 accumulators, deltas and decisions are bit-exact (codes and scales up to elements
within 1e-5 relative of a rounding boundary); fp outputs of the NVFP4 GEMM within 1e-3
relative Frobenius of the float64 oracle.
"""
import math
import os

import numpy as np
import pytest

import synth
from gpu_helpers import (as_f32, check_int8, check_nvfp4, dev_bf16, dev_f32, host, make_x,
                         rel_fro)
from oracle import dmpq as D
from oracle import formats as F
from oracle import tdc as T

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import int8_mixed_precision_gb300 as dit  # noqa: E402

GEMM_TOL = 1e-3


@pytest.fixture(scope="module")
def ws():
    return dit.workspace()


def _status_clean(ws):
    torch.cuda.synchronize()
    assert dit.device_status(ws) == 0


# ------------------------------------------------------------------------------ quantisers


@pytest.mark.parametrize("rows,k,dtype,hb", [
    (256, 128, "f32", 16),        # the single-linear workload
    (300, 1920, "bf16", 64),      # ragged rows, CogVideoX-2B hidden
    (129, 7680, "bf16", 64),      # FFN-down width
    (7, 3072, "bf16", 32),
    (1, 12288, "bf16", 64),
    (5003, 1920, "bf16", 64),     # thousands of row groups, ragged tail
    (1203, 12288, "bf16", 16),
    (3, 16384, "bf16", 64),       # the widest row the quantiser takes (256 units, one CTA)
])
@pytest.mark.parametrize("container", [torch.int8, torch.bfloat16])
def test_int8_quant_parity(rows, k, dtype, hb, container):
    x, xd = make_x(rows, k, dtype, seed=rows + k)
    q = torch.empty(rows, k, dtype=container, device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    dit.hadamard_quant_int8(xd, hb, q, s)
    qh = host(q) if container == torch.int8 else F.bf16_bits_to_f32(host(q))
    if container == torch.bfloat16:
        assert np.array_equal(qh, np.rint(qh)) and np.abs(qh).max() <= 127
        qh = qh.astype(np.int8)
    n_ex, _ = check_int8(qh, host(s), x, dtype, hb)
    assert n_ex <= max(2, q.numel() // 10000)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_int8_quant_zero_and_constant_rows(dtype):
    x = np.zeros((5, 128), np.float32)
    x[1] = 3.0
    x[2, 7] = -1e-3
    x[4] = np.linspace(-2, 2, 128, dtype=np.float32)
    xin = x if dtype == "f32" else F.f32_to_bf16_bits(x)
    q = torch.empty(5, 128, dtype=torch.int8, device="cuda")
    s = torch.empty(5, dtype=torch.float32, device="cuda")
    dit.hadamard_quant_int8(dev_f32(x) if dtype == "f32" else dev_bf16(xin), 16, q, s)
    check_int8(host(q), host(s), xin, dtype, 16)
    assert host(s)[0] == 0 and not host(q)[0].any()


@pytest.mark.parametrize("rows,k,dtype,hb", [
    (256, 128, "f32", 16),
    (300, 1920, "bf16", 64),
    (129, 7680, "bf16", 64),
    (7, 3072, "bf16", 32),
    (1000, 3072, "bf16", 64),
    (4100, 1920, "bf16", 64),     # several grid-stride passes per thread, ragged 128-row tail
    (2051, 640, "f32", 32),
])
def test_nvfp4_quant_parity(rows, k, dtype, hb, ws):
    x, xd = make_x(rows, k, dtype, seed=3 * rows + k, dist="laplace" if k == 3072 else "normal")
    buf = dit.alloc_nvfp4(rows, k)
    buf["sf"].fill_(0xAB)     # padding must be overwritten with zeros
    dit.hadamard_quant_nvfp4(xd, hb, buf["codes"], buf["sf"], buf["gs"], ws)
    _status_clean(ws)
    _, n_ex = check_nvfp4(host(buf["codes"]), host(buf["sf"]), host(buf["gs"])[0], x, dtype, hb, rows, k)
    assert n_ex <= max(2, rows * k // 10000)


def test_nvfp4_quant_given_tensor_scale_and_repeat(ws):
    rows, k = 200, 1920
    x, xd = make_x(rows, k, "bf16", seed=77)
    buf = dit.alloc_nvfp4(rows, k)
    sg_in = torch.tensor([0.004], dtype=torch.float32, device="cuda")   # small: forces saturation
    dit.hadamard_quant_nvfp4(xd, 64, buf["codes"], buf["sf"], buf["gs"], ws, tensor_scale_in=sg_in)
    check_nvfp4(host(buf["codes"]), host(buf["sf"]), host(buf["gs"])[0], x, "bf16", 64, rows, k,
                s_g=np.float32(0.004))
    # the dynamic path twice in a row (the workspace must come back to its reusable state)
    for _ in range(2):
        dit.hadamard_quant_nvfp4(xd, 64, buf["codes"], buf["sf"], buf["gs"], ws)
        check_nvfp4(host(buf["codes"]), host(buf["sf"]), host(buf["gs"])[0], x, "bf16", 64, rows, k)
    _status_clean(ws)


def test_nvfp4_quant_zero_tensor(ws):
    x = np.zeros((130, 128), np.float32)
    buf = dit.alloc_nvfp4(130, 128)
    dit.hadamard_quant_nvfp4(dev_f32(x), 16, buf["codes"], buf["sf"], buf["gs"], ws)
    assert host(buf["gs"])[0] == 0 and not host(buf["codes"]).any() and not host(buf["sf"]).any()


def test_e2m1_negative_zero_convention(ws):
    """Tiny negative values in a block with a large element: the hardware convert and the
    oracle agree on the sign of the zero code."""
    x = np.zeros((1, 64), np.float32)
    x[0, :16] = [6.0, -0.01, 0.01, -0.2, 0.2, -0.26, 0.26, -0.0, 0.0, -1e-30, 3, -3, 0.74, -0.76, 5, -5]
    sg = torch.tensor([1.0], dtype=torch.float32, device="cuda")
    buf = dit.alloc_nvfp4(1, 64)
    # hblock 16 on a one-hot pattern would mix values; quantise the raw row by undoing the
    # transform: H(H x)/16 = x, so feeding H x / 4 gives back x after the block transform
    xh = D.block_fwht_f32(x, 16).astype(np.float32)
    dit.hadamard_quant_nvfp4(dev_f32(xh), 16, buf["codes"], buf["sf"], buf["gs"], ws, tensor_scale_in=sg)
    check_nvfp4(host(buf["codes"]), host(buf["sf"]), 1.0, xh, "f32", 16, 1, 64, s_g=np.float32(1.0))


# ------------------------------------------------------------------------------ Gamma / TDC


@pytest.mark.parametrize("n,dtype", [(256 * 128, "f32"), (17776 * 64 + 5, "bf16"), (33, "bf16")])
def test_gamma_route_parity(n, dtype, ws):
    g = synth.rng(n)
    xi = g.standard_normal(n).astype(np.float32)
    xo = (xi + g.standard_normal(n).astype(np.float32) * 0.07).astype(np.float32)
    if dtype == "bf16":
        xi, xo = synth.to_bf16_bits(xi), synth.to_bf16_bits(xo)
        di, do = dev_bf16(xi), dev_bf16(xo)
    else:
        di, do = dev_f32(xi), dev_f32(xo)
    alpha, beta, thr = [1.0, 0.5, 2.0, 1.0], [0.0, 0.0, 0.0, 0.02], [0.05, 0.05, 0.05, 0.05]
    gam = torch.empty(1, dtype=torch.float32, device="cuda")
    routes = torch.empty(4, dtype=torch.int32, device="cuda")
    dit.gamma_route(di, do, alpha, beta, thr, gam, routes, ws)
    ref = D.gamma_rel_l1(as_f32(xi, dtype), as_f32(xo, dtype))
    got = float(host(gam)[0])
    assert got == pytest.approx(ref, rel=1e-5)
    want = D.route_layers(ref, alpha, beta, np.float32(thr).astype(np.float64))
    margins = [D.route_margin(ref, a, b, t) for a, b, t in zip(alpha, beta, thr)]
    for r, w, m in zip(host(routes).tolist(), want, margins):
        assert r == w or m <= 1e-5
    # deterministic across runs
    dit.gamma_route(di, do, alpha, beta, thr, gam, routes, ws)
    assert float(host(gam)[0]) == got
    _status_clean(ws)


def test_gamma_single_linear_routes_int8(ws):
    c = synth.single_linear()
    gam = torch.empty(1, dtype=torch.float32, device="cuda")
    routes = torch.empty(1, dtype=torch.int32, device="cuda")
    dit.gamma_route(dev_f32(c["x"]), dev_f32(c["x_out"]), [1.0], [0.0], [0.05], gam, routes, ws)
    assert float(host(gam)[0]) == pytest.approx(D.gamma_rel_l1(c["x"], c["x_out"]), rel=1e-5)
    assert host(routes).tolist() == [dit.ROUTE_INT8]


@pytest.mark.parametrize("n,dtype", [(17776 * 16 + 3, "bf16"), (4096 + 5, "f32")])
def test_tdc_commit_and_skip_parity(n, dtype, ws):
    g = synth.rng(n + 1)
    xi32 = g.standard_normal(n).astype(np.float32)
    d_prev32 = (g.standard_normal(n) * 0.1).astype(np.float32)
    xo32 = (xi32 + d_prev32 * (1 + g.standard_normal(n).astype(np.float32) * 0.01)).astype(np.float32)
    conv = synth.to_bf16_bits if dtype == "bf16" else (lambda a: a)
    dev = dev_bf16 if dtype == "bf16" else dev_f32
    xi, xo, dp = conv(xi32), conv(xo32), conv(d_prev32)
    di, do, ddp = dev(xi), dev(xo), dev(dp)
    dnew = torch.empty_like(di)
    gam = torch.empty(1, dtype=torch.float32, device="cuda")
    sim = torch.empty(1, dtype=torch.float32, device="cuda")
    dit.tdc_step(dit.TDC_COMMIT, di, ws, x_out=do, d1=ddp, d_new=dnew, gamma=gam, sim=sim)
    ref = T.tdc_commit(xi, xo, dp, dtype)
    assert np.array_equal(host(dnew), ref["delta"])
    assert float(host(gam)[0]) == pytest.approx(ref["gamma"], rel=1e-5)
    assert float(host(sim)[0]) == pytest.approx(ref["d"], rel=1e-5)
    # no previous delta: similarity is +inf
    dit.tdc_step(dit.TDC_COMMIT, di, ws, x_out=do, d1=None, d_new=dnew, gamma=gam, sim=sim)
    assert math.isinf(float(host(sim)[0]))
    # skip: x_in + cached delta, bit-exact
    out = torch.empty_like(di)
    dit.tdc_step(dit.TDC_SKIP, di, ws, x_out_skip=out, d1=dnew)
    assert np.array_equal(host(out), T.tdc_skip(xi, ref["delta"], dtype))
    _status_clean(ws)


def test_tdc_loop_decisions_match_oracle(ws):
    """A 12-step, 3-block delta-cache loop: decisions and routes identical to the oracle."""
    rows, k, steps, tau = 64, 256, 12, 0.05
    alpha, beta, thr = [1.0] * 4, [0.0] * 4, [0.05] * 4
    for b in range(3):
        deltas, _ = synth.tdc_deltas(steps, rows, k, seed=100 + b, jump_every=5.0)
        xs = [synth.activations(rows, k, seed=1000 * b + t, outlier_frac=0.0) for t in range(steps)]
        ref = T.run_block_loop(xs, deltas, tau, alpha, beta, np.float32(thr).astype(np.float64))
        st = dit.TdcState()
        d1 = torch.empty(rows * k, dtype=torch.bfloat16, device="cuda")
        d2 = torch.empty_like(d1)
        gam = torch.empty(1, dtype=torch.float32, device="cuda")
        sim = torch.empty(1, dtype=torch.float32, device="cuda")
        decisions, routes = [], []
        for t in range(steps):
            mode = st.decide(tau)
            xi = dev_bf16(xs[t]).reshape(-1)
            if mode == dit.TDC_SKIP:
                out = torch.empty_like(xi)
                dit.tdc_step(dit.TDC_SKIP, xi, ws, x_out_skip=out, d1=d1)
                assert np.array_equal(host(out), ref["outs"][t].reshape(-1))
                decisions.append("skip")
                routes.append(None)
                st.update(dit.TDC_SKIP)
                continue
            routes.append(st.routes(alpha, beta, thr))
            xo32 = (F.bf16_bits_to_f32(xs[t]) + F.bf16_bits_to_f32(deltas[t])).astype(np.float32)
            xo = dev_bf16(F.f32_to_bf16_bits(xo32)).reshape(-1)
            has_prev = st.n_computed > 0
            dit.tdc_step(dit.TDC_COMMIT, xi, ws, x_out=xo, d1=d1 if has_prev else None, d_new=d2,
                         gamma=gam, sim=sim)
            torch.cuda.synchronize()
            st.update(dit.TDC_COMMIT, float(host(gam)[0]), float(host(sim)[0]) if has_prev else None)
            d1, d2 = d2, d1
            decisions.append("compute")
        for t in range(steps):
            if ref["margins"][t] > 1e-5:
                assert decisions[t] == ref["decisions"][t], (b, t, decisions, ref["decisions"])
        for t in range(steps):
            if ref["margins"][t] <= 1e-5 or decisions[t] != ref["decisions"][t]:
                continue
            g_ref = ref["gammas"][t]
            if g_ref is not None and abs(g_ref - 0.05) <= 1e-5 * 0.05:
                continue        # borderline route
            assert routes[t] == ref["routes"][t], (b, t, routes[t], ref["routes"][t])


# ------------------------------------------------------------------------------ GEMMs


def _int8_dev(a, container):
    t = torch.from_numpy(a).cuda()
    return t if container == torch.int8 else t.to(torch.bfloat16)


@pytest.mark.parametrize("container", [torch.int8, torch.bfloat16])
@pytest.mark.parametrize("m,n,k", [(256, 512, 128), (300, 384, 1920), (129, 256, 7680), (1, 8, 16),
                                   (200, 136, 208), (700, 5760 // 10, 2112)])
def test_int8_gemm_exact_accumulators(m, n, k, container, ws):
    """int8-held codes run on IMMA, bf16-held codes on the CTA-pair tcgen05 kernel: both give the
    int64 oracle's accumulators bit for bit."""
    g = synth.rng(m * n + k)
    a = g.integers(-127, 128, (m, k)).astype(np.int8)
    b = g.integers(-127, 128, (n, k)).astype(np.int8)
    sa = g.random(m).astype(np.float32) * 0.01
    sb = g.random(n).astype(np.float32) * 0.01
    bias = g.standard_normal(n).astype(np.float32)
    ta, tb = _int8_dev(a, container), _int8_dev(b, container)
    acc = torch.empty(m, n, dtype=torch.int32, device="cuda")
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    dit.qgemm_int8(ta, dev_f32(sa), tb, dev_f32(sb), y, ws, bias=dev_f32(bias), acc_debug=acc)
    ref_acc = D.gemm_int8_acc(a, b)
    assert np.array_equal(host(acc).astype(np.int64), ref_acc)
    ref = D.gemm_int8(a, sa, b, sb, bias)
    assert rel_fro(host(y), ref) <= 1e-6
    yb = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    dit.qgemm_int8(ta, dev_f32(sa), tb, dev_f32(sb), yb, ws, bias=dev_f32(bias))
    assert rel_fro(F.bf16_bits_to_f32(host(yb)), F.bf16_bits_to_f32(F.f32_to_bf16_bits(ref.astype(np.float32)))) <= GEMM_TOL
    # GELU (erf form) in the epilogue: fp32 pre-activation, x * Phi(x) before the store
    dit.qgemm_int8(ta, dev_f32(sa), tb, dev_f32(sb), y, ws, bias=dev_f32(bias), act=dit.ACT_GELU_ERF)
    assert rel_fro(host(y), D.gelu_erf(ref)) <= 2e-6
    _status_clean(ws)


@pytest.mark.parametrize("container", [torch.int8, torch.bfloat16])
def test_gelu_epilogue_elementwise_error_bound(container, ws):
    """GELU in the epilogue over pre-activations spread across [-9, 9] (tails included):
    every output within |x| * 2.5e-6 of x * Phi(x) in float64, x being the kernel's own fp32
    pre-activation (acc * row scale) * column scale."""
    m, n, k = 384, 256, 16
    a = np.zeros((m, k), np.int8)
    a[:, 0] = 1
    b = np.zeros((n, k), np.int8)
    b[:, 0] = np.linspace(-127, 127, n).round().astype(np.int8)
    sa = np.linspace(1e-3, 1.0, m).astype(np.float32)
    sb = np.full(n, 9.0 / 127.0, np.float32)
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    dit.qgemm_int8(_int8_dev(a, container), dev_f32(sa), _int8_dev(b, container), dev_f32(sb), y, ws,
                   act=dit.ACT_GELU_ERF)
    _status_clean(ws)
    x = (D.gemm_int8_acc(a, b).astype(np.float32) * sa[:, None]).astype(np.float32) * sb[None, :]
    x = x.astype(np.float32)
    err = np.abs(host(y).astype(np.float64) - D.gelu_erf(x))
    assert (err <= 2.5e-6 * np.abs(x) + 1e-37).all(), float(np.max(err / np.maximum(np.abs(x), 1e-30)))
    assert host(y)[x == 0].tolist() == [0.0] * int((x == 0).sum())


@pytest.mark.parametrize("m,n,k", [(2560, 1920, 4096), (17776, 1920, 7680), (640, 1920, 12288), (300, 384, 4160)])
def test_int8_gemm_many_tiles_per_pair_bit_exact(m, n, k, ws):
    """Shapes with more 256 x 256 tiles than CTA pairs (each pair walks several tiles, the chunk
    buffers alternate across tile boundaries) and deep K: sampled rows of the accumulators equal
    the int64 oracle, and the GELU output equals the epilogue's arithmetic on those integers."""
    g = synth.rng(m + n + k + 1)
    a = g.integers(-127, 128, (m, k)).astype(np.int8)
    b = g.integers(-127, 128, (n, k)).astype(np.int8)
    sa = (g.random(m) * 0.01).astype(np.float32)
    sb = (g.random(n) * 0.01).astype(np.float32)
    ta, tb = _int8_dev(a, torch.bfloat16), _int8_dev(b, torch.bfloat16)
    acc = torch.empty(m, n, dtype=torch.int32, device="cuda")
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    dit.qgemm_int8(ta, dev_f32(sa), tb, dev_f32(sb), y, ws, acc_debug=acc, act=dit.ACT_GELU_ERF)
    _status_clean(ws)
    rows = np.unique(np.concatenate([synth.rng(m).choice(m, 24, replace=False), [0, m - 1]]))
    ref = D.gemm_int8_acc(a[rows], b)
    assert np.array_equal(host(acc[torch.from_numpy(rows).cuda()]).astype(np.int64), ref)
    x = (ref.astype(np.float32) * sa[rows, None]).astype(np.float32) * sb[None, :]
    err = np.abs(host(y[torch.from_numpy(rows).cuda()]).astype(np.float64) - D.gelu_erf(x.astype(np.float32)))
    assert (err <= 2.5e-6 * np.abs(x) + 1e-37).all()


@pytest.mark.parametrize("m,n,k", [(600, 3584, 4096), (300, 9216, 3072)])
def test_int8_gemm_banded_tile_order_exact(m, n, k, ws):
    """K <= 4096 with more N tiles than one band holds (bands of 24 MB of B: 12 tiles at K = 4096,
    16 at K = 3072): the banded walk over the tiles, with a ragged last band and ragged M, gives
    the int64 oracle's accumulators on sampled rows and every column."""
    g = synth.rng(m * 7 + n + k)
    a = g.integers(-127, 128, (m, k)).astype(np.int8)
    b = g.integers(-127, 128, (n, k)).astype(np.int8)
    sa = (g.random(m) * 0.01).astype(np.float32)
    sb = (g.random(n) * 0.01).astype(np.float32)
    acc = torch.empty(m, n, dtype=torch.int32, device="cuda")
    y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    dit.qgemm_int8(_int8_dev(a, torch.bfloat16), dev_f32(sa), _int8_dev(b, torch.bfloat16), dev_f32(sb), y, ws,
                   acc_debug=acc, act=dit.ACT_GELU_ERF)
    _status_clean(ws)
    rows = np.unique(np.concatenate([synth.rng(m + 1).choice(m, 12, replace=False), [0, 255, 256, m - 1]]))
    ref = D.gemm_int8_acc(a[rows], b)
    assert np.array_equal(host(acc[torch.from_numpy(rows).cuda()]).astype(np.int64), ref)


# INT8 GEMM shapes whose tile count leaves the last wave of CTA pairs partly empty (one or two
# full waves plus a few tiles) or gives fewer tiles than pairs.  The shapes follow the SM count,
# so that they hit those cases on any GB300 part.
PAIRS = torch.cuda.get_device_properties(0).multi_processor_count // 2
WAVE_SHAPES = [
    (((PAIRS + 12 + 7) // 8) * 256 - 77, 8 * 256 - 40, 1040),      # one wave + 12 tiles, ragged M, N, K
    (((2 * PAIRS + 4 + 3) // 4) * 256, 4 * 256, 3072),             # two waves + 4 tiles
    (((PAIRS + 12 + 7) // 8) * 256 - 77, 8 * 256 - 40, 12288),     # deep K: several exact chunks per piece
    (5 * 256 - 1, 6 * 256, 12288),                                 # 30 tiles: fewer than the pairs
]


def _rows_meeting_every_tile(m):
    """One row per (256-row tile, CTA of the pair, 32-row lane quarter), at varying lanes."""
    rows = [mt * 256 + r * 128 + q * 32 + (7 * mt + 5 * q + 3 * r) % 32
            for mt in range((m + 255) // 256) for r in range(2) for q in range(4)]
    return np.unique(np.array([x for x in rows if x < m] + [m - 1]))


@pytest.mark.parametrize("m,n,k", WAVE_SHAPES)
def test_int8_gemm_partial_last_wave_exact(m, n, k, ws):
    """The int64 oracle's accumulators on rows that meet every tile, and the exact product
    everywhere; the output with and without the raw accumulators requested is the same bit for
    bit and equals the epilogue's arithmetic on the exact integers."""
    g = synth.rng(m * 3 + n * 5 + k)
    a = g.integers(-127, 128, (m, k)).astype(np.int8)
    b = g.integers(-127, 128, (n, k)).astype(np.int8)
    sa = (g.random(m) * 0.01).astype(np.float32)
    sb = (g.random(n) * 0.01).astype(np.float32)
    ta, tb = _int8_dev(a, torch.bfloat16), _int8_dev(b, torch.bfloat16)
    acc = torch.empty(m, n, dtype=torch.int32, device="cuda")
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    y2 = torch.empty_like(y)
    dit.qgemm_int8(ta, dev_f32(sa), tb, dev_f32(sb), y, ws, acc_debug=acc)
    dit.qgemm_int8(ta, dev_f32(sa), tb, dev_f32(sb), y2, ws)
    _status_clean(ws)
    rows = _rows_meeting_every_tile(m)
    ref = D.gemm_int8_acc(a[rows], b)
    got = host(acc).astype(np.int64)
    assert np.array_equal(got[rows], ref)
    # everywhere: the float64 product of the codes is exact here (|acc| <= k * 127^2 < 2^53);
    # it agrees with the oracle on the rows above
    full = a.astype(np.float64) @ b.astype(np.float64).T
    assert np.array_equal(full[rows], ref.astype(np.float64))
    assert np.array_equal(got.astype(np.float64), full)
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))
    x = (ref.astype(np.float32) * sa[rows, None]).astype(np.float32) * sb[None, :]
    assert np.array_equal(host(y)[rows], x)


@pytest.mark.parametrize("shape", [0, 1])
def test_int8_gemm_timeout_recovers_on_every_pair(shape, monkeypatch):
    """A GEMM on every CTA pair whose producers issue no loads: all the pairs' waits run out,
    DIT_ERR_TIMEOUT is raised, and the same workspace then serves two normal calls with exact
    results."""
    import time
    ws2 = dit.workspace()
    m, n, k = WAVE_SHAPES[shape]
    g = synth.rng(77)
    a = g.integers(-127, 128, (m, k)).astype(np.int8)
    b = g.integers(-127, 128, (n, k)).astype(np.int8)
    sa, sb = np.ones(m, np.float32), np.ones(n, np.float32)
    ta, tb = _int8_dev(a, torch.bfloat16), _int8_dev(b, torch.bfloat16)
    acc = torch.empty(m, n, dtype=torch.int32, device="cuda")
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    call = lambda: dit.qgemm_int8(ta, dev_f32(sa), tb, dev_f32(sb), y, ws2, acc_debug=acc)
    monkeypatch.setenv("DIT6_TEST_STALL_PRODUCER", "1")
    t0 = time.time()
    call()
    torch.cuda.synchronize()
    assert time.time() - t0 < 30.0
    assert dit.device_status(ws2) & (1 << 5), "DIT_ERR_TIMEOUT not raised"
    monkeypatch.delenv("DIT6_TEST_STALL_PRODUCER")
    dit.clear_device_status(ws2)
    full = a.astype(np.float64) @ b.astype(np.float64).T
    rows = _rows_meeting_every_tile(m)
    assert np.array_equal(full[rows], D.gemm_int8_acc(a[rows], b).astype(np.float64))
    for _ in range(2):
        acc.zero_()
        call()
        torch.cuda.synchronize()
        assert dit.device_status(ws2) == 0
        assert np.array_equal(host(acc).astype(np.float64), full)


@pytest.mark.parametrize("m,n,k,act,with_bias", [(300, 9216, 3072, 1, False), (777, 2048, 1920, 0, True),
                                                  (1030, 4096, 4096, 1, True)])
def test_int8_requant_epilogue(m, n, k, act, with_bias, ws):
    """The INT8 GEMM whose epilogue quantises its output for the next INT8 layer: given the
    exact per-token scales of that output (from the unfused path: GEMM to bf16, then the INT8
    quantiser) its codes are the quantiser's bit for bit and its row maxima give the same
    scales; given half those scales (delayed scales that are too small) the codes are the
    oracle's given-scale quantisation of the oracle's transform of the stored output."""
    g = synth.rng(m + 3 * n + k)
    a = g.integers(-127, 128, (m, k)).astype(np.int8)
    b = g.integers(-127, 128, (n, k)).astype(np.int8)
    sa = (g.random(m) * 0.002 + 1e-4).astype(np.float32)
    sb = (g.random(n) * 0.002 + 1e-4).astype(np.float32)
    bias = dev_f32(g.standard_normal(n).astype(np.float32)) if with_bias else None
    ta, tb = _int8_dev(a, torch.bfloat16), _int8_dev(b, torch.bfloat16)
    act_code = dit.ACT_GELU_ERF if act else dit.ACT_NONE
    y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    dit.qgemm_int8(ta, dev_f32(sa), tb, dev_f32(sb), y, ws, bias=bias, act=act_code)
    q_ref = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    s_ref = torch.empty(m, dtype=torch.float32, device="cuda")
    dit.hadamard_quant_int8(y, 64, q_ref, s_ref)
    q = torch.empty_like(q_ref)
    amax = torch.zeros(m, dtype=torch.float32, device="cuda")
    dit.qgemm_int8_requant(ta, dev_f32(sa), tb, dev_f32(sb), s_ref, q, amax, ws, bias=bias, act=act_code)
    _status_clean(ws)
    assert torch.equal(q.view(torch.int16), q_ref.view(torch.int16))
    s_from_amax = (host(amax).astype(np.float32) / np.float32(127.0)).astype(np.float32)
    assert np.array_equal(s_from_amax.view(np.uint32), host(s_ref).view(np.uint32))
    # delayed scales that are too small: saturation, against the oracle on sampled rows
    half = (s_ref * 0.5).contiguous()
    q2 = torch.empty_like(q_ref)
    amax2 = torch.zeros_like(amax)
    dit.qgemm_int8_requant(ta, dev_f32(sa), tb, dev_f32(sb), half, q2, amax2, ws, bias=bias, act=act_code)
    _status_clean(ws)
    assert torch.equal(amax2, amax)
    rows = np.unique(np.concatenate([synth.rng(m + 5).choice(m, 16, replace=False), [0, m - 1]]))
    z = F.bf16_bits_to_f32(host(y)[rows])                   # the output as the unfused path stores it
    yt = D.block_fwht_f32(z, 64)
    want = D.quant_int8_rows_given(yt, host(half)[rows])
    assert np.array_equal(F.bf16_bits_to_f32(host(q2)[rows]).astype(np.int64), want.astype(np.int64))
    assert (np.abs(want) == 127).any()                      # the half scales do saturate


def _adversarial_int8(m, n, k, seed):
    """Operands that push every exact-chunk partial sum towards its 2^24 bound, mix huge and
    unit products after a large running sum, and cancel."""
    g = synth.rng(seed)
    a = np.full((m, k), 127, np.int8)
    b = np.full((n, k), 127, np.int8)
    b[1::2] = -127                                     # all-negative rows
    a[2, :] = g.choice([-127, 127], size=k)            # random signs: cancellation
    b[3, k // 2:] = 1                                  # unit products after a large sum
    a[4, ::7] = -1
    a[5] = g.integers(-127, 128, k)
    b[5] = g.integers(-127, 128, k)
    return a, b


@pytest.mark.parametrize("k", [1024, 1040, 2048, 7680, 12288])
def test_int8_gemm_bf16_pipe_exact_at_the_bound(k, ws):
    """Extreme codes (+-127 everywhere, totals up to 12288 * 127^2 ~ 2^27.6): the chunked fp32
    accumulation on the bf16 tensor pipe still gives the exact int32 accumulators."""
    m, n = 200, 392
    a, b = _adversarial_int8(m, n, k, seed=k)
    acc = torch.empty(m, n, dtype=torch.int32, device="cuda")
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    ones_m = torch.ones(m, dtype=torch.float32, device="cuda")
    ones_n = torch.ones(n, dtype=torch.float32, device="cuda")
    dit.qgemm_int8(_int8_dev(a, torch.bfloat16), ones_m, _int8_dev(b, torch.bfloat16), ones_n, y, ws, acc_debug=acc)
    assert np.array_equal(host(acc).astype(np.int64), D.gemm_int8_acc(a, b))
    _status_clean(ws)


def _nvfp4_operands(m, n, k, seed):
    g = synth.rng(seed)
    ya = (g.standard_normal((m, k)) * np.exp(g.standard_normal((m, 1)) * 0.5)).astype(np.float32)
    yb = (g.standard_normal((n, k)) * 0.02).astype(np.float32)
    qa, qb = D.quant_nvfp4(ya), D.quant_nvfp4(yb)
    out = []
    for q, rows in ((qa, m), (qb, n)):
        out.append({"codes": torch.from_numpy(D.pack_e2m1(q["codes"])).cuda(),
                    "sf": torch.from_numpy(F.sf_to_tiled(q["sf"], rows, k)).cuda(),
                    "gs": torch.tensor([float(q["s_g"])], dtype=torch.float32, device="cuda")})
    return qa, qb, out[0], out[1]


@pytest.mark.parametrize("m,n,k", [(256, 512, 128), (300, 384, 1920), (129, 256, 7680), (128, 128, 64),
                                   (77, 136, 320), (129, 384, 4096), (4096, 2688, 1024), (8192, 2048, 256)])
def test_nvfp4_gemm_parity(m, n, k, ws):
    """Each shape runs three outputs (fp32; bf16 with bias; fp32 with bias and GELU), which between
    them reach every tile configuration the call picks: 128 x 128 tiles (fp32 with K < 3072 or N
    off the 256 grid; bf16 with N off the 256 grid and K >= 4096), 128 x 256 tiles with eight
    epilogue warps (bf16; fp32 with K >= 3072 and N on the 256 grid) and with sixteen (GELU).
    The last N tile of N = 384, 136 and 2688 holds at most 128 columns (half-tile MMAs); the two
    large shapes give every CTA several tiles, so the accumulator halves change hands across tile
    boundaries, with one K stage (K = 256) and with four (K = 1024)."""
    qa, qb, A, B = _nvfp4_operands(m, n, k, seed=m + n + k)
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    dit.qgemm_nvfp4(A["codes"], A["sf"], A["gs"], B["codes"], B["sf"], B["gs"], y, ws)
    _status_clean(ws)
    ref = D.gemm_nvfp4(qa["codes"], qa["sf"], qa["s_g"], qb["codes"], qb["sf"], qb["s_g"])
    err = rel_fro(host(y), ref)
    assert err <= GEMM_TOL, f"rel Frobenius {err:.3e}"
    yb = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    bias = torch.linspace(-1, 1, n, device="cuda", dtype=torch.float32)
    dit.qgemm_nvfp4(A["codes"], A["sf"], A["gs"], B["codes"], B["sf"], B["gs"], yb, ws, bias=bias)
    refb = F.bf16_bits_to_f32(F.f32_to_bf16_bits((ref + host(bias)[None, :]).astype(np.float32)))
    assert rel_fro(F.bf16_bits_to_f32(host(yb)), refb) <= GEMM_TOL
    dit.qgemm_nvfp4(A["codes"], A["sf"], A["gs"], B["codes"], B["sf"], B["gs"], y, ws, bias=bias,
                    act=dit.ACT_GELU_ERF)
    _status_clean(ws)
    assert rel_fro(host(y), D.gelu_erf(ref + host(bias)[None, :])) <= GEMM_TOL


@pytest.mark.parametrize("m,n,k,hb,act", [(300, 512, 320, 64, 1), (256, 384, 128, 32, 0), (129, 768, 1920, 16, 1),
                                          (77, 128, 64, 64, 1), (1000, 1024, 640, 64, 0)])
def test_nvfp4_gemm_output_tensor_scale(m, n, k, hb, act, ws):
    """The GEMM that also returns its output's NVFP4 tensor scale: y is byte-identical to
    dit_qgemm_nvfp4's, the scale equals the oracle's max|H y| / (6 * 448) over y as stored, and
    the one-pass quantisation with it equals the two-pass one byte for byte."""
    qa, qb, A, B = _nvfp4_operands(m, n, k, seed=5 * m + n + k)
    bias = torch.linspace(-1, 1, n, device="cuda", dtype=torch.float32) if act else None
    y_ref = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    dit.qgemm_nvfp4(A["codes"], A["sf"], A["gs"], B["codes"], B["sf"], B["gs"], y_ref, ws, bias=bias, act=act)
    y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    sc = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    for _ in range(2):  # twice: the workspace's amax word and ticket come back reset
        dit.qgemm_nvfp4_amax(A["codes"], A["sf"], A["gs"], B["codes"], B["sf"], B["gs"], y, ws, hb, sc, bias=bias,
                             act=act)
        _status_clean(ws)
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
        ref_sg = D.nvfp4_tensor_scale(D.block_fwht_f32(F.bf16_bits_to_f32(host(y)), hb))
        assert host(sc)[0] == np.float32(ref_sg)
    two, one = dit.alloc_nvfp4(m, n), dit.alloc_nvfp4(m, n)
    dit.hadamard_quant_nvfp4(y, hb, two["codes"], two["sf"], two["gs"], ws)
    dit.hadamard_quant_nvfp4(y, hb, one["codes"], one["sf"], one["gs"], ws, tensor_scale_in=sc)
    _status_clean(ws)
    assert torch.equal(one["codes"], two["codes"]) and torch.equal(one["sf"], two["sf"])
    assert one["gs"].view(torch.int32).item() == two["gs"].view(torch.int32).item()


def test_nvfp4_gemm_output_tensor_scale_full_size(ws):
    """CogVideoX-2B FFN-up at full size (17776 x 1920 -> 7680, GELU): the returned scale is the
    one the two-pass quantiser derives from the same output, bit for bit."""
    m, k, n, hb = synth.TOKENS_2B, 1920, 7680, 64
    x, xd = make_x(m, k, "bf16", seed=71)
    wq = dit.QuantizedWeight(dev_f32(synth.weights(n, k, seed=72)), hb, ws)
    a4 = dit.alloc_nvfp4(m, k)
    dit.hadamard_quant_nvfp4(xd, hb, a4["codes"], a4["sf"], a4["gs"], ws)
    W = wq.nvfp4
    y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    sc = torch.empty(1, dtype=torch.float32, device="cuda")
    dit.qgemm_nvfp4_amax(a4["codes"], a4["sf"], a4["gs"], W["codes"], W["sf"], W["gs"], y, ws, hb, sc,
                         act=dit.ACT_GELU_ERF)
    q = dit.alloc_nvfp4(m, n)
    dit.hadamard_quant_nvfp4(y, hb, q["codes"], q["sf"], q["gs"], ws)
    _status_clean(ws)
    assert sc.view(torch.int32).item() == q["gs"].view(torch.int32).item()


# ------------------------------------------------------------------------------ NVFP4-only weights


@pytest.mark.parametrize("rows,k", [(5760 // 20, 1920), (129, 7680), (1, 64), (300, 3072)])
@pytest.mark.parametrize("container", [torch.int8, torch.bfloat16])
def test_nvfp4_to_int8_parity(rows, k, container):
    """INT8 weights derived on the GPU from NVFP4 weights equal the oracle's: scales bit-exact,
    codes bit-exact except elements on a rounding boundary."""
    g = synth.rng(rows * 3 + k)
    w = (g.standard_normal((rows, k)) * 0.02).astype(np.float32)
    w[:, ::97] *= 30.0
    r4 = D.quant_nvfp4(D.block_fwht_f32(w, 64))
    codes = torch.from_numpy(D.pack_e2m1(r4["codes"])).cuda()
    sf = torch.from_numpy(F.sf_to_tiled(r4["sf"], rows, k)).cuda()
    gs = torch.tensor([float(r4["s_g"])], dtype=torch.float32, device="cuda")
    q = torch.empty(rows, k, dtype=container, device="cuda")
    sc = torch.empty(rows, dtype=torch.float32, device="cuda")
    dit.nvfp4_to_int8(codes, sf, gs, q, sc)
    torch.cuda.synchronize()
    ref = D.nvfp4_weight_to_int8(r4["codes"], r4["sf"], r4["s_g"])
    assert np.array_equal(host(sc).view(np.uint32), ref["scale"].view(np.uint32))
    qh = _codes(q)
    bad = (qh != ref["q"]) & ~(D.int8_rounding_margin(ref["v"]) <= 1e-5)
    assert not bad.any(), int(bad.sum())


def test_nvfp4_to_int8_worked_example():
    """The hand-worked fixture (padded from K = 32 to 64 with zero codes and scales)."""
    from conftest import load_golden
    gd, _ = load_golden("nvfp4_weight_to_int8.txt")
    codes = np.zeros((2, 64), np.uint8)
    codes[0, :32] = [int(v) for v in gd["codes_row0"]]
    codes[1, :32] = [int(v) for v in gd["codes_row1"]]
    sf = np.zeros((2, 4), np.uint8)
    sf[0, :2] = [int(v, 16) for v in gd["sf_row0"]]
    q = torch.empty(2, 64, dtype=torch.int8, device="cuda")
    sc = torch.empty(2, dtype=torch.float32, device="cuda")
    dit.nvfp4_to_int8(torch.from_numpy(D.pack_e2m1(codes)).cuda(), torch.from_numpy(F.sf_to_tiled(sf, 2, 64)).cuda(),
                      torch.tensor([float(gd["s_g"][0])], device="cuda"), q, sc)
    qh = host(q)
    assert qh[0, :32].tolist() == [int(v) for v in gd["q_row0"]] and not qh[0, 32:].any()
    assert not qh[1].any()
    num, den = (np.float32(v) for v in gd["scale_row0"])
    assert host(sc)[0] == num / den and host(sc)[1] == 0


@pytest.mark.parametrize("container", ["bf16", "int8"])
def test_routed_linear_nvfp4_only_weights(container, ws):
    """A linear whose weights are resident in NVFP4 only: the INT8 route derives the INT8
    weights on the fly; output against the oracle on the GPU's own quantised operands."""
    m, k, n, hb = 300, 1920, 576, 64
    x, xd = make_x(m, k, "bf16", seed=81)
    w = synth.weights(n, k, seed=82)
    wq = dit.QuantizedWeight(dev_f32(w), hb, ws, int8_container=container, nvfp4_only=True)
    full = dit.QuantizedWeight(dev_f32(w), hb, ws, int8_container=container)
    # NVFP4 (0.5625 B/weight) alone vs NVFP4 plus the INT8 copy (1 or 2 B/weight)
    assert wq.int8 is None and wq.resident_bytes() * (4 if container == "bf16" else 2.5) < full.resident_bytes()
    lin = dit.RoutedLinear(wq, m, ws)
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    lin(xd, dit.ROUTE_INT8, y)
    _status_clean(ws)
    w8 = D.nvfp4_weight_to_int8(D.unpack_e2m1(host(wq.nvfp4["codes"])), F.sf_from_tiled(host(wq.nvfp4["sf"]), n, k),
                                host(wq.nvfp4["gs"])[0])
    assert np.array_equal(_codes(lin.w8_scratch["q"]), w8["q"])
    ref = D.gemm_int8(_codes(lin.a8["q"]), host(lin.a8["scale"]), w8["q"], w8["scale"])
    assert rel_fro(host(y), ref) <= GEMM_TOL
    # NVFP4 route of the same layer is unaffected
    lin(xd, dit.ROUTE_NVFP4, y)
    torch.cuda.synchronize()
    ref4 = D.gemm_nvfp4(D.unpack_e2m1(host(lin.a4["codes"])), F.sf_from_tiled(host(lin.a4["sf"]), m, k),
                        host(lin.a4["gs"])[0], D.unpack_e2m1(host(wq.nvfp4["codes"])),
                        F.sf_from_tiled(host(wq.nvfp4["sf"]), n, k), host(wq.nvfp4["gs"])[0])
    assert rel_fro(host(y), ref4) <= GEMM_TOL


# ------------------------------------------------------------------------------ routed linear


def _codes(t):
    """INT8 codes on the host from either container."""
    return host(t) if t.dtype == torch.int8 else F.bf16_bits_to_f32(host(t)).astype(np.int8)


@pytest.mark.parametrize("route,container", [(dit.ROUTE_NVFP4, "bf16"), (dit.ROUTE_INT8, "bf16"),
                                             (dit.ROUTE_INT8, "int8")])
def test_single_linear_end_to_end(route, container, ws):
    """The 256x128 single linear (Hadamard block 16) along both routes, stage by stage."""
    c = synth.single_linear()
    wq = dit.QuantizedWeight(dev_f32(c["w"]), 16, ws, int8_container=container)
    lin = dit.RoutedLinear(wq, 256, ws)
    y = torch.empty(256, 512, dtype=torch.float32, device="cuda")
    lin(dev_f32(c["x"]), route, y)
    _status_clean(ws)
    wp = D.prepare_weight(c["w"], 16)
    if route == dit.ROUTE_INT8:
        wqh, aqh = _codes(wq.int8["q"]), _codes(lin.a8["q"])
        check_int8(wqh, host(wq.int8["scale"]), c["w"], "f32", 16)
        check_int8(aqh, host(lin.a8["scale"]), c["x"], "f32", 16)
        ref = D.gemm_int8(aqh, host(lin.a8["scale"]), wqh, host(wq.int8["scale"]))
    else:
        check_nvfp4(host(wq.nvfp4["codes"]), host(wq.nvfp4["sf"]), host(wq.nvfp4["gs"])[0], c["w"], "f32", 16, 512, 128)
        check_nvfp4(host(lin.a4["codes"]), host(lin.a4["sf"]), host(lin.a4["gs"])[0], c["x"], "f32", 16, 256, 128)
        ref = D.gemm_nvfp4(D.unpack_e2m1(host(lin.a4["codes"])), F.sf_from_tiled(host(lin.a4["sf"]), 256, 128),
                           host(lin.a4["gs"])[0], D.unpack_e2m1(host(wq.nvfp4["codes"])),
                           F.sf_from_tiled(host(wq.nvfp4["sf"]), 512, 128), host(wq.nvfp4["gs"])[0])
    assert rel_fro(host(y), ref) <= GEMM_TOL
    # and the whole path against the all-oracle routed linear
    assert rel_fro(host(y), D.routed_linear(c["x"], wp, 16, route)) <= GEMM_TOL


# ------------------------------------------------------------------------------ full size


def test_full_size_cogvideox_2b_sampled(ws):
    """Full CogVideoX-2B QKV shape (17776 x 1920 -> 5760): quantisers checked on sampled rows
    (with the whole-tensor scale from the oracle), GEMM outputs on sampled rows."""
    m, k, n = synth.TOKENS_2B, 1920, 5760
    x, xd = make_x(m, k, "bf16", seed=2024)
    w = synth.weights(n, k, seed=2025)
    wq = dit.QuantizedWeight(dev_f32(w), 64, ws)
    lin = dit.RoutedLinear(wq, m, ws)
    y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    rows = np.unique(np.concatenate([synth.rng(5).choice(m, 48, replace=False), np.arange(m - 16, m)]))
    for route in (dit.ROUTE_NVFP4, dit.ROUTE_INT8):
        lin(xd, route, y)
        torch.cuda.synchronize()
        yh = F.bf16_bits_to_f32(host(y))[rows]
        if route == dit.ROUTE_NVFP4:
            yfull = D.block_fwht_f32(F.bf16_bits_to_f32(x), 64)
            sg = D.nvfp4_tensor_scale(yfull)
            assert np.float32(host(lin.a4["gs"])[0]) == sg
            codes = D.unpack_e2m1(host(lin.a4["codes"]))[rows]
            sf = F.sf_from_tiled(host(lin.a4["sf"]), m, k)[rows]
            r = D.quant_nvfp4(yfull[rows], s_g=sg)
            ex = (F.e2m1_rounding_margin(r["v"]) <= 1e-5) | (F.e4m3_rounding_margin(r["sbf"]) <= 1e-5).repeat(16, axis=1)
            assert not ((codes != r["codes"]) & ~ex).any()
            ref = D.gemm_nvfp4(codes, sf, sg, D.unpack_e2m1(host(wq.nvfp4["codes"])),
                               F.sf_from_tiled(host(wq.nvfp4["sf"]), n, k), host(wq.nvfp4["gs"])[0])
        else:
            q = _codes(lin.a8["q"])[rows]
            s = host(lin.a8["scale"])[rows]
            xr = x[rows]
            check_int8(q, s, xr, "bf16", 64)
            ref = D.gemm_int8(q, s, _codes(wq.int8["q"]), host(wq.int8["scale"]))
        refb = F.bf16_bits_to_f32(F.f32_to_bf16_bits(ref.astype(np.float32)))
        assert rel_fro(yh, refb) <= GEMM_TOL
    _status_clean(ws)


def test_tdc_chained_blocks_full_size(ws):
    """Two chained CogVideoX-2B-sized blocks (17776 x 1920 bf16) through 8 denoising steps with
    DeltaCachedBlock: decisions, PDR routes and every block output identical to the oracle."""
    rows, k, steps, tau = synth.TOKENS_2B, 1920, 8, 0.05
    alpha, beta, thr = [1.0] * 4, [0.0] * 4, [0.05] * 4
    thr64 = np.float32(thr).astype(np.float64)
    xs = [synth.activations(rows, k, seed=500 + t, outlier_frac=0.0) for t in range(steps)]
    deltas = [synth.tdc_deltas(steps, rows, k, seed=600 + b, jump_every=4.0)[0] for b in range(2)]
    ref0 = T.run_block_loop(xs, deltas[0], tau, alpha, beta, thr64)
    ref1 = T.run_block_loop(ref0["outs"], deltas[1], tau, alpha, beta, thr64)
    refs = [ref0, ref1]
    gam = torch.zeros(2, dtype=torch.float32, device="cuda")
    sim = torch.zeros(2, dtype=torch.float32, device="cuda")
    blocks = [dit.DeltaCachedBlock(rows * k, torch.bfloat16, tau, alpha, beta, thr, ws, gam[b:b + 1], sim[b:b + 1])
              for b in range(2)]
    for t in range(steps):
        x = dev_bf16(xs[t]).reshape(-1)
        for b, blk in enumerate(blocks):
            mode = blk.decide()
            x_next = torch.empty_like(x)
            want = refs[b]["decisions"][t]
            if refs[b]["margins"][t] > 1e-5:
                assert (mode == dit.TDC_SKIP) == (want == "skip"), (t, b)
            if mode == dit.TDC_SKIP:
                blk.skip(x, x_next)
            else:
                if refs[b]["routes"][t] is not None:
                    g_ref = refs[b]["gammas"][t]
                    if g_ref is None or abs(g_ref - 0.05) > 1e-5 * 0.05:
                        assert blk.routes() == refs[b]["routes"][t], (t, b)
                dlt = dev_bf16(deltas[b][t]).reshape(-1)
                x_next.copy_((x.float() + dlt.float()).to(torch.bfloat16))
                blk.commit(x, x_next)
            assert np.array_equal(host(x_next), refs[b]["outs"][t].reshape(-1)), (t, b)
            x = x_next
        h = torch.stack([gam, sim]).cpu()
        for b, blk in enumerate(blocks):
            blk.absorb(float(h[0, b]), float(h[1, b]))
    _status_clean(ws)


@pytest.mark.parametrize("route", ["nvfp4", "nvfp4_gelu", "nvfp4_fp32", "int8"])
def test_gemm_bounded_wait_reports_timeout_and_recovers(route, monkeypatch):
    """A GEMM whose producer issues no loads (test hook): the consumers' bounded waits run out
    after ~1 s, the kernel records DIT_ERR_TIMEOUT in the workspace status word, frees its
    tensor memory and exits; the next normal call on the same context is correct."""
    import time
    ws2 = dit.workspace()
    # the NVFP4 routes reach the three tile configurations: bf16 output (128 x 256, eight epilogue
    # warps), GELU (sixteen), fp32 output with K < 3072 (128 x 128, two CTAs per SM)
    m, n, k = 256, 256, 128
    g = synth.rng(55)
    if route.startswith("nvfp4"):
        qa, qb, A, B = _nvfp4_operands(m, n, k, seed=56)
        ref = D.gemm_nvfp4(qa["codes"], qa["sf"], qa["s_g"], qb["codes"], qb["sf"], qb["s_g"])
        act = dit.ACT_GELU_ERF if route == "nvfp4_gelu" else dit.ACT_NONE
        if act:
            ref = D.gelu_erf(ref)
        if route == "nvfp4":   # bf16 output: compare with the oracle as bf16 would store it
            ref = F.bf16_bits_to_f32(F.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
        ybuf = torch.zeros(m, n, dtype=torch.bfloat16 if route == "nvfp4" else torch.float32, device="cuda")

        def call(y):
            dit.qgemm_nvfp4(A["codes"], A["sf"], A["gs"], B["codes"], B["sf"], B["gs"], ybuf, ws2, act=act)
            y.copy_(ybuf.float())
    else:
        a = g.integers(-127, 128, (m, k)).astype(np.int8)
        b = g.integers(-127, 128, (n, k)).astype(np.int8)
        sa, sb = np.ones(m, np.float32), np.ones(n, np.float32)
        ref = D.gemm_int8(a, sa, b, sb)
        ta, tb = _int8_dev(a, torch.bfloat16), _int8_dev(b, torch.bfloat16)
        call = lambda y: dit.qgemm_int8(ta, dev_f32(sa), tb, dev_f32(sb), y, ws2)
    y = torch.zeros(m, n, dtype=torch.float32, device="cuda")
    monkeypatch.setenv("DIT6_TEST_STALL_PRODUCER", "1")
    t0 = time.time()
    call(y)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert dit.device_status(ws2) & (1 << 5), "DIT_ERR_TIMEOUT not raised"
    assert elapsed < 30.0
    monkeypatch.delenv("DIT6_TEST_STALL_PRODUCER")
    dit.clear_device_status(ws2)
    call(y)
    torch.cuda.synchronize()
    assert dit.device_status(ws2) == 0
    assert rel_fro(host(y), ref) <= GEMM_TOL


def test_int8_requant_bounded_wait_reports_timeout_and_recovers(monkeypatch):
    """The requantising INT8 GEMM (sixteen epilogue warps) with a producer that issues no loads:
    the waits run out, DIT_ERR_TIMEOUT is raised, and the next normal call on the same workspace
    gives the quantiser's codes bit for bit."""
    import time
    ws2 = dit.workspace()
    m, n, k = 256, 512, 1024
    g = synth.rng(57)
    ta = _int8_dev(g.integers(-127, 128, (m, k)).astype(np.int8), torch.bfloat16)
    tb = _int8_dev(g.integers(-127, 128, (n, k)).astype(np.int8), torch.bfloat16)
    sa, sb = dev_f32(np.full(m, 1e-3, np.float32)), dev_f32(np.full(n, 1e-3, np.float32))
    y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    dit.qgemm_int8(ta, sa, tb, sb, y, ws2)
    q_ref = torch.empty_like(y)
    s_ref = torch.empty(m, dtype=torch.float32, device="cuda")
    dit.hadamard_quant_int8(y, 64, q_ref, s_ref)
    q = torch.zeros_like(y)
    amax = torch.zeros(m, dtype=torch.float32, device="cuda")
    monkeypatch.setenv("DIT6_TEST_STALL_PRODUCER", "1")
    t0 = time.time()
    dit.qgemm_int8_requant(ta, sa, tb, sb, s_ref, q, amax, ws2)
    torch.cuda.synchronize()
    assert dit.device_status(ws2) & (1 << 5), "DIT_ERR_TIMEOUT not raised"
    assert time.time() - t0 < 30.0
    monkeypatch.delenv("DIT6_TEST_STALL_PRODUCER")
    dit.clear_device_status(ws2)
    amax.zero_()
    dit.qgemm_int8_requant(ta, sa, tb, sb, s_ref, q, amax, ws2)
    torch.cuda.synchronize()
    assert dit.device_status(ws2) == 0
    assert torch.equal(q.view(torch.int16), q_ref.view(torch.int16))


def test_delta_cache_checkpoint_resume(ws):
    """A block's delta cache saved mid-run (decision state + cached delta) and loaded into a
    fresh block continues exactly like the original: same decisions, same outputs bit for bit."""
    n, steps, cut = 4096 + 32, 10, 4
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    x_in = torch.randn(n, generator=g, device="cuda").to(torch.bfloat16)
    base = torch.randn(n, generator=g, device="cuda") * 0.05
    deltas = [(base * (1 + 0.002 * t)).to(torch.bfloat16) for t in range(steps)]
    gam = torch.zeros(2, dtype=torch.float32, device="cuda")
    sim = torch.zeros(2, dtype=torch.float32, device="cuda")

    def make(slot):
        return dit.DeltaCachedBlock(n, torch.bfloat16, 0.007, [1.0], [0.0], [0.05], ws, gam[slot:slot + 1],
                                    sim[slot:slot + 1])

    def run(blk, slot, t0, t1):
        trace = []
        for t in range(t0, t1):
            out = torch.empty_like(x_in)
            mode = blk.decide()
            if mode == dit.TDC_SKIP:
                blk.skip(x_in, out)
            else:
                out.copy_((x_in.float() + deltas[t].float()).to(torch.bfloat16))
                blk.commit(x_in, out)
                torch.cuda.synchronize()
                blk.absorb(float(gam[slot]), float(sim[slot]))
            trace.append((mode, blk.routes(), out.clone()))
        return trace

    a = make(0)
    run(a, 0, 0, cut)
    sd = a.state_dict()
    rest_a = run(a, 0, cut, steps)
    b = make(1)
    b.load_state_dict(sd)
    rest_b = run(b, 1, cut, steps)
    modes = [m for m, _, _ in rest_a]
    assert modes == [m for m, _, _ in rest_b] and dit.TDC_SKIP in modes and dit.TDC_COMMIT in modes
    assert [r for _, r, _ in rest_a] == [r for _, r, _ in rest_b]
    for (_, _, oa), (_, _, ob) in zip(rest_a, rest_b):
        assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    _status_clean(ws)


# ------------------------------------------------------------------------------ PDR: outlier ratio, BF16 route


@pytest.mark.parametrize("n,dtype", [(17776 * 1920, "bf16"), (300 * 1920 + 7, "bf16"), (4096 + 3, "f32"), (5, "f32")])
def test_outlier_ratio_parity(n, dtype, ws):
    """Count of |x| > 6 RMS against the oracle: exact, except elements within 1e-6 relative of
    the threshold (the GPU's RMS comes from a different summation order)."""
    g = synth.rng(n % 9973)
    x = g.standard_normal(n).astype(np.float32)
    x[:: 97] *= 40.0                                       # outlier channels
    xd = dev_f32(x) if dtype == "f32" else dev_bf16(F.f32_to_bf16_bits(x))
    xv = x if dtype == "f32" else F.bf16_bits_to_f32(F.f32_to_bf16_bits(x))
    ratio = torch.empty(1, dtype=torch.float32, device="cuda")
    count = torch.empty(1, dtype=torch.int64, device="cuda")
    dit.outlier_ratio(xd, ws, ratio, count)
    _status_clean(ws)
    x64 = xv.astype(np.float64)
    thr = 6.0 * math.sqrt(float(np.sum(x64 * x64)) / n)
    want = int(np.count_nonzero(np.abs(x64) > thr))
    near = int(np.count_nonzero(np.abs(np.abs(x64) - thr) <= 1e-6 * thr))
    assert abs(int(count.item()) - want) <= near
    assert D.outlier_ratio(xv) == want / n
    assert ratio.item() == pytest.approx(int(count.item()) / n, rel=1e-6)


@pytest.mark.parametrize("m,n,k", [(256, 512, 128), (300, 384, 1920), (129, 256, 7680), (1, 8, 16), (700, 576, 2112)])
@pytest.mark.parametrize("act", [0, 1])
def test_gemm_bf16_parity(m, n, k, act, ws):
    """The BF16 route against the float64 oracle: fp32 output within 1e-5 relative Frobenius
    (fp32 accumulation of exact bf16 products), bf16 output against the oracle rounded to bf16."""
    g = synth.rng(m + n + k + act)
    xb = F.f32_to_bf16_bits(g.standard_normal((m, k)).astype(np.float32))
    wb = F.f32_to_bf16_bits((g.standard_normal((n, k)) * 0.05).astype(np.float32))
    bias = (g.standard_normal(n) * 0.1).astype(np.float32)
    ref = D.gemm_bf16(F.bf16_bits_to_f32(xb), F.bf16_bits_to_f32(wb), bias)
    if act:
        ref = D.gelu_erf(ref)
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    dit.gemm_bf16(dev_bf16(xb), dev_bf16(wb), y, ws, bias=dev_f32(bias), act=act)
    _status_clean(ws)
    assert rel_fro(host(y), ref) <= 1e-5
    yb = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    dit.gemm_bf16(dev_bf16(xb), dev_bf16(wb), yb, ws, bias=dev_f32(bias), act=act)
    refb = F.bf16_bits_to_f32(F.f32_to_bf16_bits(ref.astype(np.float32)))
    assert rel_fro(F.bf16_bits_to_f32(host(yb)), refb) <= GEMM_TOL


def test_routed_linear_bf16_route_and_pdr_override(ws):
    """A block input with a high outlier ratio sends every layer to BF16 (PDR); the BF16 route
    of a linear computes X W^T on the untransformed weight."""
    m, k, n = 300, 1920, 576
    x, xd = make_x(m, k, "bf16", seed=91)
    w = synth.weights(n, k, seed=92)
    wq = dit.QuantizedWeight(dev_f32(w), 64, ws, keep_bf16=True)
    lin = dit.RoutedLinear(wq, m, ws)
    ratio = torch.empty(1, dtype=torch.float32, device="cuda")
    dit.outlier_ratio(xd, ws, ratio)
    r = ratio.item()
    assert r > 0
    st = dit.TdcState()
    st.update(dit.TDC_COMMIT, 0.01, None)
    assert st.routes([1.0] * 4, [0.0] * 4, [0.05] * 4, r, r / 2) == [dit.ROUTE_BF16] * 4
    assert st.routes([1.0] * 4, [0.0] * 4, [0.05] * 4, r, 2 * r) == [dit.ROUTE_NVFP4] * 4
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    lin(xd, dit.ROUTE_BF16, y)
    _status_clean(ws)
    ref = D.gemm_bf16(F.bf16_bits_to_f32(x), F.bf16_bits_to_f32(F.f32_to_bf16_bits(w)))
    assert rel_fro(host(y), ref) <= 1e-5
