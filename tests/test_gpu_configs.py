"""Full-size parity of the CogVideoX-5B block linears and the 1080p long sequence (GPU).

Every kernel runs at the real size; the oracle checks seeded row samples (plus the ragged
tail rows) stage by stage: the quantised codes and scales of activations and weights against
the oracle's quantisers (the NVFP4 tensor scale from the oracle's whole-tensor amax), and the
GEMM rows against the float64 oracle GEMM of the GPU's own quantised operands.
"""
import numpy as np
import pytest

import synth
from gpu_helpers import check_int8, dev_bf16, dev_f32, host, rel_fro
from oracle import dmpq as D
from oracle import formats as F

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import int8_mixed_precision_gb300 as dit  # noqa: E402

TOL = 1e-3
HB = 64


@pytest.fixture(scope="module")
def ws():
    return dit.workspace()


def _codes(t):
    return host(t) if t.dtype == torch.int8 else F.bf16_bits_to_f32(host(t)).astype(np.int8)


def _sample_rows(m, seed, n=40):
    return np.unique(np.concatenate([synth.rng(seed).choice(m, n, replace=False), np.arange(m - 8, m)]))


def _global_scale(x_bits, chunk=8192):
    """The oracle's NVFP4 tensor scale of the transformed tensor, computed in row chunks."""
    amax = np.float32(0)
    for r0 in range(0, x_bits.shape[0], chunk):
        y = D.block_fwht_f32(F.bf16_bits_to_f32(x_bits[r0:r0 + chunk]), HB)
        amax = max(amax, np.float32(np.max(np.abs(y))))
    return np.float32(amax / D.FP4_X_E4M3)


def _check_nvfp4_rows(codes_dev, sf_dev, sg, x_rows_f32, rows_idx, m, k):
    r = D.quant_nvfp4(D.block_fwht_f32(x_rows_f32, HB), s_g=sg)
    codes = D.unpack_e2m1(host(codes_dev[torch.from_numpy(rows_idx).cuda()]))
    sf_all = host(sf_dev)
    rr, cc = np.meshgrid(rows_idx, np.arange(k // 16), indexing="ij")
    sf = sf_all[F.sf_tiled_offset(rr, cc, m, k)]
    blk_ex = F.e4m3_rounding_margin(r["sbf"]) <= 1e-5
    assert not ((sf != r["sf"]) & ~blk_ex).any()
    el_ex = (F.e2m1_rounding_margin(r["v"]) <= 1e-5) | blk_ex.repeat(16, axis=1)
    assert not ((codes != r["codes"]) & ~el_ex).any()
    return codes, sf


def _routed_linear_full(m, k, n, dist, mult, frac, seed, routes, ws, x_bits=None, act=0, keep=None):
    """Quantise a full [m x k] activation and an [n x k] weight on the GPU along the given
    routes, run the GEMM (with the epilogue activation act), and check sampled rows of every
    stage against the oracle.  keep: route whose full bf16 output is returned (host bits)."""
    if x_bits is None:
        x_bits = synth.activations(m, k, dist=dist, outlier_frac=frac, outlier_mult=mult, seed=seed)
    w = synth.weights(n, k, seed=seed + 1)
    xd = dev_bf16(x_bits)
    wq = dit.QuantizedWeight(dev_f32(w), HB, ws)
    lin = dit.RoutedLinear(wq, m, ws)
    y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    rows = _sample_rows(m, seed)
    wrows = _sample_rows(n, seed + 2, 24)
    xr = F.bf16_bits_to_f32(x_bits[rows])
    kept = None
    for route in routes:
        lin(xd, route, y, act=act)
        torch.cuda.synchronize()
        yh = F.bf16_bits_to_f32(host(y[torch.from_numpy(rows).cuda()]))
        if route == dit.ROUTE_INT8:
            qa = _codes(lin.a8["q"])[rows]
            sa = host(lin.a8["scale"])[rows]
            check_int8(qa, sa, xr, "f32", HB)
            qw = _codes(wq.int8["q"])
            check_int8(qw[wrows], host(wq.int8["scale"])[wrows], w[wrows], "f32", HB)
            ref = D.gemm_int8(qa, sa, qw, host(wq.int8["scale"]))
        else:
            sg = _global_scale(x_bits)
            assert np.float32(host(lin.a4["gs"])[0]) == sg
            codes, sf = _check_nvfp4_rows(lin.a4["codes"], lin.a4["sf"], sg, xr, rows, m, k)
            wsg = D.nvfp4_tensor_scale(D.block_fwht_f32(w, HB))
            assert np.float32(host(wq.nvfp4["gs"])[0]) == wsg
            _check_nvfp4_rows(wq.nvfp4["codes"], wq.nvfp4["sf"], wsg, w[wrows], wrows, n, k)
            ref = D.gemm_nvfp4(codes, sf, sg, D.unpack_e2m1(host(wq.nvfp4["codes"])),
                               F.sf_from_tiled(host(wq.nvfp4["sf"]), n, k), wsg)
        if act == dit.ACT_GELU_ERF:
            ref = D.gelu_erf(ref)
        refb = F.bf16_bits_to_f32(F.f32_to_bf16_bits(ref.astype(np.float32)))
        assert rel_fro(yh, refb) <= TOL, (route, rel_fro(yh, refb))
        if route == keep:
            kept = host(y)
    torch.cuda.synchronize()
    assert dit.device_status(ws) == 0
    return kept


@pytest.mark.parametrize("layer,k,n", [("qkv", 3072, 9216), ("out", 3072, 3072), ("ffn_up", 3072, 12288),
                                       ("ffn_down", 12288, 3072)])
def test_cogvideox_5b_block_linears(layer, k, n, ws):
    """CogVideoX-5B-shaped linears: 17776 tokens, Laplace(0,1) with 0.5% channels x100."""
    _routed_linear_full(synth.TOKENS_2B, k, n, "laplace", 100.0, 0.005, 3000 + k + n,
                        (dit.ROUTE_NVFP4, dit.ROUTE_INT8), ws)


@pytest.mark.parametrize("up_route,down_routes", [(1, (0, 1)), (0, (1,))])
def test_cogvideox_2b_ffn_chain_with_gelu(up_route, down_routes, ws):
    """The CogVideoX-2B FFN as one chain: 17776 x 1920 -> 7680 with GELU (erf form) fused in
    the up projection's epilogue, whose bf16 output is the down projection's input
    (7680 -> 1920).  Each stage is checked on sampled rows against the oracle, the down
    projection on the GPU's own GELU output (its NVFP4 tensor scale from that whole tensor)."""
    m = synth.TOKENS_2B
    h = _routed_linear_full(m, 1920, 7680, "normal", 50.0, 0.01, 5000, (up_route,), ws, act=dit.ACT_GELU_ERF,
                            keep=up_route)
    assert h is not None and h.shape == (m, 7680)
    _routed_linear_full(m, 7680, 1920, None, None, None, 5100, down_routes, ws, x_bits=h)


def test_long_sequence_1080p_ffn_up(ws):
    """1080p-shaped sequence: 104746 tokens, FFN up 3072 -> 12288, both routes."""
    _routed_linear_full(synth.TOKENS_1080P, 3072, 12288, "laplace", 100.0, 0.005, 4000,
                        (dit.ROUTE_NVFP4, dit.ROUTE_INT8), ws)


def test_long_sequence_1080p_ffn_down_int8(ws):
    """1080p-shaped sequence: FFN down 12288 -> 3072 (104746 x 12288 activation), INT8 route."""
    _routed_linear_full(synth.TOKENS_1080P, 12288, 3072, "laplace", 100.0, 0.005, 4100, (dit.ROUTE_INT8,), ws)


def test_long_sequence_gamma_and_tdc(ws):
    """Gamma and the delta-cache commit over a 104746 x 3072 bf16 pair (643 MB each)."""
    m, k = synth.TOKENS_1080P, 3072
    xi = synth.activations(m, k, dist="laplace", outlier_frac=0.005, outlier_mult=100.0, seed=4200)
    xo = synth.gamma_pair(xi, 0.06, 4201)
    di, do = dev_bf16(xi), dev_bf16(xo)
    gam = torch.empty(1, dtype=torch.float32, device="cuda")
    r = torch.empty(1, dtype=torch.int32, device="cuda")
    dit.gamma_route(di, do, [1.0], [0.0], [0.05], gam, r, ws)
    ref = D.gamma_rel_l1(F.bf16_bits_to_f32(xi), F.bf16_bits_to_f32(xo))
    assert gam.item() == pytest.approx(ref, rel=1e-5)
    assert r.tolist() == [dit.ROUTE_INT8]
    dnew = torch.empty_like(di)
    sim = torch.empty(1, dtype=torch.float32, device="cuda")
    dit.tdc_step(dit.TDC_COMMIT, di, ws, x_out=do, d1=None, d_new=dnew, gamma=gam, sim=sim)
    rows = _sample_rows(m, 4202)
    want = F.f32_to_bf16_bits(F.bf16_bits_to_f32(xo[rows]) - F.bf16_bits_to_f32(xi[rows]))
    assert np.array_equal(host(dnew[torch.from_numpy(rows).cuda()]), want)
    assert gam.item() == pytest.approx(ref, rel=1e-5)
