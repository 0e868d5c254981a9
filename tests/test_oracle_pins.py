"""Pins of the CPU oracle against things other than itself (no GPU).

Each check ties an oracle function to a closed form, a library routine, brute force on
tiny inputs, or a hand-worked fixture under tests/golden/.  The "planted mistake" tests at
the end patch a plausible error into a copy of an oracle function (on the CPU) and show
that the matching pin fails.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import torch

import synth
from conftest import load_golden
from oracle import dmpq as D
from oracle import formats as F
from oracle import tdc as T

# ------------------------------------------------------------------------------- helpers


def brute_e2m1(v):
    """Nearest of the 16 E2M1 values by exhaustive search, ties to the even code, sign kept."""
    out = []
    for x in np.asarray(v, np.float32).ravel():
        a = abs(float(x))
        if a > 6.0:
            best = 7
        else:
            d = [abs(a - F.E2M1_VALUES[c]) for c in range(8)]
            m = min(d)
            cands = [c for c in range(8) if d[c] == m]
            best = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        out.append(best | (8 if math.copysign(1.0, float(x)) < 0 else 0))
    return np.array(out, np.uint8).reshape(np.shape(v))


def brute_e4m3(v):
    """Nearest non-negative finite E4M3 value by exhaustive search (ties even), sat. 448."""
    vals = [F.E4M3_VALUES[c] for c in range(127)]
    out = []
    for x in np.asarray(v, np.float32).ravel():
        a = float(x)
        if a >= 448.0:
            out.append(126)
            continue
        d = [abs(a - vals[c]) for c in range(127)]
        m = min(d)
        cands = [c for c in range(127) if d[c] == m]
        out.append(cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0])
    return np.array(out, np.uint8).reshape(np.shape(v))


def check_fwht(fwht, b, seed=0):
    x = synth.rng(seed).standard_normal((5, 4 * b)).astype(np.float32)
    ref = D.block_hadamard_f64(x, b)
    got = fwht(x, b).astype(np.float64)
    return np.max(np.abs(got - ref)) <= 1e-5 * max(1.0, np.max(np.abs(ref)))


def check_nvfp4_codes(quant, seed=0):
    """Codes are the brute-force nearest E2M1 of v; scales the brute-force nearest E4M3 of
    sbf; the block holding the tensor amax gets the top scale 448 (code 0x7e); every block
    with a normal-range scale has its largest |v| within E4M3 rounding (1/16) of 6."""
    g = synth.rng(seed)
    y = (g.standard_normal((6, 64)) * np.exp(g.standard_normal((6, 1)))).astype(np.float32)
    y[0, :16] = 0.0
    r = quant(y)
    if not np.array_equal(r["codes"], np.where(r["zero_blk"].repeat(16, axis=1), 0, brute_e2m1(r["v"]))):
        return False
    if not np.array_equal(r["sf"], brute_e4m3(r["sbf"])):
        return False
    yb = np.abs(y.reshape(6, 4, 16)).max(axis=2)
    top = np.unravel_index(np.argmax(yb), yb.shape)
    if int(r["sf"][top]) != 0x7E:
        return False
    vmax = np.abs(r["v"].reshape(6, 4, 16)).max(axis=2).astype(np.float64)
    normal = F.E4M3_VALUES[r["sf"]] >= 2.0 ** -6
    return bool(np.all(np.abs(vmax[normal] - 6.0) <= 6.0 / 15.0))


# ------------------------------------------------------------------------------- Hadamard


@pytest.mark.parametrize("b", [1, 2, 4, 8, 16, 32, 64, 128])
def test_hadamard_matches_scipy_sylvester(b):
    assert np.array_equal(D.hadamard_sylvester(b), scipy.linalg.hadamard(b).astype(np.float64))


@pytest.mark.parametrize("b", [2, 16, 64, 128])
def test_hadamard_orthogonality(b):
    h = D.hadamard_sylvester(b)
    assert np.array_equal(h @ h.T, b * np.eye(b))


@pytest.mark.parametrize("b", [16, 32, 64, 128])
def test_fwht_stage_order_equals_matrix_product(b):
    assert check_fwht(D.block_fwht_f32, b)


@pytest.mark.parametrize("b", [16, 64])
def test_fwht_involution_and_norm(b):
    x = synth.rng(3).standard_normal((7, 3 * b)).astype(np.float32)
    y = D.block_hadamard_f64(x, b)
    assert np.allclose(D.block_hadamard_f64(y, b), x, atol=1e-12)
    n0 = np.linalg.norm(x.astype(np.float64).reshape(7, 3, b), axis=2)
    n1 = np.linalg.norm(y.reshape(7, 3, b), axis=2)
    assert np.allclose(n0, n1, rtol=1e-12)


def test_fwht_spreads_an_outlier():
    """A single outlier channel becomes a flat +-v/sqrt(b) row inside its block."""
    x = np.zeros((1, 64), np.float32)
    x[0, 5] = 64.0
    y = D.block_fwht_f32(x, 64)
    assert np.allclose(np.abs(y), 8.0)


# ------------------------------------------------------------------------------- formats


def test_e2m1_table_matches_golden():
    _, rows = load_golden("e2m1_codes.txt")
    for code, val in rows:
        got = F.E2M1_VALUES[int(code)]
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e2m1_rounding_golden():
    _, rows = load_golden("e2m1_rounding.txt")
    v = np.array([float(r[0]) for r in rows], np.float32)
    want = np.array([int(r[1]) for r in rows], np.uint8)
    assert np.array_equal(F.e2m1_encode(v), want)


def test_e2m1_roundtrip_all_codes():
    assert np.array_equal(F.e2m1_encode(F.E2M1_VALUES.astype(np.float32)), np.arange(16, dtype=np.uint8))


def test_e2m1_encode_vs_brute_force():
    g = synth.rng(11)
    v = np.concatenate([
        g.uniform(-8, 8, 4000).astype(np.float32),
        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 6.0, 6.5, -0.0], np.float32),
        np.nextafter(np.float32([0.25, 0.75, 2.5, 5.0]), np.float32(10)),
        np.nextafter(np.float32([0.25, 0.75, 2.5, 5.0]), np.float32(-10)),
    ])
    assert np.array_equal(F.e2m1_encode(v), brute_e2m1(v))


def test_e4m3_table_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.E4M3_VALUES
    assert np.array_equal(np.isnan(codes), np.isnan(ours))
    m = ~np.isnan(ours)
    assert np.array_equal(codes[m], ours[m])


def test_e4m3_golden():
    _, rows = load_golden("e4m3_values.txt")
    for code, val in rows:
        got = F.E4M3_VALUES[int(code, 16)]
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e4m3_encode_vs_torch_and_brute_force():
    g = synth.rng(5)
    grid = F.E4M3_VALUES[:127]
    mids = (0.5 * (grid[:-1] + grid[1:])).astype(np.float32)
    v = np.concatenate([
        np.exp(g.uniform(np.log(1e-4), np.log(448.0), 3000)).astype(np.float32),
        mids, np.nextafter(mids, np.float32(1e9)), np.nextafter(mids, np.float32(0)),
        np.float32([0.0, 448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11]),
    ])
    ours = F.e4m3_encode_nonneg(v)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)
    assert np.array_equal(ours, brute_e4m3(v))
    # saturation above the largest finite value (the library cast gives NaN there)
    assert np.all(F.e4m3_encode_nonneg(np.float32([449.0, 1e6])) == 126)


def test_bf16_matches_torch():
    g = synth.rng(9)
    x = np.concatenate([g.standard_normal(5000).astype(np.float32) * 100,
                        np.float32([1.00390625, 1.01171875, -3.0078125, 0.0, -0.0])])
    ours = F.f32_to_bf16_bits(x)
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.uint16).numpy() if hasattr(torch, "uint16") else \
        torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(ours, lib.astype(np.uint16))
    assert np.array_equal(F.bf16_bits_to_f32(ours),
                          torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy())


def test_sf_layout_golden_and_bijective():
    _, rows = load_golden("sf_layout.txt")
    for r, c, off in rows:
        assert int(F.sf_tiled_offset(int(r), int(c), 256, 128)) == int(off)
    for rows_, k in [(256, 128), (300, 1920), (17, 64)]:
        rp, cp = F.sf_padded_shape(rows_, k)
        rr, cc = np.meshgrid(np.arange(rp), np.arange(cp), indexing="ij")
        offs = F.sf_tiled_offset(rr, cc, rows_, k).ravel()
        assert np.array_equal(np.sort(offs), np.arange(rp * cp))
        sf = synth.rng(1).integers(0, 255, (rows_, k // 16)).astype(np.uint8)
        assert np.array_equal(F.sf_from_tiled(F.sf_to_tiled(sf, rows_, k), rows_, k), sf)


# ------------------------------------------------------------------------------- quantisers


def test_nvfp4_golden_block():
    kv, _ = load_golden("nvfp4_block.txt")
    y = np.array([float(t) for t in kv["y"]], np.float32)[None, :]
    r = D.quant_nvfp4(y, s_g=np.float32(kv["s_g"][0]))
    assert int(r["sf"][0, 0]) == int(kv["sf"][0], 16)
    assert r["codes"][0].tolist() == [int(t) for t in kv["codes"]]


def test_nvfp4_codes_and_scales_brute_force():
    assert check_nvfp4_codes(D.quant_nvfp4)


def test_nvfp4_dequant_error_bound():
    """Each element's error is at most half the local E2M1 gap times its block scale."""
    y = D.block_fwht_f32(synth.activations(64, 256, seed=4, dtype="f32"), 64)
    r = D.quant_nvfp4(y)
    deq = D.dequant_nvfp4(r["codes"], r["sf"], r["s_g"])
    bs = (F.E4M3_VALUES[r["sf"]] * float(r["s_g"])).repeat(16, axis=1)
    a = np.minimum(np.abs(r["v"].astype(np.float64)), 6.0)
    half_gap = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))
    sat = np.maximum(np.abs(r["v"].astype(np.float64)) - 6.0, 0.0)
    assert np.all(np.abs(deq - y) <= (half_gap + sat) * bs * (1 + 1e-6) + 1e-30)


def test_nvfp4_zero_tensor_and_zero_block():
    r = D.quant_nvfp4(np.zeros((3, 32), np.float32))
    assert r["s_g"] == 0 and not r["codes"].any() and not r["sf"].any()
    y = np.zeros((1, 32), np.float32)
    y[0, 16:] = 1.0
    r = D.quant_nvfp4(y)
    assert not r["codes"][0, :16].any() and r["sf"][0, 0] == 0 and r["sf"][0, 1] == 0x7E


def test_int8_golden_row():
    kv, _ = load_golden("int8_row.txt")
    y = np.array([float(t) for t in kv["y"]], np.float32)[None, :]
    r = D.quant_int8_rows(y)
    assert float(r["scale"][0]) == float(kv["scale"][0])
    assert r["q"][0].tolist() == [int(t) for t in kv["q"]]


def test_int8_brute_force_and_bounds():
    y = D.block_fwht_f32(synth.activations(32, 128, seed=8, dtype="f32"), 64)
    r = D.quant_int8_rows(y)
    q = r["q"].astype(np.int64)
    assert np.all(np.abs(q) <= 127)
    # brute force: nearest integer of v, ties to even, over all candidates -127..127
    cand = np.arange(-127, 128)
    v = r["v"].astype(np.float64)
    for i in range(0, v.size, 97):
        x = v.flat[i]
        d = np.abs(cand - x)
        best = cand[d == d.min()]
        want = best[0] if len(best) == 1 else best[best % 2 == 0][0]
        assert q.flat[i] == want
    # the row maximum maps to +-127 and the dequant error is at most s/2
    assert np.all(np.max(np.abs(q), axis=1) == 127)
    deq = D.dequant_int8(r["q"], r["scale"])
    assert np.all(np.abs(deq - y) <= r["scale"][:, None].astype(np.float64) * 0.5 * (1 + 1e-5))


def test_int8_zero_row():
    y = np.zeros((2, 16), np.float32)
    y[1, 3] = -2.0
    r = D.quant_int8_rows(y)
    assert r["scale"][0] == 0 and not r["q"][0].any() and r["q"][1, 3] == -127


def test_int8_given_scales_hand_values_and_saturation():
    """Quantisation with caller-supplied scales: hand-worked values at s = 0.5 (y/s = 0.48,
    0.52, 1.5, 2.5, -3.5 -> 0, 1, 2, 2, -4 under round-half-even), saturation at +-127 when y
    exceeds 127 s, and s = 0 giving zeros."""
    y = np.array([[0.24, 0.26, 0.75, 1.25, -1.75, 100.0, -100.0],
                  [1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0]], np.float32)
    q = D.quant_int8_rows_given(y, np.array([0.5, 0.0], np.float32))
    assert q[0].tolist() == [0, 1, 2, 2, -4, 127, -127]
    assert not q[1].any()


def test_int8_given_scales_reduce_to_the_dynamic_rule():
    """With s = amax_row / 127 the given-scale rule is the per-token rule, code for code; with
    half that scale every |v| beyond 63.5 saturates and the rest double (brute force)."""
    y = D.block_fwht_f32(synth.activations(16, 128, seed=9, dtype="f32"), 64)
    r = D.quant_int8_rows(y)
    assert np.array_equal(D.quant_int8_rows_given(y, r["scale"]), r["q"])
    half = (r["scale"] * np.float32(0.5)).astype(np.float32)
    q = D.quant_int8_rows_given(y, half).astype(np.int64)
    cand = np.arange(-127, 128)
    for i in range(0, y.size, 37):
        x = float(np.float32(y.flat[i] * (np.float32(1.0) / half[i // y.shape[1]])))
        d = np.abs(cand - x)
        best = cand[d == d.min()]
        assert q.flat[i] == (best[0] if len(best) == 1 else best[best % 2 == 0][0])


# ------------------------------------------------------------------------------- GEMMs


def test_int8_gemm_vs_triple_loop():
    g = synth.rng(21)
    a = g.integers(-127, 128, (5, 48)).astype(np.int8)
    b = g.integers(-127, 128, (7, 48)).astype(np.int8)
    acc = D.gemm_int8_acc(a, b)
    for m in range(5):
        for n in range(7):
            s = 0
            for k in range(48):
                s += int(a[m, k]) * int(b[n, k])
            assert acc[m, n] == s
    sa, sb = g.random(5).astype(np.float32), g.random(7).astype(np.float32)
    y = D.gemm_int8(a, sa, b, sb)
    assert y[2, 3] == pytest.approx(acc[2, 3] * float(sa[2]) * float(sb[3]), rel=1e-15)


def test_int8_gemm_extreme_accumulator_exact():
    """The largest accumulator at K = 12288 (12288 * 127^2) is exact."""
    a = np.full((1, 12288), -127, np.int8)
    b = np.full((2, 12288), -127, np.int8)
    b[1] = 127
    acc = D.gemm_int8_acc(a, b)
    assert acc[0, 0] == 12288 * 127 * 127 and acc[0, 1] == -12288 * 127 * 127


def test_nvfp4_gemm_vs_loops():
    g = synth.rng(22)
    ya = g.standard_normal((3, 32)).astype(np.float32)
    yb = g.standard_normal((4, 32)).astype(np.float32)
    qa, qb = D.quant_nvfp4(ya), D.quant_nvfp4(yb)
    y = D.gemm_nvfp4(qa["codes"], qa["sf"], qa["s_g"], qb["codes"], qb["sf"], qb["s_g"])
    for m in range(3):
        for n in range(4):
            s = 0.0
            for k in range(32):
                av = F.E2M1_VALUES[qa["codes"][m, k]] * F.E4M3_VALUES[qa["sf"][m, k // 16]]
                bv = F.E2M1_VALUES[qb["codes"][n, k]] * F.E4M3_VALUES[qb["sf"][n, k // 16]]
                s += av * bv
            assert y[m, n] == pytest.approx(s * float(qa["s_g"]) * float(qb["s_g"]), rel=1e-14)


def test_routed_linear_tracks_dense_product_and_hadamard_helps():
    """(XH)(WH)^T = XW^T up to quantisation error; the Hadamard lowers the per-token INT8
    error on outlier-channel activations (gist.science EN 2.A Outlier Smoothing)."""
    c = synth.single_linear()
    x, w = c["x"], c["w"]
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    err = {}
    for b in (1, 16):
        wp = D.prepare_weight(w, b) if b > 1 else {"nvfp4": D.quant_nvfp4(w), "int8": D.quant_int8_rows(w)}
        for route in (D.ROUTE_NVFP4, D.ROUTE_INT8):
            y = D.routed_linear(x, wp, b, route) if b > 1 else (
                D.gemm_nvfp4(**_q(D.quant_nvfp4(x), wp["nvfp4"])) if route == D.ROUTE_NVFP4 else
                D.gemm_int8(D.quant_int8_rows(x)["q"], D.quant_int8_rows(x)["scale"], wp["int8"]["q"], wp["int8"]["scale"]))
            err[(b, route)] = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert err[(16, D.ROUTE_INT8)] < 0.02
    assert err[(16, D.ROUTE_NVFP4)] < 0.15
    assert err[(16, D.ROUTE_INT8)] < err[(1, D.ROUTE_INT8)]
    assert err[(16, D.ROUTE_INT8)] < err[(16, D.ROUTE_NVFP4)]


def _q(qa, qw):
    return dict(a_codes=qa["codes"], a_sf=qa["sf"], a_sg=qa["s_g"], b_codes=qw["codes"], b_sf=qw["sf"], b_sg=qw["s_g"])


# ------------------------------------------------------------------------------- Gamma, routing


@pytest.mark.parametrize("gam", [0.0, 0.013, 0.05, 0.2])
def test_gamma_closed_form_scaling(gam):
    x = synth.rng(2).standard_normal((9, 33))
    assert D.gamma_rel_l1(x, (1 + gam) * x) == pytest.approx(gam, rel=1e-12, abs=1e-15)


def test_gamma_closed_form_random_signs():
    x = synth.rng(2).standard_normal((64, 64))
    s = np.where(synth.rng(3).random((64, 64)) < 0.5, -1.0, 1.0)
    assert D.gamma_rel_l1(x, x + 0.07 * s * x) == pytest.approx(0.07, rel=1e-12)


def test_gamma_degenerate():
    z = np.zeros((2, 2))
    assert D.gamma_rel_l1(z, z) == 0.0
    assert D.gamma_rel_l1(z, z + 1) == math.inf


def test_single_linear_gamma_routes_int8():
    """Gamma of the 256x128 single linear is ~ 0.1 sqrt(2/pi) / mean|X| ~ 0.052 > 0.05."""
    c = synth.single_linear()
    g = D.gamma_rel_l1(c["x"], c["x_out"])
    mean_abs = math.sqrt(2 / math.pi) * (124 + 4 * 30) / 128
    assert g == pytest.approx(0.1 * math.sqrt(2 / math.pi) / mean_abs, rel=0.03)
    assert D.route_layers(g, 1.0, 0.0, 0.05) == [D.ROUTE_INT8]


def test_route_rule():
    assert D.route_layers(0.05, 1.0, 0.0, 0.05) == [D.ROUTE_NVFP4]      # strict >
    assert D.route_layers(0.0500001, 1.0, 0.0, 0.05) == [D.ROUTE_INT8]
    assert D.route_layers(0.01, [1.0, 10.0], [0.0, 0.0], [0.05, 0.05]) == [D.ROUTE_NVFP4, D.ROUTE_INT8]
    assert D.route_layers(0.01, 1.0, 0.045, 0.05) == [D.ROUTE_INT8]      # beta shifts the error
    assert D.route_layers(None, [1.0] * 4, 0.0, 0.05) == [D.ROUTE_INT8] * 4


# ------------------------------------------------------------------------------- TDC / PDR


def test_tdc_golden_sequence():
    kv, _ = load_golden("tdc_sequence.txt")
    base = np.array([1, -1, 2, -2, 1, -1, 2, -2], np.float32) / 64
    cs = [float(c) for c in kv["c"]]
    xs = [np.ones(8, np.float32)] * len(cs)
    ds = [(np.float32(c) * base).astype(np.float32) for c in cs]
    r = T.run_block_loop(xs, ds, 0.05, 1.0, 0.0, 0.05, dtype="f32")
    assert r["decisions"] == kv["decisions"]
    want_routes = [None if t == "-" else [D.ROUTE_INT8 if t == "int8" else D.ROUTE_NVFP4] for t in kv["routes"]]
    assert r["routes"] == want_routes


def test_tdc_constant_delta_skips_forever():
    x = [np.ones(16, np.float32)] * 12
    d = [np.full(16, 0.125, np.float32)] * 12
    r = T.run_block_loop(x, d, 0.05, 1.0, 0.0, 0.05, dtype="f32")
    assert r["decisions"] == ["compute"] * 2 + ["skip"] * 10
    # a skip reuses the last computed delta exactly
    assert np.array_equal(r["outs"][5], x[5] + d[1])


def test_tdc_scaled_delta_similarity_exact():
    x = np.zeros(8, np.float32)
    dp = np.array([1, 2, -4, 8, 0.5, -1, 2, 4], np.float32)
    c = T.tdc_commit(x, x + 1.5 * dp, dp, dtype="f32")
    assert c["d"] == 0.5
    assert np.array_equal(c["delta"], 1.5 * dp)


def test_tdc_jump_forces_compute():
    x = [np.ones(8, np.float32)] * 6
    base = np.linspace(-1, 1, 8).astype(np.float32)
    d = [base, base, base * 3, base * 3, base * 3, base * 3]
    r = T.run_block_loop(x, d, 0.05, 1.0, 0.0, 0.05, dtype="f32")
    # steps 2,3 skip on d = 0 (the jump at step 2 is not seen); step 4 as well; the jump
    # is seen only by a compute step: here none is forced, so the cache keeps base
    assert r["decisions"][:3] == ["compute", "compute", "skip"]
    d2 = [base, base * 1.04, base * 3, base * 3, base * 3, base * 3]
    r2 = T.run_block_loop(x, d2, 0.05, 1.0, 0.0, 0.05, dtype="f32")
    # d = 0.04: skip once (e_acc 0.04), then compute (0.08 > 0.05), which sees the jump
    # (d = |3/1.04 - 1| = 1.88) and forces another compute
    assert r2["decisions"] == ["compute", "compute", "skip", "compute", "compute", "skip"]


def test_tdc_bf16_commit_and_skip_rounding():
    xi = synth.to_bf16_bits(np.float32([1.0, 2.0, -3.0, 0.0]))
    xo = synth.to_bf16_bits(np.float32([1.5, 2.015625, -2.0, 0.25]))
    c = T.tdc_commit(xi, xo, None, "bf16")
    assert F.bf16_bits_to_f32(c["delta"]).tolist() == [0.5, 0.015625, 1.0, 0.25]
    assert c["gamma"] == pytest.approx((0.5 + 0.015625 + 1.0 + 0.25) / 6.0)
    out = T.tdc_skip(xi, c["delta"], "bf16")
    assert F.bf16_bits_to_f32(out).tolist() == [1.5, 2.015625, -2.0, 0.25]


# ------------------------------------------------------------------------------- planted mistakes


def test_planted_fwht_sign_error_is_caught():
    def bad(x, b):
        y = D.block_fwht_f32(x, b).copy()
        y[..., 1::2] *= -1            # a - b written as b - a on the last stage
        return y
    assert not check_fwht(bad, 64)


def test_planted_fwht_missing_normalisation_is_caught():
    assert not check_fwht(lambda x, b: D.block_fwht_f32(x, b) * np.float32(math.sqrt(b)), 16)


def test_planted_ties_away_rounding_is_caught():
    def bad(y):
        r = D.quant_nvfp4(y)
        r = dict(r)
        r["codes"] = np.where(np.isin(np.abs(r["v"]), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]),
                              r["codes"] + 1, r["codes"]).astype(np.uint8)
        return r
    y = np.zeros((1, 16), np.float32)
    y[0, :4] = [6.0, 0.75, 2.5, 5.0]
    # 0.75, 2.5, 5.0 sit exactly on midpoints at s_b = 1: ties-away changes them
    good = D.quant_nvfp4(y, s_g=np.float32(1.0))
    bad_r = dict(good)
    bad_r["codes"] = np.where(np.isin(np.abs(good["v"]), [0.75, 2.5, 5.0]), good["codes"] + 1, good["codes"])
    assert not np.array_equal(bad_r["codes"], brute_e2m1(good["v"]))
    assert np.array_equal(good["codes"], brute_e2m1(good["v"]))


def test_planted_wrong_tensor_scale_constant_is_caught(monkeypatch):
    """s_g = amax / 448 (the E2M1 factor 6 dropped) is caught by the top-scale pin."""
    monkeypatch.setattr(D, "FP4_X_E4M3", np.float32(448.0))
    assert not check_nvfp4_codes(D.quant_nvfp4)


def test_planted_scale_truncation_is_caught(monkeypatch):
    """E4M3 scales truncated instead of rounded to nearest are caught by brute force."""
    real = F.e4m3_encode_nonneg

    def trunc(v):
        c = real(v)
        below = F.E4M3_VALUES[c] > np.asarray(v, np.float32).astype(np.float64)
        return np.where(below & (c > 0), c - 1, c).astype(np.uint8)
    monkeypatch.setattr(F, "e4m3_encode_nonneg", trunc)
    assert not check_nvfp4_codes(D.quant_nvfp4)


def test_planted_missing_tensor_scale_in_v_is_caught(monkeypatch):
    """v = y / dec(s_b) (s_g forgotten) is caught by the |v| ~ 6 pin."""
    real = D.quant_nvfp4

    def bad(y, s_g=None):
        r = dict(real(y, s_g))
        r["v"] = (r["v"] * r["s_g"]).astype(np.float32)
        r["codes"] = np.where(r["zero_blk"].repeat(16, axis=1), 0, F.e2m1_encode(r["v"])).astype(np.uint8)
        return r
    assert not check_nvfp4_codes(bad)


def test_planted_transposed_operand_is_caught():
    g = synth.rng(30)
    a = g.integers(-5, 5, (4, 4)).astype(np.int8)
    b = g.integers(-5, 5, (4, 4)).astype(np.int8)
    acc_bad = np.asarray(a, np.int64) @ np.asarray(b, np.int64)   # B not transposed
    naive = np.array([[sum(int(a[m, k]) * int(b[n, k]) for k in range(4)) for n in range(4)] for m in range(4)])
    assert np.array_equal(D.gemm_int8_acc(a, b), naive)
    assert not np.array_equal(acc_bad, naive)


# ----------------------------------------------------------------------------------------
# GELU (erf form) of the FFN between the up and down projections
# ----------------------------------------------------------------------------------------


def test_gelu_erf_matches_integrated_normal_density():
    """x * Phi(x) with Phi obtained by quadrature of the standard normal density (no erf)."""
    from scipy.integrate import quad
    xs = np.array([-6.0, -3.0, -1.5, -0.7, -0.1, 0.0, 0.05, 0.3, 1.0, 2.2, 4.0])
    pdf = lambda t: math.exp(-0.5 * t * t) / math.sqrt(2.0 * math.pi)
    for x in xs:
        phi = quad(pdf, -np.inf, x, epsabs=1e-15, epsrel=1e-13)[0]
        assert D.gelu_erf(np.array([x]))[0] == pytest.approx(x * phi, rel=1e-10, abs=1e-15)


def test_gelu_erf_table_values_and_identities():
    # Phi(1) = 0.8413447461, Phi(-1) = 0.1586552539, Phi(2) = 0.9772498681 (normal tables)
    g = D.gelu_erf(np.array([1.0, -1.0, 2.0, 0.0]))
    assert g[0] == pytest.approx(0.8413447461, abs=1e-10)
    assert g[1] == pytest.approx(-0.1586552539, abs=1e-10)
    assert g[2] == pytest.approx(2 * 0.9772498681, abs=1e-9)
    assert g[3] == 0.0
    x = synth.rng(5).normal(0, 3, 1000)
    # Phi(x) + Phi(-x) = 1  =>  GELU(x) - GELU(-x) = x
    assert np.allclose(D.gelu_erf(x) - D.gelu_erf(-x), x, rtol=0, atol=1e-13)
    # far tail: Phi(-10) = 7.6198530241605e-24 keeps its relative accuracy
    assert D.gelu_erf(np.array([-10.0]))[0] == pytest.approx(-10 * 7.6198530241605e-24, rel=1e-9)


def test_planted_tanh_gelu_is_caught():
    """The tanh approximation of GELU is a different function: the quadrature pin rejects it."""
    x = np.linspace(-4, 4, 81)
    tanh_form = 0.5 * x * (1 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3)))
    assert np.max(np.abs(tanh_form - D.gelu_erf(x))) > 1e-4


# ----------------------------------------------------------------------------------------
# INT8 weights derived from NVFP4-only weights
# ----------------------------------------------------------------------------------------


def _golden_nvfp4_to_int8():
    g, _ = load_golden("nvfp4_weight_to_int8.txt")
    codes = np.array([[int(v) for v in g["codes_row0"]], [int(v) for v in g["codes_row1"]]], np.uint8)
    sf = np.array([[int(v, 16) for v in g["sf_row0"]], [int(v, 16) for v in g["sf_row1"]]], np.uint8)
    return g, codes, sf, np.float32(g["s_g"][0])


def test_nvfp4_weight_to_int8_worked_example():
    g, codes, sf, sg = _golden_nvfp4_to_int8()
    r = D.nvfp4_weight_to_int8(codes, sf, sg)
    assert r["q"][0].tolist() == [int(v) for v in g["q_row0"]]
    assert r["q"][1].tolist() == [int(v) for v in g["q_row1"]]
    num, den = (np.float32(v) for v in g["scale_row0"])
    assert r["scale"][0] == num / den and r["scale"][1] == 0


def test_nvfp4_weight_to_int8_scales_with_the_tensor_scale():
    """A power-of-two tensor scale changes no code and scales the row scale exactly."""
    g = synth.rng(71)
    codes = g.integers(0, 16, (6, 64)).astype(np.uint8)
    sf = g.integers(0x20, 0x50, (6, 4)).astype(np.uint8)
    a = D.nvfp4_weight_to_int8(codes, sf, np.float32(0.25))
    b = D.nvfp4_weight_to_int8(codes, sf, np.float32(4.0))
    assert np.array_equal(a["q"], b["q"])
    assert np.array_equal(b["scale"], a["scale"] * np.float32(16.0))


def test_nvfp4_weight_to_int8_error_bound():
    """|q s - w| <= s / 2 (plus the float32 rounding of 1/s) for the dequantised NVFP4 weight."""
    g = synth.rng(72)
    codes = g.integers(0, 16, (16, 128)).astype(np.uint8)
    sf = g.integers(0x18, 0x60, (16, 8)).astype(np.uint8)
    r = D.nvfp4_weight_to_int8(codes, sf, np.float32(0.01))
    w = D.dequant_nvfp4(codes, sf, np.float32(0.01))
    err = np.abs(r["q"].astype(np.float64) * r["scale"][:, None] - w)
    assert (err <= r["scale"][:, None] * (0.5 + 1e-5)).all()


def test_planted_wrong_block_scale_index_is_caught():
    g, codes, sf, sg = _golden_nvfp4_to_int8()
    r = D.nvfp4_weight_to_int8(codes, sf[:, ::-1].copy(), sg)     # the blocks' scales swapped
    assert r["q"][0].tolist() != [int(v) for v in g["q_row0"]]


# ----------------------------------------------------------------------------------------
# PDR outlier ratio and the BF16 route
# ----------------------------------------------------------------------------------------


def test_outlier_ratio_hand_counted():
    """n = 1000 values: 990 ones and 10 spikes of 40.  Sum of squares 990 + 10 * 1600 = 16990,
    RMS = sqrt(16.99) = 4.1219, 6 RMS = 24.73: the 10 spikes exceed it, the ones do not."""
    x = np.ones(1000)
    x[::100] = 40.0
    assert D.outlier_ratio(x) == 10 / 1000
    x[::100] = -40.0                                  # the sign does not matter
    assert D.outlier_ratio(x) == 10 / 1000
    # spikes of 20 (< 6 RMS = 6 sqrt((990 + 4000) / 1000) = 13.40)? 20 > 13.40: still outliers
    x[::100] = 20.0
    assert D.outlier_ratio(x) == 10 / 1000
    # spikes of 5: RMS = sqrt((990 + 250) / 1000) = 1.1136, 6 RMS = 6.68 > 5: none
    x[::100] = 5.0
    assert D.outlier_ratio(x) == 0.0
    assert D.outlier_ratio(np.zeros(7)) == 0.0 and D.outlier_ratio(np.zeros(0)) == 0.0
    # spikes of 7 sit between 6 mean|x| (6.36) and 6 RMS (6 sqrt(1.48) = 7.30): an RMS rule
    # counts none, a mean-|x| rule would count all ten
    x[::100] = 7.0
    assert D.outlier_ratio(x) == 0.0


def test_outlier_ratio_gaussian_tail():
    """For N(0,1) data RMS -> 1, and the ratio at k = 2 tends to P(|Z| > 2) = 0.0455 (tables)."""
    z = synth.rng(73).standard_normal(2_000_000)
    assert D.outlier_ratio(z, 2.0) == pytest.approx(0.0455, abs=1.5e-3)


def test_route_layers_pdr_override():
    assert D.route_layers_pdr(0.01, [1, 1], [0, 0], [0.05, 0.05], 0.02, 0.01) == [D.ROUTE_BF16] * 2
    assert D.route_layers_pdr(0.01, [1, 1], [0, 0], [0.05, 0.05], 0.01, 0.01) == [D.ROUTE_NVFP4] * 2  # strict >
    assert D.route_layers_pdr(None, [1], [0], [0.05], 0.0, math.inf) == [D.ROUTE_INT8]


def test_gemm_bf16_small_brute_force():
    x = np.array([[1.0, 2.0, -1.0], [0.5, 0.0, 4.0]])
    w = np.array([[1.0, 1.0, 1.0], [2.0, -1.0, 0.25], [0.0, 3.0, -2.0], [1.0, 0.0, 0.0]])
    want = np.array([[2.0, -0.25, 8.0, 1.0], [4.5, 2.0, -8.0, 0.5]])        # worked by hand
    assert np.array_equal(D.gemm_bf16(x, w), want)
    assert np.array_equal(D.gemm_bf16(x, w, bias=np.array([1.0, 0, 0, -1])), want + [1.0, 0, 0, -1])
