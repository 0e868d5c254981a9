"""C ABI checks that need no GPU: the library builds and loads, exports every symbol that
include/dit6.h declares, validates arguments on the host, and its host-side delta-cache and
routing logic agrees with the oracle."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import synth
from conftest import ROOT
from oracle import dmpq as D
from oracle import formats as F
from oracle import tdc as T


@pytest.fixture(scope="module")
def L():
    from int8_mixed_precision_gb300 import _lib, build
    if not os.path.exists(_lib.library_path()):
        try:
            build.build_library()
        except RuntimeError as e:          # no nvcc on this machine
            pytest.skip(str(e))
    return _lib.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dit6.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dit_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["dit_gamma_route", "dit_hadamard_quant_nvfp4", "dit_hadamard_quant_int8",
              "dit_qgemm_nvfp4", "dit_qgemm_nvfp4_amax", "dit_nvfp4_to_int8", "dit_qgemm_int8",
              "dit_outlier_ratio", "dit_gemm_bf16", "dit_route_host_pdr", "dit_tdc_step", "dit_sf_index", "dit_status_str",
              "dit_l1_partials", "dit_nvfp4_amax", "dit_shard_finish", "dit_shard_finish_host"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings(L):
    for code, name in enumerate(["DIT_OK", "DIT_ERR_INVALID_ARG", "DIT_ERR_ALIGNMENT", "DIT_ERR_UNSUPPORTED",
                                 "DIT_ERR_CUDA", "DIT_ERR_TIMEOUT"]):
        assert L.dit_status_str(code).decode() == name


def test_sf_index_matches_oracle_layout(L):
    for rows, k in [(256, 128), (300, 1920), (17, 64), (129, 7680)]:
        rp, cp = F.sf_padded_shape(rows, k)
        assert L.dit_sf_bytes(rows, k) == rp * cp
        rr, cc = np.meshgrid(np.arange(0, rp, 7), np.arange(cp), indexing="ij")
        want = F.sf_tiled_offset(rr, cc, rows, k)
        got = np.vectorize(lambda r, c: L.dit_sf_index(int(r), int(c), rows, k))(rr, cc)
        assert np.array_equal(got, want)
    assert L.dit_sf_index(0, 0, 10, 24) == -1       # k not a multiple of 16


def test_host_argument_validation_without_device_work(L):
    nul = None
    wsb = L.dit_workspace_bytes()
    fake_misaligned = ctypes.c_void_p(0x1001)
    ws = ctypes.c_void_p(0x2000)
    # null pointers, bad sizes, unsupported shapes and misalignment are rejected on the host
    assert L.dit_hadamard_quant_int8(nul, 1, 4, 128, 64, nul, 2, nul, nul) == 1
    assert L.dit_hadamard_quant_int8(fake_misaligned, 1, 4, 100, 64, fake_misaligned, 2, fake_misaligned, nul) == 3
    assert L.dit_hadamard_quant_int8(fake_misaligned, 1, 4, 128, 48, fake_misaligned, 2, fake_misaligned, nul) == 3
    assert L.dit_hadamard_quant_int8(fake_misaligned, 1, 4, 128, 64, fake_misaligned, 2, fake_misaligned, nul) == 2
    assert L.dit_hadamard_quant_int8(ws, 1, 4, 128, 64, ws, 0, ws, nul) == 1       # fp32 is no code container
    assert L.dit_hadamard_quant_int8(ws, 1, 4, 16448, 64, ws, 2, ws, nul) == 3     # a row wider than 16384
    assert L.dit_hadamard_quant_nvfp4(ws, 1, 4, 128, 64, nul, nul, nul, nul, ws, wsb, nul) == 1
    f = ctypes.c_float * 17
    assert L.dit_gamma_route(fake_misaligned, fake_misaligned, 1, 10, f(), f(), f(), 17, ws, ws, ws, wsb, nul) == 1
    assert L.dit_gamma_route(fake_misaligned, fake_misaligned, 1, 10, f(), f(), f(), 1, ws, ws, ws, wsb, nul) == 2
    # the workspace-free Gamma/route: null input, too many layers, misaligned input
    assert L.dit_gamma_route_noalloc(nul, ws, 1, 10, f(), f(), f(), 1, ws, ws, nul) == 1
    assert L.dit_gamma_route_noalloc(ws, ws, 1, 10, f(), f(), f(), 17, ws, ws, nul) == 1
    assert L.dit_gamma_route_noalloc(fake_misaligned, fake_misaligned, 1, 10, f(), f(), f(), 1, ws, ws, nul) == 2
    assert L.dit_qgemm_int8(fake_misaligned, ws, fake_misaligned, ws, 2, 4, 8, 100, nul, 0, ws, 1, nul, ws, wsb, nul) == 3
    assert L.dit_qgemm_int8(ws, ws, ws, ws, 0, 4, 8, 128, nul, 0, ws, 1, nul, ws, wsb, nul) == 1
    assert L.dit_qgemm_nvfp4(ws, ws, ws, ws, ws, ws, 4, 8, 96, nul, 0, ws, 1, ws, wsb, nul) == 3
    assert L.dit_qgemm_nvfp4(ws, ws, ws, ws, ws, ws, 4, 8, 128, nul, 0, ws, 1, ws, 100, nul) == 1
    # GEMM with its output's tensor scale: missing scale output, unsupported block, n % 64, misalignment
    G = L.dit_qgemm_nvfp4_amax
    assert G(ws, ws, ws, ws, ws, ws, 4, 128, 128, nul, 0, ws, 64, nul, ws, wsb, nul) == 1
    assert G(ws, ws, ws, ws, ws, ws, 4, 128, 128, nul, 0, ws, 128, ws, ws, wsb, nul) == 3
    assert G(ws, ws, ws, ws, ws, ws, 4, 96, 128, nul, 0, ws, 64, ws, ws, wsb, nul) == 3
    assert G(ws, ws, ws, ws, ws, ws, 4, 128, 128, nul, 0, fake_misaligned, 64, ws, ws, wsb, nul) == 2
    # NVFP4 -> INT8 weights: missing pointer, k not a multiple of 64, misaligned codes
    assert L.dit_nvfp4_to_int8(nul, ws, ws, 4, 128, ws, 2, ws, nul) == 1
    assert L.dit_nvfp4_to_int8(ws, ws, ws, 4, 96, ws, 2, ws, nul) == 3
    assert L.dit_nvfp4_to_int8(fake_misaligned, ws, ws, 4, 128, ws, 2, ws, nul) == 2
    # outlier ratio: null output, negative k; BF16 GEMM: n not a multiple of 8, misaligned bias
    assert L.dit_outlier_ratio(ws, 1, 64, 6.0, nul, nul, ws, wsb, nul) == 1
    assert L.dit_outlier_ratio(ws, 1, 64, -1.0, ws, nul, ws, wsb, nul) == 1
    assert L.dit_outlier_ratio(fake_misaligned, 1, 64, 6.0, ws, nul, ws, wsb, nul) == 2
    assert L.dit_gemm_bf16(ws, ws, 4, 12, 64, nul, 0, ws, 1, ws, wsb, nul) == 3
    assert L.dit_gemm_bf16(ws, ws, 4, 16, 64, fake_misaligned, 0, ws, 1, ws, wsb, nul) == 2
    # an activation code outside dit_act
    assert L.dit_qgemm_int8(ws, ws, ws, ws, 2, 4, 8, 128, nul, 5, ws, 1, nul, ws, wsb, nul) == 1
    assert L.dit_qgemm_nvfp4(ws, ws, ws, ws, ws, ws, 4, 8, 128, nul, 2, ws, 1, ws, wsb, nul) == 1
    # token-sharded form: bad mode, d1 == d_new, misaligned partials; finishing without inputs
    assert L.dit_l1_partials(2, ws, ws, nul, nul, 1, 64, ws, ws, wsb, nul) == 1
    assert L.dit_l1_partials(1, ws, ws, ws, ws, 1, 64, ws, ws, wsb, nul) == 1
    assert L.dit_l1_partials(0, ws, ws, nul, nul, 1, 64, ctypes.c_void_p(0x2004), ws, wsb, nul) == 2
    assert L.dit_nvfp4_amax(ws, 1, 4, 96, 64, ws, ws, wsb, nul) == 3
    assert L.dit_shard_finish(nul, 0, nul, nul, nul, nul, 0, nul, nul, nul, nul, nul) == 1
    assert L.dit_shard_finish(ws, 3, nul, nul, nul, nul, 0, ws, nul, nul, nul, nul) == 1
    assert L.dit_shard_finish(ws, 2, nul, nul, nul, nul, 0, nul, ws, nul, nul, nul) == 1   # sim needs 4 sums
    assert L.dit_shard_finish(nul, 0, ws, nul, nul, nul, 0, nul, nul, nul, nul, nul) == 1  # amax without output
    ws2 = ctypes.c_void_p(0x4000)
    assert L.dit_tdc_step(0, fake_misaligned, fake_misaligned, nul, ws, ws2, 1, 64, ws, ws, ws, wsb, nul) == 2
    assert L.dit_tdc_step(0, ws, ws, nul, ws, ws, 1, 64, ws, ws, ws, wsb, nul) == 1   # d1 == d_new
    assert L.dit_tdc_step(7, ws, ws, nul, ws, ws, 1, 64, ws, ws, ws, wsb, nul) == 1


def test_host_tdc_state_machine_matches_oracle(L):
    import int8_mixed_precision_gb300 as dit
    g = synth.rng(12)
    for trial in range(20):
        tau = float(g.choice([0.02, 0.05, 0.1]))
        st_c, st_o = dit.TdcState(), T.TdcState()
        for step in range(40):
            dc = st_c.decide(tau)
            do = T.tdc_decide(st_o, tau)
            assert (dc == dit.TDC_SKIP) == (do == T.SKIP)
            if do == T.SKIP:
                st_c.update(dit.TDC_SKIP)
                T.tdc_apply(st_o, T.SKIP)
                continue
            alpha, beta, thr = [1.0, 2.0], [0.0, 0.01], [0.05, 0.05]
            assert st_c.routes(alpha, beta, thr) == T.compute_routes(
                st_o, alpha, beta, np.float32(thr).astype(np.float64))
            gam = float(np.float32(g.uniform(0, 0.2)))
            d = float(np.float32(g.exponential(0.03))) if st_o.n_computed > 0 else None
            st_c.update(dit.TDC_COMMIT, gam, d)
            T.tdc_apply(st_o, T.COMPUTE, {"gamma": gam, "d": d})
            assert st_c.e_acc == st_o.e_acc and st_c.n_computed == st_o.n_computed


def test_host_tdc_golden_sequence(L):
    """The hand-worked sequence of tests/golden/tdc_sequence.txt through the C state machine,
    with Gamma and d taken from the oracle's commits."""
    import int8_mixed_precision_gb300 as dit
    from conftest import load_golden
    kv, _ = load_golden("tdc_sequence.txt")
    base = np.array([1, -1, 2, -2, 1, -1, 2, -2], np.float32) / 64
    x = np.ones(8, np.float32)
    st = dit.TdcState()
    d1 = None
    decisions, routes = [], []
    for c in [float(v) for v in kv["c"]]:
        if st.decide(0.05) == dit.TDC_SKIP:
            decisions.append("skip")
            routes.append("-")
            st.update(dit.TDC_SKIP)
            continue
        decisions.append("compute")
        routes.append("int8" if st.routes([1.0], [0.0], [0.05])[0] == dit.ROUTE_INT8 else "nvfp4")
        cm = T.tdc_commit(x, x + np.float32(c) * base, d1, "f32")
        st.update(dit.TDC_COMMIT, cm["gamma"], cm["d"])
        d1 = cm["delta"]
    assert decisions == kv["decisions"] and routes == kv["routes"]


def test_workspace_and_version(L):
    assert L.dit_workspace_bytes() >= 33 * 1024
    assert L.dit_ws_status_offset() == 0
    assert L.dit_version().decode().count(".") == 2


def test_tdc_state_round_trip(L):
    """The delta-cache decision state survives to_dict / from_dict: a restored copy makes the
    same decisions as the original from then on."""
    import int8_mixed_precision_gb300 as dit
    st = dit.TdcState()
    seq = [(0, 0.11, None), (0, 0.07, 0.02), (1,), (0, 0.05, 0.01)]
    for ev in seq:
        if ev[0] == dit.TDC_SKIP:
            st.update(dit.TDC_SKIP)
        else:
            st.update(dit.TDC_COMMIT, ev[1], ev[2])
    cp = dit.TdcState.from_dict(st.to_dict())
    assert cp.to_dict() == st.to_dict()
    for tau in (0.005, 0.02, 0.1):
        assert cp.decide(tau) == st.decide(tau)
    for s_ in (st, cp):
        s_.update(dit.TDC_SKIP)
    assert cp.to_dict() == st.to_dict() and cp.routes([1.0], [0.0], [0.05]) == st.routes([1.0], [0.0], [0.05])


def test_host_pdr_routes_match_oracle(L):
    """The host routing with the PDR outlier-ratio override against the oracle's."""
    import int8_mixed_precision_gb300 as dit
    g = synth.rng(74)
    for _ in range(200):
        st = dit.TdcState()
        gamma = None
        if g.random() < 0.8:
            gamma = float(g.random() * 0.2)
            st.update(dit.TDC_COMMIT, gamma, None)
        alpha, beta, thr = [1.0, 0.5], [0.0, 0.01], [0.05, 0.04]
        ratio, rho = float(g.random() * 0.02), float(g.choice([0.005, 0.01, math.inf]))
        f32 = lambda v: np.float32(v).astype(np.float64)      # the C interface takes float parameters
        want = D.route_layers_pdr(gamma, f32(alpha), f32(beta), f32(thr), ratio, rho)
        assert st.routes(alpha, beta, thr, ratio, rho) == want


def test_shard_finish_host_rules():
    """The finishing arithmetic of the token-sharded form on host values: Gamma and the
    similarity are fp64 ratios with the 0/0 -> 0 and x/0 -> +inf rule of the unsharded calls,
    routes follow E_rel > thr, and the tensor scale is amax / 2688 in one fp32 division."""
    import int8_mixed_precision_gb300 as dit
    r = dit.shard_finish_host([3.0, 60.0, 1.0, 8.0], 448.0, [1.0, 1.0], [0.0, 0.0], [0.05, 0.049])
    assert r["gamma"] == np.float32(0.05) and r["sim"] == 0.125
    assert r["routes"] == [D.ROUTE_NVFP4, D.ROUTE_INT8]      # 0.05 > 0.05 is false; > 0.049 true
    assert np.float32(r["tensor_scale"]) == np.float32(np.float32(448.0) / np.float32(2688.0))
    assert dit.shard_finish_host([0.0, 0.0, 5.0, 0.0])["gamma"] == 0.0
    assert math.isinf(dit.shard_finish_host([0.0, 0.0, 5.0, 0.0])["sim"])
    assert math.isinf(dit.shard_finish_host([1.0, 0.0])["gamma"])
    for amax in (0.0, 1e-30, 3.0e38, 6.0 * 448.0 * 1.7):
        assert np.float32(dit.shard_finish_host(amax=amax)["tensor_scale"]) == \
            D.nvfp4_tensor_scale(np.array([amax], np.float32))
