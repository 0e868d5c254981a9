"""Pins of the oracle's rounding-boundary margins (CPU only).

The GPU parity tests exempt from the bit-exact comparison only the codes, scales, routes and
skip decisions whose oracle pre-rounding value lies within 1e-5 (relative) of a rounding
boundary.  The helpers that measure that distance decide what is exempt, so each is pinned
here against values worked by hand (tests/golden/rounding_margins.txt), against the rounding
functions themselves (a value whose margin is clear of 1e-5 keeps its code under a relative
perturbation of 1e-6; a value on a boundary has margin 0), and against planted mistakes that
a plausible slip would make (an absolute instead of a relative band, the wrong neighbouring
boundary, a dropped term, a margin that is infinite too often).
"""
from __future__ import annotations

import math

import numpy as np
import pytest

from conftest import load_golden
from oracle import dmpq as D
from oracle import formats as F
from oracle import tdc as T

EXEMPT = 1e-5


def _rows():
    _, rows = load_golden("rounding_margins.txt")
    return rows


def _margin(helper: str, arg: str, fns=None) -> float:
    fns = fns or {}
    if helper == "e2m1":
        return float(fns.get("e2m1", F.e2m1_rounding_margin)(np.array([np.float32(arg)]))[0])
    if helper == "e4m3":
        return float(fns.get("e4m3", F.e4m3_rounding_margin)(np.array([np.float32(arg)]))[0])
    if helper == "int8":
        return float(fns.get("int8", D.int8_rounding_margin)(np.array([np.float32(arg)]))[0])
    if helper == "route":
        g, a, b, t = map(float, arg.split(","))
        return float(fns.get("route", D.route_margin)(g, a, b, t))
    if helper == "decision":
        n, e, d, tau = arg.split(",")
        st = T.TdcState(n_computed=int(n), e_acc=float(e), d=float(d))
        return float(fns.get("decision", T.decision_margin)(st, float(tau)))
    raise KeyError(helper)


def _mismatches(fns=None) -> list:
    """Fixture rows whose margin or exemption the helpers (or substitutes for them) miss."""
    bad = []
    for helper, arg, want, exempt in _rows():
        got = _margin(helper, arg, fns)
        w = float(want)
        ok_value = (math.isinf(w) and math.isinf(got)) or (not math.isinf(got) and abs(got - w) <= 1e-6 * abs(w) + 1e-12)
        ok_exempt = (got <= EXEMPT) == (exempt == "1")
        if not (ok_value and ok_exempt):
            bad.append((helper, arg, want, got))
    return bad


def test_margins_match_the_worked_values():
    assert len(_rows()) >= 25
    assert _mismatches() == []


# --------------------------------------------------------- consistency with the rounding rules


def test_e2m1_margin_detects_every_code_change():
    """Across the whole E2M1 range: a value whose margin exceeds 2e-6 keeps its code when moved by
    1e-6 relative either way, and every midpoint of the grid has margin 0."""
    g = np.random.default_rng(3)
    v = np.concatenate([g.uniform(-7, 7, 200000), g.uniform(-0.3, 0.3, 50000)]).astype(np.float32)
    m = F.e2m1_rounding_margin(v)
    clear = m > 2e-6
    for f in (1 + 1e-6, 1 - 1e-6):
        moved = F.e2m1_encode((v.astype(np.float64) * f).astype(np.float32))
        assert np.array_equal(moved[clear], F.e2m1_encode(v)[clear])
    mids = 0.5 * (F.E2M1_MAGNITUDES[:-1] + F.E2M1_MAGNITUDES[1:])
    assert np.all(F.e2m1_rounding_margin(np.concatenate([mids, -mids]).astype(np.float32)) == 0)
    # and a value just past a midpoint does change code: the boundaries are where the margin is 0
    for mid in mids:
        lo, hi = np.float32(mid * (1 - 1e-6)), np.float32(mid * (1 + 1e-6))
        assert F.e2m1_encode(np.array([lo]))[0] != F.e2m1_encode(np.array([hi]))[0]


def test_e4m3_margin_detects_every_code_change():
    """Over the E4M3 range (subnormals to the top binade): clear of 2e-6 means the scale code
    survives a 1e-6 relative move; the midpoints themselves have margin 0."""
    g = np.random.default_rng(4)
    v = np.exp(g.uniform(np.log(2.0 ** -11), np.log(448.0), 300000)).astype(np.float32)
    m = F.e4m3_rounding_margin(v)
    clear = m > 2e-6
    base = F.e4m3_encode_nonneg(v)
    for f in (1 + 1e-6, 1 - 1e-6):
        moved = F.e4m3_encode_nonneg((v.astype(np.float64) * f).astype(np.float32))
        assert np.array_equal(moved[clear], base[clear])
    pos = F.E4M3_VALUES[:127]
    mids = (0.5 * (pos[:-1] + pos[1:])).astype(np.float32)
    assert np.all(F.e4m3_rounding_margin(mids) == 0)


def test_int8_margin_detects_every_code_change():
    """Round-half-even to integers over the INT8 range: clear of 2e-6 keeps the integer under a
    1e-6 relative move; every half-integer has margin 0."""
    g = np.random.default_rng(5)
    v = g.uniform(-127.4, 127.4, 300000).astype(np.float32)
    m = D.int8_rounding_margin(v)
    clear = m > 2e-6
    for f in (1 + 1e-6, 1 - 1e-6):
        moved = np.rint((v.astype(np.float64) * f).astype(np.float32))
        assert np.array_equal(moved[clear], np.rint(v)[clear])
    halves = np.arange(-126.5, 127.0, 1.0).astype(np.float32)
    assert np.all(D.int8_rounding_margin(halves) == 0)


def test_route_margin_detects_every_route_change():
    """A route whose margin exceeds 2e-6 does not flip when Gamma moves by 1e-6 relative."""
    g = np.random.default_rng(6)
    for _ in range(20000):
        gam, a, b, thr = g.uniform(0, 0.2), g.uniform(0.5, 2), g.uniform(-0.05, 0.05), g.uniform(0.01, 0.1)
        if D.route_margin(gam, a, b, thr) > 2e-6 * (1 + abs(a * gam) / thr):
            r = D.route_layers(gam, a, b, thr)
            assert D.route_layers(gam * (1 + 1e-6), a, b, thr) == r
            assert D.route_layers(gam * (1 - 1e-6), a, b, thr) == r


def test_decision_margin_detects_every_skip_change():
    """Finite exactly when the skip rule is in force (two computed deltas, finite d), and a
    decision clear of 2e-6 does not flip when e_acc + d moves by 1e-6 relative."""
    g = np.random.default_rng(7)
    assert T.decision_margin(T.TdcState(n_computed=0), 0.05) == math.inf
    assert T.decision_margin(T.TdcState(n_computed=1, d=0.01), 0.05) == math.inf
    for _ in range(20000):
        st = T.TdcState(n_computed=int(g.integers(2, 10)), e_acc=g.uniform(0, 0.05), d=g.uniform(0, 0.05))
        tau = g.uniform(0.02, 0.1)
        m = T.decision_margin(st, tau)
        assert math.isfinite(m)
        if m > 2e-6:
            dec = T.tdc_decide(st, tau)
            for f in (1 + 1e-6, 1 - 1e-6):
                moved = T.TdcState(n_computed=st.n_computed, e_acc=st.e_acc * f, d=st.d * f)
                assert T.tdc_decide(moved, tau) == dec


# --------------------------------------------------------------------- planted mistakes


def _e2m1_absolute(v):
    a = np.abs(np.asarray(v, np.float32).astype(np.float64))
    mids = 0.5 * (F.E2M1_MAGNITUDES[:-1] + F.E2M1_MAGNITUDES[1:])
    return np.min(np.abs(a[..., None] - mids), axis=-1)


def _e4m3_wrong_neighbour(v):
    a = np.asarray(v, np.float32).astype(np.float64)
    grid = F.E4M3_VALUES[:127]
    mids = 0.5 * (grid[:-1] + grid[1:])
    idx = np.clip(np.searchsorted(mids, a), 0, len(mids) - 2)
    return np.minimum(np.abs(a - mids[idx]) / mids[idx], np.abs(a - mids[idx + 1]) / mids[idx + 1])


def _int8_absolute(v):
    v = np.asarray(v, np.float32).astype(np.float64)
    return np.abs(v - (np.floor(v) + 0.5))


def _route_without_beta(gamma, alpha, beta, thr):
    return abs(alpha * gamma - thr) / abs(thr)


def _decision_inf_too_often(st, tau):
    if st.n_computed < 3 or not math.isfinite(st.d):
        return math.inf
    return abs(st.e_acc + st.d - tau) / tau


@pytest.mark.parametrize("helper,wrong", [("e2m1", _e2m1_absolute), ("e4m3", _e4m3_wrong_neighbour),
                                          ("int8", _int8_absolute), ("route", _route_without_beta),
                                          ("decision", _decision_inf_too_often)])
def test_planted_margin_mistakes_are_caught(helper, wrong):
    assert [b for b in _mismatches({helper: wrong}) if b[0] == helper], f"a wrong {helper} margin passed"
