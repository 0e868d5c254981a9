"""Temporal Delta Cache (TDC) and Purified Delta Refresh (PDR) -- oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Passages restated (6Bit-Diffusion, arXiv 2603.18742):

* gist.science EN 2.B: the residual delta of a block is Delta_t = X_out - X_in; the
  similarity of the last two computed deltas (Delta_{t-1}, Delta_{t-2}) is monitored; if
  it is high the block is skipped and its output is the input plus the delta cached at
  the last full computation; an accumulated error tracks drift from consecutive skips and,
  once it exceeds a threshold, the cache is refreshed and the block recomputed.
* gist.science IT 2.B "Riuso": X_out,t ~= X_in,t + Delta_{t-1}.
* gist.science EN 2.C, second bullet; ZH 2.C third bullet: a block that resumes
  computing after a skip has no routing metric and falls back to INT8.

Readings where the pages are silent:
(i)   similarity is measured as a relative L1 distance d = |Delta_new - Delta_prev|_1 /
      |Delta_prev|_1 (the same form as Gamma); "similarity high" means d small;
(ii)  the accumulated error is the sum of d over the current run of skips, reset on a
      compute step;
(iii) a block skips iff e_acc + d <= tau ("exceeds" is strict), else it computes;
(iv)  the cached delta reused on a skip is the last computed one (D1);
(v)   the first two steps of a block always compute (two deltas are needed for d);
(vi)  deltas are stored in the activation type (bf16 for bf16 activations);
(vii) after a skip Gamma is missing, so the next compute step routes every layer to INT8
      (the PDR safe fallback) and its delta becomes the new cached delta.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import formats as F
from .dmpq import ROUTE_INT8, route_layers

COMPUTE = "compute"
SKIP = "skip"


def _as_f32(x, dtype: str) -> np.ndarray:
    return F.bf16_bits_to_f32(x) if dtype == "bf16" else np.asarray(x, dtype=np.float32)


def _store(v32: np.ndarray, dtype: str) -> np.ndarray:
    return F.f32_to_bf16_bits(v32) if dtype == "bf16" else v32.astype(np.float32)


def tdc_commit(x_in, x_out, d1_old, dtype: str = "bf16") -> dict:
    """Compute step: form the new delta, its similarity to the previous delta, and Gamma.

    delta   = store(x_out - x_in)              (float32 difference, then the storage type)
    gamma_t = sum|x_out - x_in| / sum|x_in|    (float64 over the float32 differences)
    d       = sum|delta - d1_old| / sum|d1_old| (float64, stored values; None if no d1_old)
    """
    xi = _as_f32(x_in, dtype)
    xo = _as_f32(x_out, dtype)
    diff = (xo - xi).astype(np.float32)
    delta = _store(diff, dtype)
    num = float(np.sum(np.abs(diff.astype(np.float64))))
    den = float(np.sum(np.abs(xi.astype(np.float64))))
    gamma = (0.0 if num == 0 else math.inf) if den == 0 else num / den
    d = None
    if d1_old is not None:
        dn = _as_f32(delta, dtype).astype(np.float64)
        dp = _as_f32(d1_old, dtype).astype(np.float64)
        n2 = float(np.sum(np.abs(dn - dp)))
        d2 = float(np.sum(np.abs(dp)))
        d = (0.0 if n2 == 0 else math.inf) if d2 == 0 else n2 / d2
    return {"delta": delta, "gamma": gamma, "d": d, "num": num, "den": den}


def tdc_skip(x_in, d1, dtype: str = "bf16") -> np.ndarray:
    """Skip step: X_out = X_in + D1 (float32 sum, then the storage type)."""
    return _store((_as_f32(x_in, dtype) + _as_f32(d1, dtype)).astype(np.float32), dtype)


@dataclass
class TdcState:
    """Per-block cache state: computed-delta count, accumulated error, last similarity,
    and the Gamma of the previous step (None when missing)."""
    n_computed: int = 0
    e_acc: float = 0.0
    d: float = math.inf
    gamma_prev: float | None = None
    history: list = field(default_factory=list)


def tdc_decide(state: TdcState, tau: float) -> str:
    """Skip or compute for the coming step (readings (iii) and (v) above)."""
    if state.n_computed < 2:
        return COMPUTE
    return SKIP if state.e_acc + state.d <= tau else COMPUTE


def decision_margin(state: TdcState, tau: float) -> float:
    """|e_acc + d - tau| / tau: a decision whose margin is <= 1e-5 is borderline."""
    if state.n_computed < 2 or not math.isfinite(state.d):
        return math.inf
    return abs(state.e_acc + state.d - tau) / tau


def tdc_apply(state: TdcState, decision: str, commit: dict | None = None) -> None:
    """Update the state after a step: a skip adds d to e_acc and drops Gamma; a compute
    resets e_acc, counts the delta, takes its similarity and its Gamma."""
    if decision == SKIP:
        state.e_acc += state.d
        state.gamma_prev = None
        return
    state.e_acc = 0.0
    state.n_computed += 1
    if commit["d"] is not None:
        state.d = commit["d"]
    state.gamma_prev = commit["gamma"]


def compute_routes(state: TdcState, alpha, beta, thr) -> list[int]:
    """Routes of a compute step: DMPQ from Gamma_{t-1}, or all-INT8 when it is missing."""
    return route_layers(state.gamma_prev, alpha, beta, thr)


class BlockLoop:
    """One block driven through denoising steps one step at a time (synthetic block).

    A computed step's output is x_in + delta_true (no trained block exists, the delta is
    given).  ``step`` returns the decision, the routes of a compute step (None on a skip), the
    Gamma it was routed with (None when missing), the decision margin and the step's output
    (None on a skip unless ``want_skip_output``).
    """

    def __init__(self, tau, alpha, beta, thr, dtype="bf16"):
        self.tau, self.alpha, self.beta, self.thr, self.dtype = tau, alpha, beta, thr, dtype
        self.st = TdcState()
        self.d1 = None

    def step(self, x_in, delta_true, want_skip_output: bool = True) -> dict:
        st, dtype = self.st, self.dtype
        dec = tdc_decide(st, self.tau)
        margin = decision_margin(st, self.tau)
        if dec == SKIP:
            out = tdc_skip(x_in, self.d1, dtype) if want_skip_output else None
            tdc_apply(st, SKIP)
            return {"decision": dec, "routes": None, "gamma": None, "margin": margin, "out": out}
        r = compute_routes(st, self.alpha, self.beta, self.thr)
        g = st.gamma_prev
        xo = _store((_as_f32(x_in, dtype) + _as_f32(delta_true, dtype)).astype(np.float32), dtype)
        c = tdc_commit(x_in, xo, self.d1, dtype)
        self.d1 = c["delta"]
        tdc_apply(st, COMPUTE, c)
        return {"decision": dec, "routes": r, "gamma": g, "margin": margin, "out": xo}


def run_block_loop(x_in_seq, delta_true_seq, tau, alpha, beta, thr, dtype="bf16") -> dict:
    """Drive one block through a sequence of denoising steps (synthetic block).

    ``x_in_seq[t]`` is the block input at step t; a computed step's output is
    x_in + delta_true_seq[t].  Returns the decision sequence, the routes of every compute
    step, the Gamma each compute step was routed with (None when missing), per-step outputs
    and decision margins.
    """
    loop = BlockLoop(tau, alpha, beta, thr, dtype)
    decisions, routes, outs, margins, gammas = [], [], [], [], []
    for xi, dt in zip(x_in_seq, delta_true_seq):
        r = loop.step(xi, dt)
        decisions.append(r["decision"])
        routes.append(r["routes"])
        gammas.append(r["gamma"])
        margins.append(r["margin"])
        outs.append(r["out"])
    return {"decisions": decisions, "routes": routes, "outs": outs, "margins": margins,
            "gammas": gammas}


__all__ = [
    "COMPUTE", "SKIP", "ROUTE_INT8", "TdcState", "tdc_commit", "tdc_skip", "tdc_decide",
    "tdc_apply", "compute_routes", "decision_margin", "BlockLoop", "run_block_loop",
]
