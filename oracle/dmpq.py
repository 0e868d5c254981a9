"""Dynamic Mixed-Precision Quantisation (DMPQ) path of one routed linear layer -- oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).  Plain numpy, float64 / int64 for
the exact quantities, float32 exactly where the method's quantiser computes in float32.

Passages restated (6Bit-Diffusion, arXiv 2603.18742):

* gist.science (EN) "2. Methodology", A. DMPQ, Mechanism 1-3: the predictor Gamma is the
  relative L1 distance between a block's input and output; a pre-fitted linear model
  E_rel = alpha * Gamma + beta predicts the quantisation error; a layer whose predicted
  error exceeds a threshold is routed to INT8, otherwise to NVFP4.
* gist.science (IT) "2. Metodologia Proposta", A: Gamma_{t-1} is the relative L1 distance
  between output and input of the block at the previous step.
* gist.science (EN) A, "Outlier Smoothing"; (ZH) 2.A: an online block Hadamard (fast
  Hadamard) transform over local activation blocks.
* gist.science (ZH) 2.A "weight handling": weights are quantised offline.
* NVFP4 is E2M1 with micro-scaled blocks (gist.science IT, "Contributi Chiave" 4).

Readings where the pages are silent (all listed in the design notes of the repository):
Gamma is one scalar per block and step over the whole activation tensor; "exceeds" is
strict (>); a missing Gamma routes to INT8 (gist.science EN, C. PDR, second bullet); the
Hadamard is the Sylvester matrix in natural order, normalised by 1/sqrt(b), applied to
both routes and to the weights along K; NVFP4 uses the two-level scale recipe (one fp32
tensor scale, one E4M3 scale per 16 elements); INT8 is per-token symmetric over +-127
with round-half-even.
"""
from __future__ import annotations

import math

import numpy as np

from . import formats as F

ROUTE_NVFP4 = 0
ROUTE_INT8 = 1
ROUTE_BF16 = 2

# ----------------------------------------------------------------------------------------
# Gamma predictor and routing
# ----------------------------------------------------------------------------------------


def gamma_rel_l1(x_in: np.ndarray, x_out: np.ndarray) -> float:
    """Gamma = sum|x_out - x_in| / sum|x_in| over every element, in float64.

    gist.science EN 2.A Mechanism 1; IT 2.A.  sum|x_in| == 0 gives 0 when the numerator
    is 0 too, else +inf.  The difference is taken in float64 of the stored values.
    """
    xi = np.asarray(x_in, dtype=np.float64)
    xo = np.asarray(x_out, dtype=np.float64)
    num = float(np.sum(np.abs(xo - xi)))
    den = float(np.sum(np.abs(xi)))
    if den == 0.0:
        return 0.0 if num == 0.0 else math.inf
    return num / den


def route_layers(gamma: float | None, alpha, beta, thr) -> list[int]:
    """Route each linear layer of a block from the block's Gamma of the previous step.

    gist.science EN 2.A Mechanism 2-3: E_rel = alpha * Gamma + beta; E_rel > thr -> INT8,
    else NVFP4.  ``gamma is None`` means the predictor is missing (first step of a block,
    or the previous step was skipped by the delta cache): every layer goes to INT8, the
    safe fallback of gist.science EN 2.C (PDR), second bullet.  E_rel in float64.
    """
    alpha = np.atleast_1d(np.asarray(alpha, dtype=np.float64))
    beta = np.atleast_1d(np.asarray(beta, dtype=np.float64))
    thr = np.atleast_1d(np.asarray(thr, dtype=np.float64))
    n = max(len(alpha), len(beta), len(thr))
    alpha, beta, thr = (np.broadcast_to(a, (n,)) for a in (alpha, beta, thr))
    if gamma is None:
        return [ROUTE_INT8] * n
    e = alpha * float(gamma) + beta
    return [ROUTE_INT8 if e[i] > thr[i] else ROUTE_NVFP4 for i in range(n)]


def outlier_ratio(x: np.ndarray, k_sigma: float = 6.0) -> float:
    """Fraction of the elements of a block activation with |x| > k_sigma * RMS(x), float64.

    gist.science EN 2.C (first bullet) and ZH 2.C: PDR forces full precision when a layer's
    input has a high outlier ratio, which the pages do not define.  Reading: RMS over the
    whole tensor, k_sigma = 6, strict >.  An empty or all-zero tensor has ratio 0.
    """
    x = np.asarray(x, np.float64).ravel()
    if x.size == 0:
        return 0.0
    rms = math.sqrt(float(np.sum(x * x)) / x.size)
    return float(np.count_nonzero(np.abs(x) > k_sigma * rms)) / x.size


def route_layers_pdr(gamma: float | None, alpha, beta, thr, ratio: float, rho: float) -> list[int]:
    """route_layers, overridden by the outlier-ratio rule of PDR (EN 2.C, ZH 2.C): a block whose
    input's outlier ratio exceeds rho (strict >) runs every layer in BF16.  rho = +inf turns
    the override off (the default of the workloads)."""
    routes = route_layers(gamma, alpha, beta, thr)
    return [ROUTE_BF16] * len(routes) if ratio > rho else routes


def route_margin(gamma: float, alpha: float, beta: float, thr: float) -> float:
    """|E_rel - thr| / thr: a route whose margin is <= 1e-5 is a borderline decision."""
    e = alpha * gamma + beta
    return abs(e - thr) / abs(thr) if thr != 0 else abs(e)


# ----------------------------------------------------------------------------------------
# Block Hadamard transform
# ----------------------------------------------------------------------------------------


def hadamard_sylvester(b: int) -> np.ndarray:
    """Unnormalised Sylvester Hadamard matrix of order b (natural order), float64.

    Built by the doubling recursion H_2n = [[H_n, H_n], [H_n, -H_n]].
    """
    if b < 1 or b & (b - 1):
        raise ValueError("block size must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < b:
        h = np.block([[h, h], [h, -h]])
    return h


def block_hadamard_f64(x: np.ndarray, b: int) -> np.ndarray:
    """y = x (H_b / sqrt(b)) on every contiguous block of b along the last axis (float64).

    gist.science EN 2.A "Outlier Smoothing": a Hadamard transform over local activation
    blocks.  The matrix product is the definition; ``block_fwht_f32`` is the fast form.
    """
    x = np.asarray(x, dtype=np.float64)
    rows, k = x.reshape(-1, x.shape[-1]).shape
    if k % b:
        raise ValueError("K must be a multiple of the Hadamard block")
    h = hadamard_sylvester(b) / math.sqrt(b)
    y = x.reshape(rows, k // b, b) @ h        # H is symmetric
    return y.reshape(x.shape)


def block_fwht_f32(x: np.ndarray, b: int) -> np.ndarray:
    """Fast block Hadamard in float32, stage by stage, then the 1/sqrt(b) scale.

    Stage h = 1, 2, 4, ..., b/2: every pair (i, i+h) with bit h of i clear becomes
    (a + b, a - b), each a float32 add / subtract.  The result is multiplied by
    float32(1/sqrt(b)) (a power of two, hence exact, for b = 16 and 64).  This fixed
    stage order is what the quantisers compute in; it equals ``block_hadamard_f64`` up to
    float32 rounding.
    """
    x = np.asarray(x, dtype=np.float32)
    shape = x.shape
    rows, k = x.reshape(-1, shape[-1]).shape
    if k % b:
        raise ValueError("K must be a multiple of the Hadamard block")
    y = x.reshape(rows, k // b, b).copy()
    h = 1
    while h < b:
        y = y.reshape(rows, k // b, b // (2 * h), 2, h)
        a = y[:, :, :, 0, :].copy()
        c = y[:, :, :, 1, :].copy()
        y[:, :, :, 0, :] = a + c
        y[:, :, :, 1, :] = a - c
        y = y.reshape(rows, k // b, b)
        h *= 2
    y = y * np.float32(1.0 / math.sqrt(b))
    return y.reshape(shape).astype(np.float32)


# ----------------------------------------------------------------------------------------
# NVFP4 activation / weight quantisation
# ----------------------------------------------------------------------------------------

FP4_X_E4M3 = np.float32(6.0 * 448.0)     # 2688: largest E2M1 value times largest E4M3 value


def nvfp4_tensor_scale(y: np.ndarray) -> np.float32:
    """s_g = amax|y| / (6 * 448) over the whole tensor, one float32 division."""
    amax = np.float32(np.max(np.abs(np.asarray(y, dtype=np.float32)))) if y.size else np.float32(0)
    return np.float32(amax / FP4_X_E4M3)


def quant_nvfp4(y: np.ndarray, s_g: np.float32 | None = None) -> dict:
    """NVFP4-quantise an already transformed float32 tensor y [rows x K], K % 16 == 0.

    Two-level recipe (the pages give only "E2M1, micro-scaled"; this is the plain reading
    of one fp32 tensor scale and one E4M3 scale per 16 elements):

      s_g  = amax|y| / 2688                                   (float32; or the given s_g)
      sbf  = amax_b / (6 * s_g)           per 16-element block (float32: 6*s_g rounded,
                                                                then a division)
      s_b  = E4M3 round-nearest-even of sbf, saturating at 448
      bs   = dec(s_b) * s_g                                   (float32)
      v    = y * (1 / bs)                 (float32: reciprocal rounded, then a product)
      q    = E2M1 round-nearest-even of v, saturating at +-6

    s_g == 0 gives all scales and codes 0; a block whose s_b decodes to 0 gets codes 0.
    Returns codes [rows x K] (one code per byte, unpacked), sf [rows x K/16] E4M3 codes,
    s_g, and the pre-rounding values v and sbf (for the rounding-boundary exemption).
    """
    y = np.asarray(y, dtype=np.float32)
    rows, k = y.shape
    if k % 16:
        raise ValueError("K must be a multiple of 16")
    if s_g is None:
        s_g = nvfp4_tensor_scale(y)
    s_g = np.float32(s_g)
    yb = y.reshape(rows, k // 16, 16)
    amax_b = np.max(np.abs(yb), axis=2).astype(np.float32)
    if s_g == 0:
        sbf = np.zeros_like(amax_b)
        sf = np.zeros(amax_b.shape, dtype=np.uint8)
    else:
        six_sg = np.float32(np.float32(6.0) * s_g)
        sbf = (amax_b / six_sg).astype(np.float32)
        sf = F.e4m3_encode_nonneg(sbf)
    dec = F.E4M3_VALUES[sf].astype(np.float32)
    bs = (dec * s_g).astype(np.float32)
    zero_blk = bs == 0
    with np.errstate(divide="ignore"):
        inv = np.where(zero_blk, np.float32(0), np.float32(1.0) / np.where(zero_blk, 1, bs)).astype(np.float32)
    v = (yb * inv[:, :, None]).astype(np.float32)
    q = F.e2m1_encode(v)
    q = np.where(zero_blk[:, :, None], np.uint8(0), q).astype(np.uint8)
    return {
        "codes": q.reshape(rows, k),
        "sf": sf,
        "s_g": s_g,
        "v": v.reshape(rows, k),
        "sbf": sbf,
        "zero_blk": zero_blk,
    }


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Two E2M1 codes per byte along K: element 2i in the low nibble, 2i+1 in the high."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def dequant_nvfp4(codes: np.ndarray, sf: np.ndarray, s_g) -> np.ndarray:
    """dec(q) * dec(s_b) * s_g in float64 (codes unpacked [rows x K], sf [rows x K/16])."""
    rows, k = codes.shape
    val = F.E2M1_VALUES[codes].reshape(rows, k // 16, 16)
    sc = F.E4M3_VALUES[sf][:, :, None] * float(s_g)
    return (val * sc).reshape(rows, k)


# ----------------------------------------------------------------------------------------
# INT8 per-token (per-row) symmetric quantisation
# ----------------------------------------------------------------------------------------


def quant_int8_rows(y: np.ndarray) -> dict:
    """Per-row symmetric INT8 of an already transformed float32 tensor y [rows x K].

      s = amax_row|y| / 127            (float32 division)
      v = y * (1 / s)                  (float32: reciprocal rounded, then a product)
      q = clamp(round-half-even(v), -127, 127)

    amax_row == 0 gives s = 0 and q = 0.  The same function quantises weights per output
    channel (rows of W).
    """
    y = np.asarray(y, dtype=np.float32)
    amax = np.max(np.abs(y), axis=1).astype(np.float32) if y.shape[1] else np.zeros(y.shape[0], np.float32)
    s = (amax / np.float32(127.0)).astype(np.float32)
    zero = s == 0
    with np.errstate(divide="ignore"):
        inv = np.where(zero, np.float32(0), np.float32(1.0) / np.where(zero, 1, s)).astype(np.float32)
    v = (y * inv[:, None]).astype(np.float32)
    q = np.clip(np.rint(v), -127, 127).astype(np.int8)
    q[zero] = 0
    return {"q": q, "scale": s, "v": v}


def quant_int8_rows_given(y: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Per-row symmetric INT8 of a transformed float32 tensor y [rows x K] with given per-row
    scales s: the per-token rule of gist.science (EN) 2.A Mechanism 3 with the scale supplied
    instead of derived (the fused INT8 epilogue's input; delayed scales are not on the pages):

      v = y * (1 / s)                  (float32: reciprocal rounded, then a product)
      q = clamp(round-half-even(v), -127, 127)

    s == 0 gives q = 0.  With s = amax_row|y| / 127 this is ``quant_int8_rows``; a smaller s
    saturates the entries beyond 127 s.
    """
    y = np.asarray(y, dtype=np.float32)
    s = np.asarray(s, dtype=np.float32)
    zero = s == 0
    with np.errstate(divide="ignore"):
        inv = np.where(zero, np.float32(0), np.float32(1.0) / np.where(zero, 1, s)).astype(np.float32)
    v = (y * inv[:, None]).astype(np.float32)
    q = np.clip(np.rint(v), -127, 127).astype(np.int8)
    q[zero] = 0
    return q


def int8_rounding_margin(v: np.ndarray) -> np.ndarray:
    """Relative distance of v to the nearest half-integer (a round-half-even boundary)."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    m = np.floor(v) + 0.5
    return np.abs(v - m) / np.maximum(np.abs(m), 0.5)


def dequant_int8(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    return np.asarray(q, dtype=np.float64) * np.asarray(s, dtype=np.float64)[:, None]


# ----------------------------------------------------------------------------------------
# Quantised GEMMs  Y[m, n] = sum_k A[m, k] B[n, k]   (both operands K-major)
# ----------------------------------------------------------------------------------------


def gemm_int8_acc(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Exact integer accumulators acc[m, n] = sum_k a[m, k] * b[n, k] (int64)."""
    return np.asarray(a, dtype=np.int64) @ np.asarray(b, dtype=np.int64).T


def gemm_int8(a, a_scale, b, b_scale, bias=None) -> np.ndarray:
    """INT8 route output in float64: acc * s_a[m] * s_w[n] (+ bias[n])."""
    acc = gemm_int8_acc(a, b).astype(np.float64)
    y = acc * np.asarray(a_scale, np.float64)[:, None] * np.asarray(b_scale, np.float64)[None, :]
    if bias is not None:
        y = y + np.asarray(bias, np.float64)[None, :]
    return y


def gemm_nvfp4(a_codes, a_sf, a_sg, b_codes, b_sf, b_sg, bias=None) -> np.ndarray:
    """NVFP4 route output in float64: s_gA s_gB sum_k dec(qA) dec(sA) dec(qB) dec(sB)."""
    ad = dequant_nvfp4(a_codes, a_sf, 1.0)
    bd = dequant_nvfp4(b_codes, b_sf, 1.0)
    y = (ad @ bd.T) * (float(a_sg) * float(b_sg))
    if bias is not None:
        y = y + np.asarray(bias, np.float64)[None, :]
    return y


def gemm_bf16(x: np.ndarray, w: np.ndarray, bias=None) -> np.ndarray:
    """BF16 route (PDR full precision): Y = X W^T on the untransformed bf16 operands, float64."""
    y = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T
    if bias is not None:
        y = y + np.asarray(bias, np.float64)[None, :]
    return y


# ----------------------------------------------------------------------------------------
# One routed linear layer, end to end
# ----------------------------------------------------------------------------------------


def prepare_weight(w: np.ndarray, b: int) -> dict:
    """Offline weight preparation (gist.science ZH 2.A, weight handling): W [N x K] gets the
    same block Hadamard along K, then both an NVFP4 copy and a per-output-channel INT8
    copy, so that (X H)(W H)^T = X W^T."""
    wt = block_fwht_f32(np.asarray(w, np.float32), b)
    return {"nvfp4": quant_nvfp4(wt), "int8": quant_int8_rows(wt), "wt": wt}


def nvfp4_weight_to_int8(codes: np.ndarray, sf: np.ndarray, s_g) -> dict:
    """INT8 weights derived from NVFP4-only weights ([ZH] 2.A, weight handling: every weight is
    quantised offline to NVFP4, and converted only when a layer needs INT8 activations).

    Reading: the NVFP4 weight's value in float32 -- dec(code) * dec(block scale) is exact (at
    most 6 significant bits), then one rounding for the product with the tensor scale s_g --
    quantised per output channel like quant_int8_rows.  No second Hadamard transform: the
    NVFP4 weight is already in the rotated basis.  codes [rows x K] unpacked, sf [rows x K/16].
    """
    rows, k = codes.shape
    val = F.E2M1_VALUES[codes].astype(np.float32).reshape(rows, k // 16, 16)
    sc = F.E4M3_VALUES[sf].astype(np.float32)[:, :, None]
    w = ((val * sc).astype(np.float32) * np.float32(s_g)).astype(np.float32).reshape(rows, k)
    r = quant_int8_rows(w)
    r["w"] = w
    return r


def routed_linear(x: np.ndarray, wprep: dict, b: int, route: int) -> np.ndarray:
    """Y = quantised (X H)(W H)^T along the given route, float64."""
    y = block_fwht_f32(np.asarray(x, np.float32), b)
    if route == ROUTE_INT8:
        qa = quant_int8_rows(y)
        qw = wprep["int8"]
        return gemm_int8(qa["q"], qa["scale"], qw["q"], qw["scale"])
    qa = quant_nvfp4(y)
    qw = wprep["nvfp4"]
    return gemm_nvfp4(qa["codes"], qa["sf"], qa["s_g"], qw["codes"], qw["sf"], qw["s_g"])


def gelu_erf(x: np.ndarray) -> np.ndarray:
    """x * Phi(x) with Phi the standard normal CDF, float64: the FFN activation of the
    CogVideoX-shaped block (erf form, not the tanh approximation).  Phi(x) is written as
    erfc(-x / sqrt 2) / 2, which equals (1 + erf(x / sqrt 2)) / 2 without the cancellation of
    the latter for large negative x."""
    from scipy.special import erfc
    x = np.asarray(x, np.float64)
    return 0.5 * x * erfc(-x / math.sqrt(2.0))
