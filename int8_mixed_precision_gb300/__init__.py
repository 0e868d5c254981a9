"""Python binding of libdit6: the GB300 routed NVFP4/INT8 linear layer + Temporal Delta Cache.

Argument marshalling only: every step of the path runs in the CUDA kernels of
``csrc/`` behind the C ABI declared in ``include/dit6.h``.  PyTorch supplies device memory
and the current stream.  There is no fallback: if the library is missing, every call
raises ``LibraryMissing``.
"""
from __future__ import annotations

import ctypes
import math
import os

from ._lib import LibraryMissing, lib, library_path  # noqa: F401

ROUTE_NVFP4 = 0
ROUTE_INT8 = 1
ROUTE_BF16 = 2
TDC_COMMIT = 0
TDC_SKIP = 1
ACT_NONE = 0
ACT_GELU_ERF = 1
MAX_LAYERS = 16


class DitError(RuntimeError):
    pass


def _torch():
    import torch
    return torch


def _dt(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    if t.dtype == torch.int8:
        return 2
    raise DitError(f"unsupported dtype {t.dtype}")


def _p(t):
    """Device pointer of a buffer argument.  The kernels read every buffer as a dense array on
    the current device, so a host tensor or a strided view is refused here, before any launch."""
    if t is None:
        return None
    if not t.is_cuda:
        raise DitError(f"buffers must be CUDA tensors (got one on {t.device})")
    if not t.is_contiguous():
        raise DitError("buffers must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _need(t, nbytes: int, what: str) -> None:
    """Refuse a buffer smaller than the bytes the call will read or write."""
    if t is not None and t.numel() * t.element_size() < nbytes:
        raise DitError(f"{what}: {t.numel() * t.element_size()} bytes, the call needs {nbytes}")


def _same_device(*ts) -> None:
    devs = {t.device for t in ts if t is not None}
    if len(devs) > 1:
        raise DitError(f"buffers on different devices: {sorted(str(d) for d in devs)}")


def _bias_ok(bias, n: int) -> None:
    if bias is not None:
        if bias.dtype != _torch().float32:
            raise DitError("bias must be float32")
        _need(bias, 4 * n, "bias")


def _nvfp4_gemm_args(a, a_sf, a_gs, b, b_sf, b_gs, bias):
    if a.dim() != 2 or b.dim() != 2 or b.shape[1] != a.shape[1]:
        raise DitError("NVFP4 GEMM: a [m, k/2] and b [n, k/2] packed codes with the same k")
    m, n, k = a.shape[0], b.shape[0], a.shape[1] * 2
    _need(a_sf, sf_bytes(m, k), "a_sf")
    _need(b_sf, sf_bytes(n, k), "b_sf")
    _need(a_gs, 4, "a_gs")
    _need(b_gs, 4, "b_gs")
    _bias_ok(bias, n)
    return m, n, k


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, what: str) -> None:
    if status != 0:
        raise DitError(f"{what}: {lib().dit_status_str(status).decode()}")


def status_str(code: int) -> str:
    return lib().dit_status_str(code).decode()


def version() -> str:
    return lib().dit_version().decode()


def workspace_bytes() -> int:
    return int(lib().dit_workspace_bytes())


def workspace(device="cuda"):
    """A zero-filled workspace buffer (uint8) for one stream of calls."""
    return _torch().zeros(workspace_bytes(), dtype=_torch().uint8, device=device)


def device_status(ws) -> int:
    """The OR of (1 << status) raised on the device since the workspace was last cleared
    (synchronises with the device)."""
    off = int(lib().dit_ws_status_offset())
    return int(ws[off:off + 4].view(_torch().int32).item())


def clear_device_status(ws) -> None:
    off = int(lib().dit_ws_status_offset())
    ws[off:off + 4].zero_()


def sf_bytes(rows: int, k: int) -> int:
    return int(lib().dit_sf_bytes(rows, k))


def sf_index(row: int, kblock: int, rows: int, k: int) -> int:
    return int(lib().dit_sf_index(row, kblock, rows, k))


# ----------------------------------------------------------------------------------------
# device entry points
# ----------------------------------------------------------------------------------------


def _gamma_args(x_in, x_out, n, gamma, routes):
    if x_out.dtype != x_in.dtype or x_out.numel() != x_in.numel():
        raise DitError("x_in and x_out must have the same dtype and size")
    _need(gamma, 4, "gamma")
    _need(routes, 4 * n, "routes")


def gamma_route(x_in, x_out, alpha, beta, thr, gamma, routes, ws, stream=None):
    """Gamma = |x_out - x_in|_1 / |x_in|_1 and per-layer routes (device outputs)."""
    n = len(alpha)
    arr = ctypes.c_float * max(n, 1)
    _gamma_args(x_in, x_out, n, gamma, routes)
    _same_device(x_in, x_out, gamma, routes, ws)
    st = lib().dit_gamma_route(_p(x_in), _p(x_out), _dt(x_in), x_in.numel(), arr(*alpha),
                               arr(*beta), arr(*thr), n, _p(gamma), _p(routes), _p(ws),
                               ws.numel(), _stream(stream))
    _check(st, "dit_gamma_route")


def gamma_route_noalloc(x_in, x_out, alpha, beta, thr, gamma, routes, stream=None):
    """Same as gamma_route, with the reduction scratch held inside the library (a fixed
    device array) instead of a caller workspace; for callers that cannot allocate.  Calls
    share that array, so calls running concurrently on different streams race."""
    n = len(alpha)
    arr = ctypes.c_float * max(n, 1)
    _gamma_args(x_in, x_out, n, gamma, routes)
    _same_device(x_in, x_out, gamma, routes)
    st = lib().dit_gamma_route_noalloc(_p(x_in), _p(x_out), _dt(x_in), x_in.numel(), arr(*alpha),
                                       arr(*beta), arr(*thr), n, _p(gamma), _p(routes), _stream(stream))
    _check(st, "dit_gamma_route_noalloc")


def hadamard_quant_nvfp4(x, hblock, codes, sf, tensor_scale, ws, tensor_scale_in=None, stream=None):
    rows, k = x.shape
    _need(codes, rows * k // 2, "codes")
    _need(sf, sf_bytes(rows, k), "sf")
    _need(tensor_scale, 4, "tensor_scale")
    _need(tensor_scale_in, 4, "tensor_scale_in")
    _same_device(x, codes, sf, tensor_scale, tensor_scale_in, ws)
    st = lib().dit_hadamard_quant_nvfp4(_p(x), _dt(x), rows, k, hblock, _p(codes), _p(sf),
                                        _p(tensor_scale), _p(tensor_scale_in), _p(ws), ws.numel(),
                                        _stream(stream))
    _check(st, "dit_hadamard_quant_nvfp4")


def hadamard_quant_int8(x, hblock, q, row_scale, stream=None):
    """q: int8 codes, or the same integers in a bf16 tensor (operands of the bf16-pipe GEMM)."""
    rows, k = x.shape
    if q.numel() < rows * k:
        raise DitError(f"q: {q.numel()} codes, the call writes {rows * k}")
    _need(row_scale, 4 * rows, "row_scale")
    _same_device(x, q, row_scale)
    st = lib().dit_hadamard_quant_int8(_p(x), _dt(x), rows, k, hblock, _p(q), _dt(q), _p(row_scale),
                                       _stream(stream))
    _check(st, "dit_hadamard_quant_int8")


def qgemm_nvfp4(a, a_sf, a_gs, b, b_sf, b_gs, y, ws, bias=None, act=ACT_NONE, stream=None):
    m, n, k = _nvfp4_gemm_args(a, a_sf, a_gs, b, b_sf, b_gs, bias)
    if y.numel() < m * n:
        raise DitError(f"y: {y.numel()} elements, the call writes {m * n}")
    _same_device(a, a_sf, a_gs, b, b_sf, b_gs, bias, y, ws)
    st = lib().dit_qgemm_nvfp4(_p(a), _p(a_sf), _p(a_gs), _p(b), _p(b_sf), _p(b_gs), m, n, k,
                               _p(bias), act, _p(y), _dt(y), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dit_qgemm_nvfp4")


def qgemm_nvfp4_amax(a, a_sf, a_gs, b, b_sf, b_gs, y, ws, hblock, tensor_scale_out, bias=None, act=ACT_NONE,
                     stream=None):
    """NVFP4 GEMM into bf16 y whose epilogue also writes y's NVFP4 tensor scale (the one
    hadamard_quant_nvfp4(y, hblock, ...) would derive) to tensor_scale_out (device float [1])."""
    m, n, k = _nvfp4_gemm_args(a, a_sf, a_gs, b, b_sf, b_gs, bias)
    _need(y, 2 * m * n, "y")
    _need(tensor_scale_out, 4, "tensor_scale_out")
    _same_device(a, a_sf, a_gs, b, b_sf, b_gs, bias, y, tensor_scale_out, ws)
    st = lib().dit_qgemm_nvfp4_amax(_p(a), _p(a_sf), _p(a_gs), _p(b), _p(b_sf), _p(b_gs), m, n, k, _p(bias), act,
                                    _p(y), hblock, _p(tensor_scale_out), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dit_qgemm_nvfp4_amax")


def qgemm_int8(a, a_scale, b, b_scale, y, ws, bias=None, acc_debug=None, act=ACT_NONE, stream=None):
    """a, b: int8 codes (IMMA path) or bf16-held integer codes (tcgen05 bf16 path)."""
    if a.dtype != b.dtype:
        raise DitError("qgemm_int8: a and b must use the same code container")
    if a.dim() != 2 or b.dim() != 2 or b.shape[1] != a.shape[1]:
        raise DitError("qgemm_int8: a [m, k] and b [n, k] codes with the same k")
    m, n, k = a.shape[0], b.shape[0], a.shape[1]
    _need(a_scale, 4 * m, "a_scale")
    _need(b_scale, 4 * n, "b_scale")
    _bias_ok(bias, n)
    if y.numel() < m * n:
        raise DitError(f"y: {y.numel()} elements, the call writes {m * n}")
    _need(acc_debug, 4 * m * n, "acc_debug")
    _same_device(a, a_scale, b, b_scale, bias, y, acc_debug, ws)
    st = lib().dit_qgemm_int8(_p(a), _p(a_scale), _p(b), _p(b_scale), _dt(a), m, n, k, _p(bias), act,
                              _p(y), _dt(y), _p(acc_debug), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dit_qgemm_int8")


def qgemm_int8_requant(a, a_scale, b, b_scale, next_scale, q_next, row_amax, ws, bias=None, act=ACT_NONE,
                       stream=None):
    """INT8 GEMM (bf16-held codes) whose epilogue quantises its output for the next INT8 layer
    with the caller's per-token scales next_scale [m]: q_next [m, n] receives the bf16-held codes
    dit_hadamard_quant_int8(output, 64) would write with those scales, row_amax [m] (zero-filled
    by the caller) the output's exact per-row max|H z| / 8."""
    if a.dtype != _torch().bfloat16 or b.dtype != _torch().bfloat16:
        raise DitError("qgemm_int8_requant: a and b must be bf16-held codes")
    if a.dim() != 2 or b.dim() != 2 or b.shape[1] != a.shape[1]:
        raise DitError("qgemm_int8_requant: a [m, k] and b [n, k] codes with the same k")
    m, n, k = a.shape[0], b.shape[0], a.shape[1]
    _need(a_scale, 4 * m, "a_scale")
    _need(b_scale, 4 * n, "b_scale")
    _need(next_scale, 4 * m, "next_scale")
    _need(row_amax, 4 * m, "row_amax")
    _need(q_next, 2 * m * n, "q_next")
    _bias_ok(bias, n)
    _same_device(a, a_scale, b, b_scale, bias, next_scale, q_next, row_amax, ws)
    st = lib().dit_qgemm_int8_requant(_p(a), _p(a_scale), _p(b), _p(b_scale), m, n, k, _p(bias), act,
                                      _p(next_scale), _p(q_next), _p(row_amax), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dit_qgemm_int8_requant")


def tdc_step(mode, x_in, ws, x_out=None, x_out_skip=None, d1=None, d_new=None, gamma=None,
             sim=None, stream=None):
    for name, t in (("x_out", x_out), ("x_out_skip", x_out_skip), ("d1", d1), ("d_new", d_new)):
        if t is not None and (t.dtype != x_in.dtype or t.numel() != x_in.numel()):
            raise DitError(f"tdc_step: {name} must have x_in's dtype and size")
    _need(gamma, 4, "gamma")
    _need(sim, 4, "sim")
    _same_device(x_in, x_out, x_out_skip, d1, d_new, gamma, sim, ws)
    st = lib().dit_tdc_step(mode, _p(x_in), _p(x_out), _p(x_out_skip), _p(d1), _p(d_new),
                            _dt(x_in), x_in.numel(), _p(gamma), _p(sim), _p(ws), ws.numel(),
                            _stream(stream))
    _check(st, "dit_tdc_step")


# ----------------------------------------------------------------------------------------
# token-sharded form: per-shard partials, all-reduced by the caller, then finished
# ----------------------------------------------------------------------------------------

L1_GAMMA = 0
L1_TDC_COMMIT = 1


def l1_partials(mode, x_in, x_out, partials, ws, d1=None, d_new=None, stream=None):
    """This shard's L1 sums into partials (device float64): [sum|x_out - x_in|, sum|x_in|] for
    L1_GAMMA; for L1_TDC_COMMIT also d_new = x_out - x_in (stored) and [sum|d_new - d1|,
    sum|d1|] (zeros without d1)."""
    for name, t in (("x_out", x_out), ("d1", d1), ("d_new", d_new)):
        if t is not None and (t.dtype != x_in.dtype or t.numel() != x_in.numel()):
            raise DitError(f"l1_partials: {name} must have x_in's dtype and size")
    if partials.dtype != _torch().float64:
        raise DitError("l1_partials: partials must be float64")
    _need(partials, 8 * (4 if mode == L1_TDC_COMMIT else 2), "partials")
    _same_device(x_in, x_out, d1, d_new, partials, ws)
    st = lib().dit_l1_partials(mode, _p(x_in), _p(x_out), _p(d1), _p(d_new), _dt(x_in), x_in.numel(),
                               _p(partials), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dit_l1_partials")


def nvfp4_amax(x, hblock, amax, ws, stream=None):
    """max|block Hadamard (x)| over this shard [rows x k] into amax (device float32 [1])."""
    rows, k = x.shape
    _need(amax, 4, "amax")
    _same_device(x, amax, ws)
    st = lib().dit_nvfp4_amax(_p(x), _dt(x), rows, k, hblock, _p(amax), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dit_nvfp4_amax")


def shard_finish(partials=None, amax=None, alpha=(), beta=(), thr=(), gamma=None, sim=None, routes=None,
                 tensor_scale=None, stream=None):
    """From all-reduced partials / amax (device): Gamma, the delta similarity, the routes and the
    NVFP4 tensor scale, with the arithmetic of the unsharded calls (device outputs)."""
    n = len(alpha)
    arr = ctypes.c_float * max(n, 1)
    npart = 0 if partials is None else (4 if partials.numel() >= 4 else 2)
    _same_device(partials, amax, gamma, sim, routes, tensor_scale)
    st = lib().dit_shard_finish(_p(partials), npart, _p(amax), arr(*alpha), arr(*beta), arr(*thr), n, _p(gamma),
                                _p(sim), _p(routes), _p(tensor_scale), _stream(stream))
    _check(st, "dit_shard_finish")


def shard_finish_host(partials=None, amax=None, alpha=(), beta=(), thr=()) -> dict:
    """The finishing arithmetic on host values (a list of 2 or 4 sums, a float amax)."""
    n = len(alpha)
    arr = ctypes.c_float * max(n, 1)
    p = None if partials is None else (ctypes.c_double * len(partials))(*[float(v) for v in partials])
    npart = 0 if partials is None else len(partials)
    am = None if amax is None else ctypes.byref(ctypes.c_float(float(amax)))
    g, sm, ts = ctypes.c_float(), ctypes.c_float(), ctypes.c_float()
    rt = (ctypes.c_int32 * max(n, 1))()
    st = lib().dit_shard_finish_host(p, npart, am, arr(*alpha), arr(*beta), arr(*thr), n,
                                     ctypes.byref(g) if p else None, ctypes.byref(sm) if npart == 4 else None,
                                     rt if (p and n) else None, ctypes.byref(ts) if am else None)
    _check(st, "dit_shard_finish_host")
    out = {}
    if p:
        out["gamma"] = g.value
        out["routes"] = list(rt)[:n]
        if npart == 4:
            out["sim"] = sm.value
    if am:
        out["tensor_scale"] = ts.value
    return out


# ----------------------------------------------------------------------------------------
# host-side delta-cache state machine (C implementation, no device work)
# ----------------------------------------------------------------------------------------


class TdcState(ctypes.Structure):
    _fields_ = [("n_computed", ctypes.c_int64), ("e_acc", ctypes.c_double),
                ("d", ctypes.c_double), ("gamma", ctypes.c_double), ("gamma_valid", ctypes.c_int)]

    def __init__(self):
        super().__init__()
        lib().dit_tdc_state_init(ctypes.byref(self))

    def decide(self, tau: float) -> int:
        return int(lib().dit_tdc_decide(ctypes.byref(self), tau))

    def update(self, mode: int, gamma: float = 0.0, sim: float | None = None) -> None:
        has = sim is not None
        lib().dit_tdc_update(ctypes.byref(self), mode, float(gamma), float(sim if has else math.inf),
                             int(has))

    def to_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}

    @classmethod
    def from_dict(cls, d: dict) -> "TdcState":
        st = cls()
        for name, _ in cls._fields_:
            setattr(st, name, d[name])
        return st

    def routes(self, alpha, beta, thr, outlier_ratio: float | None = None, rho: float = math.inf) -> list[int]:
        """Routes from Gamma; with an outlier ratio above rho every layer goes to BF16 (PDR)."""
        n = len(alpha)
        arr = ctypes.c_float * n
        out = (ctypes.c_int32 * n)()
        if outlier_ratio is None:
            lib().dit_route_host(ctypes.byref(self), arr(*alpha), arr(*beta), arr(*thr), n, out)
        else:
            lib().dit_route_host_pdr(ctypes.byref(self), arr(*alpha), arr(*beta), arr(*thr), n,
                                     float(outlier_ratio), float(rho), out)
        return list(out)


# ----------------------------------------------------------------------------------------
# buffer helpers (torch device memory) and one routed linear layer
# ----------------------------------------------------------------------------------------


def alloc_nvfp4(rows: int, k: int, device="cuda") -> dict:
    torch = _torch()
    return {"codes": torch.empty(rows, k // 2, dtype=torch.uint8, device=device),
            "sf": torch.empty(sf_bytes(rows, k), dtype=torch.uint8, device=device),
            "gs": torch.empty(1, dtype=torch.float32, device=device)}


def alloc_int8(rows: int, k: int, device="cuda", container: str = "bf16") -> dict:
    """INT8 codes in an int8 tensor, or in a bf16 tensor ("bf16": the fast GEMM path)."""
    torch = _torch()
    dt = torch.bfloat16 if container == "bf16" else torch.int8
    return {"q": torch.empty(rows, k, dtype=dt, device=device),
            "scale": torch.empty(rows, dtype=torch.float32, device=device)}


def outlier_ratio(x, ws, ratio, count=None, k_sigma: float = 6.0, stream=None):
    """ratio (device float [1]) = fraction of |x| > k_sigma * RMS(x); count (device int64 [1])."""
    _need(ratio, 4, "ratio")
    _need(count, 8, "count")
    _same_device(x, ratio, count, ws)
    st = lib().dit_outlier_ratio(_p(x), _dt(x), x.numel(), float(k_sigma), _p(ratio), _p(count), _p(ws),
                                 ws.numel(), _stream(stream))
    _check(st, "dit_outlier_ratio")


def gemm_bf16(x, w, y, ws, bias=None, act=ACT_NONE, stream=None):
    """The BF16 route: y = act(x w^T (+ bias)) on untransformed bf16 operands."""
    m, k = x.shape
    n = w.shape[0]
    if w.dim() != 2 or w.shape[1] != k:
        raise DitError("gemm_bf16: x [m, k] and w [n, k] with the same k")
    _bias_ok(bias, n)
    if y.numel() < m * n:
        raise DitError(f"y: {y.numel()} elements, the call writes {m * n}")
    _same_device(x, w, bias, y, ws)
    st = lib().dit_gemm_bf16(_p(x), _p(w), m, n, k, _p(bias), act, _p(y), _dt(y), _p(ws), ws.numel(),
                             _stream(stream))
    _check(st, "dit_gemm_bf16")


def nvfp4_to_int8(codes, sf, tensor_scale, q, row_scale, stream=None):
    """Per-output-channel INT8 (int8 or bf16-held codes in q) of NVFP4 weights [rows x K]."""
    rows, k = codes.shape[0], codes.shape[1] * 2
    _need(sf, sf_bytes(rows, k), "sf")
    _need(tensor_scale, 4, "tensor_scale")
    if q.numel() < rows * k:
        raise DitError(f"q: {q.numel()} codes, the call writes {rows * k}")
    _need(row_scale, 4 * rows, "row_scale")
    _same_device(codes, sf, tensor_scale, q, row_scale)
    st = lib().dit_nvfp4_to_int8(_p(codes), _p(sf), _p(tensor_scale), rows, k, _p(q), _dt(q), _p(row_scale),
                                 _stream(stream))
    _check(st, "dit_nvfp4_to_int8")


class QuantizedWeight:
    """A weight W [N x K] prepared offline: block Hadamard along K, then an NVFP4 copy and a
    per-output-channel INT8 copy, all on the device.  nvfp4_only=True keeps the NVFP4 copy
    alone; the INT8 weights are then derived from it when a layer routes INT8 (int8_into)."""

    def __init__(self, w, hblock: int, ws, int8_container: str = "bf16", nvfp4_only: bool = False,
                 keep_bf16: bool = False):
        """keep_bf16: also keep the untransformed weight in bf16, for the BF16 route of PDR."""
        n, k = w.shape
        self.n, self.k, self.hblock = n, k, hblock
        self.int8_container = int8_container
        self.bf16 = w.to(_torch().bfloat16).contiguous() if keep_bf16 else None
        self.nvfp4 = alloc_nvfp4(n, k, w.device)
        hadamard_quant_nvfp4(w, hblock, self.nvfp4["codes"], self.nvfp4["sf"], self.nvfp4["gs"], ws)
        self.int8 = None
        if not nvfp4_only:
            self.int8 = alloc_int8(n, k, w.device, int8_container)
            hadamard_quant_int8(w, hblock, self.int8["q"], self.int8["scale"])

    def without_int8(self) -> "QuantizedWeight":
        """The same weight with its NVFP4 copy only (shared, not copied)."""
        other = object.__new__(QuantizedWeight)
        other.__dict__.update(self.__dict__)
        other.int8 = None
        return other

    def resident_bytes(self) -> int:
        tensors = list(self.nvfp4.values()) + (list(self.int8.values()) if self.int8 else []) + \
            ([self.bf16] if self.bf16 is not None else [])
        return sum(t.numel() * t.element_size() for t in tensors)

    def int8_into(self, scratch, stream=None) -> dict:
        """The INT8 weights: the resident copy, or (NVFP4-only) converted into scratch, a dict
        like alloc_int8's with at least N rows, and returned as views of it."""
        if self.int8 is not None:
            return self.int8
        q, s = scratch["q"][:self.n], scratch["scale"][:self.n]
        nvfp4_to_int8(self.nvfp4["codes"], self.nvfp4["sf"], self.nvfp4["gs"], q, s, stream=stream)
        return {"q": q, "scale": s}


class RoutedLinear:
    """Y = quant(X H) quant(W H)^T along a route chosen per call; the activation buffers for
    both routes are allocated once for a maximum token count."""

    def __init__(self, weight: QuantizedWeight, max_tokens: int, ws, device="cuda", int8_scratch=None,
                 act_buffers=None):
        """int8_scratch: for NVFP4-only weights, a buffer (alloc_int8 of at least N rows x K)
        the INT8 weights are derived into on each INT8-routed call; several layers may share
        one.  Allocated here when not given.  act_buffers: (alloc_nvfp4, alloc_int8) buffers of
        at least max_tokens x K for the quantised activations, shared by layers whose calls are
        ordered on one stream; allocated here when not given."""
        self.w = weight
        self.ws = ws
        container = weight.int8_container
        if act_buffers is not None:
            self.a4, self.a8 = act_buffers
        else:
            self.a4 = alloc_nvfp4(max_tokens, weight.k, device)
            self.a8 = alloc_int8(max_tokens, weight.k, device, container)
        self.w8_scratch = None
        if weight.int8 is None:
            self.w8_scratch = int8_scratch if int8_scratch is not None else alloc_int8(weight.n, weight.k, device,
                                                                                      container)

    def __call__(self, x, route: int, y, bias=None, tensor_scale_in=None, act=ACT_NONE, stream=None):
        m = x.shape[0]
        w = self.w
        if route == ROUTE_BF16:
            if w.bf16 is None:
                raise DitError("BF16 route needs QuantizedWeight(..., keep_bf16=True)")
            gemm_bf16(x if x.dtype == _torch().bfloat16 else x.to(_torch().bfloat16), w.bf16, y, self.ws, bias=bias,
                      act=act, stream=stream)
            return y
        if route == ROUTE_INT8:
            q, s = self.a8["q"][:m], self.a8["scale"][:m]
            hadamard_quant_int8(x, w.hblock, q, s, stream=stream)
            w8 = w.int8_into(self.w8_scratch, stream=stream)
            qgemm_int8(q, s, w8["q"], w8["scale"], y, self.ws, bias=bias, act=act, stream=stream)
        else:
            c = self.a4["codes"][:m]
            hadamard_quant_nvfp4(x, w.hblock, c, self.a4["sf"], self.a4["gs"], self.ws,
                                 tensor_scale_in=tensor_scale_in, stream=stream)
            qgemm_nvfp4(c, self.a4["sf"], self.a4["gs"], w.nvfp4["codes"], w.nvfp4["sf"],
                        w.nvfp4["gs"], y, self.ws, bias=bias, act=act, stream=stream)
        return y


# ----------------------------------------------------------------------------------------
# one DiT block under the Temporal Delta Cache with PDR routing (host control, device data)
# ----------------------------------------------------------------------------------------


class DeltaCachedBlock:
    """Drives one block through denoising steps: skip (X_out = X_in + cached delta) or compute
    (routed linears + delta commit), with the decision and PDR routing of the C state machine.

    Gamma and the delta similarity come back from the device in bulk: call ``absorb`` with the
    host copies after the step (``gamma_dev``/``sim_dev`` are slots of caller-owned arrays),
    so a denoising step needs one device-to-host copy for all blocks.
    """

    def __init__(self, n_elems: int, dtype, tau: float, alpha, beta, thr, ws, gamma_dev, sim_dev,
                 device="cuda"):
        torch = _torch()
        self.tau, self.alpha, self.beta, self.thr = tau, list(alpha), list(beta), list(thr)
        self.ws, self.gamma_dev, self.sim_dev = ws, gamma_dev, sim_dev
        self.d = [torch.empty(n_elems, dtype=dtype, device=device), torch.empty(n_elems, dtype=dtype, device=device)]
        self.state = TdcState()
        self.pending = False
        self.had_delta = False

    def decide(self) -> int:
        return self.state.decide(self.tau)

    def routes(self, outlier_ratio: float | None = None, rho: float = math.inf) -> list[int]:
        """Routes of this block's layers; with outlier_ratio (the block input's, from
        outlier_ratio()) above rho every layer runs BF16 (PDR)."""
        return self.state.routes(self.alpha, self.beta, self.thr, outlier_ratio, rho)

    def skip(self, x_in, x_out, stream=None):
        tdc_step(TDC_SKIP, x_in.reshape(-1), self.ws, x_out_skip=x_out.reshape(-1), d1=self.d[0], stream=stream)
        self.state.update(TDC_SKIP)

    def commit(self, x_in, x_out, stream=None):
        tdc_step(TDC_COMMIT, x_in.reshape(-1), self.ws, x_out=x_out.reshape(-1),
                 d1=self.d[0] if self.had_delta else None, d_new=self.d[1], gamma=self.gamma_dev,
                 sim=self.sim_dev, stream=stream)
        self.d.reverse()
        self.pending = True

    def absorb(self, gamma: float, sim: float) -> None:
        """Fold a committed step's Gamma and similarity (host values) into the state."""
        if not self.pending:
            return
        self.state.update(TDC_COMMIT, gamma, sim if self.had_delta else None)
        self.had_delta = True
        self.pending = False

    def state_dict(self) -> dict:
        """What resuming this block's delta cache needs: the decision state (host) and the
        cached delta of the last computed step (copied to the host).  A commit must have been
        absorbed first."""
        if self.pending:
            raise DitError("absorb the pending commit before saving the delta-cache state")
        return {"tdc": self.state.to_dict(), "had_delta": self.had_delta,
                "delta": self.d[0].detach().cpu() if self.had_delta else None,
                "tau": self.tau, "alpha": list(self.alpha), "beta": list(self.beta), "thr": list(self.thr)}

    def load_state_dict(self, sd: dict) -> None:
        if sd["delta"] is not None and sd["delta"].numel() != self.d[0].numel():
            raise DitError("delta-cache state of a different block size")
        self.state = TdcState.from_dict(sd["tdc"])
        self.had_delta = bool(sd["had_delta"])
        self.pending = False
        self.tau, self.alpha, self.beta, self.thr = sd["tau"], list(sd["alpha"]), list(sd["beta"]), list(sd["thr"])
        if sd["delta"] is not None:
            self.d[0].copy_(sd["delta"].to(self.d[0].dtype))
