"""ctypes loader of the in-tree libdit6.so with the signatures of include/dit6.h."""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_LOCK = threading.Lock()
_LIB = None


class LibraryMissing(RuntimeError):
    pass


def library_path() -> str:
    return os.path.join(_HERE, "libdit6.so")


_vp, _i64, _i32, _f, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.POINTER(ctypes.c_float), ctypes.c_size_t

SIGNATURES = {
    "dit_status_str": (ctypes.c_char_p, [_i32]),
    "dit_version": (ctypes.c_char_p, []),
    "dit_workspace_bytes": (_sz, []),
    "dit_ws_status_offset": (_sz, []),
    "dit_gamma_route": (_i32, [_vp, _vp, _i32, _i64, _f, _f, _f, _i32, _vp, _vp, _vp, _sz, _vp]),
    "dit_gamma_route_noalloc": (_i32, [_vp, _vp, _i32, _i64, _f, _f, _f, _i32, _vp, _vp, _vp]),
    "dit_hadamard_quant_nvfp4": (_i32, [_vp, _i32, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dit_hadamard_quant_int8": (_i32, [_vp, _i32, _i64, _i64, _i32, _vp, _i32, _vp, _vp]),
    "dit_qgemm_nvfp4": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _i32, _vp, _i32, _vp, _sz,
                                _vp]),
    "dit_qgemm_nvfp4_amax": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _i32, _vp, _i32, _vp, _vp,
                                     _sz, _vp]),
    "dit_nvfp4_to_int8": (_i32, [_vp, _vp, _vp, _i64, _i64, _vp, _i32, _vp, _vp]),
    "dit_qgemm_int8": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i64, _i64, _vp, _i32, _vp, _i32, _vp, _vp, _sz,
                               _vp]),
    "dit_qgemm_int8_requant": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _i32, _vp, _vp, _vp, _vp, _sz,
                                       _vp]),
    "dit_tdc_step": (_i32, [_i32, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _vp, _vp, _vp, _sz, _vp]),
    "dit_tdc_state_init": (None, [_vp]),
    "dit_tdc_decide": (_i32, [_vp, ctypes.c_double]),
    "dit_tdc_update": (None, [_vp, _i32, ctypes.c_double, ctypes.c_double, _i32]),
    "dit_route_host": (None, [_vp, _f, _f, _f, _i32, ctypes.POINTER(ctypes.c_int32)]),
    "dit_route_host_pdr": (None, [_vp, _f, _f, _f, _i32, ctypes.c_double, ctypes.c_double,
                                  ctypes.POINTER(ctypes.c_int32)]),
    "dit_outlier_ratio": (_i32, [_vp, _i32, _i64, ctypes.c_float, _vp, _vp, _vp, _sz, _vp]),
    "dit_gemm_bf16": (_i32, [_vp, _vp, _i64, _i64, _i64, _vp, _i32, _vp, _i32, _vp, _sz, _vp]),
    "dit_l1_partials": (_i32, [_i32, _vp, _vp, _vp, _vp, _i32, _i64, _vp, _vp, _sz, _vp]),
    "dit_nvfp4_amax": (_i32, [_vp, _i32, _i64, _i64, _i32, _vp, _vp, _sz, _vp]),
    "dit_shard_finish": (_i32, [_vp, _i32, _vp, _f, _f, _f, _i32, _vp, _vp, _vp, _vp, _vp]),
    "dit_shard_finish_host": (_i32, [ctypes.POINTER(ctypes.c_double), _i32, _f, _f, _f, _f, _i32, _f, _f,
                                     ctypes.POINTER(ctypes.c_int32), _f]),
    "dit_sf_index": (_i64, [_i64, _i64, _i64, _i64]),
    "dit_sf_bytes": (_sz, [_i64, _i64]),
}


def lib() -> ctypes.CDLL:
    """The loaded library; raises LibraryMissing (never falls back) when it is not built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    with _LOCK:
        if _LIB is None:
            path = library_path()
            if not os.path.exists(path):
                raise LibraryMissing(
                    f"{path} is not built: run `python -m int8_mixed_precision_gb300.build` "
                    "(nvcc, sm_103a) -- there is no CPU fallback")
            h = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _LIB = h
    return _LIB
