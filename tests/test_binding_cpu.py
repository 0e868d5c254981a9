"""The Python binding refuses, on the host and before any launch, buffers the kernels cannot
read safely: host tensors, buffers smaller than the call reads or writes, operands whose K
disagree, and a bias that is not float32."""
import os

import pytest
import torch

import int8_mixed_precision_gb300 as dit


@pytest.fixture(scope="module", autouse=True)
def library():
    from int8_mixed_precision_gb300 import _lib, build
    if not os.path.exists(_lib.library_path()):
        try:
            build.build_library()
        except RuntimeError as e:          # no nvcc on this machine
            pytest.skip(str(e))
    return _lib.lib()


def _ws():
    return torch.zeros(dit.workspace_bytes(), dtype=torch.uint8)


def test_host_tensors_are_refused():
    m, n, k = 8, 16, 64
    a = torch.zeros(m, k, dtype=torch.bfloat16)
    b = torch.zeros(n, k, dtype=torch.bfloat16)
    y = torch.empty(m, n, dtype=torch.bfloat16)
    with pytest.raises(dit.DitError, match="CUDA"):
        dit.qgemm_int8(a, torch.ones(m), b, torch.ones(n), y, _ws())
    x = torch.zeros(m, k, dtype=torch.bfloat16)
    with pytest.raises(dit.DitError, match="CUDA"):
        dit.hadamard_quant_int8(x, 64, torch.empty(m, k, dtype=torch.int8), torch.empty(m))


def test_undersized_outputs_are_refused():
    m, n, k = 8, 16, 64
    a = torch.zeros(m, k, dtype=torch.bfloat16)
    b = torch.zeros(n, k, dtype=torch.bfloat16)
    with pytest.raises(dit.DitError, match="y:"):
        dit.qgemm_int8(a, torch.ones(m), b, torch.ones(n), torch.empty(m, n - 1, dtype=torch.bfloat16), _ws())
    with pytest.raises(dit.DitError, match="a_scale"):
        dit.qgemm_int8(a, torch.ones(m - 1), b, torch.ones(n), torch.empty(m, n, dtype=torch.bfloat16), _ws())
    with pytest.raises(dit.DitError, match="acc_debug"):
        dit.qgemm_int8(a, torch.ones(m), b, torch.ones(n), torch.empty(m, n, dtype=torch.bfloat16), _ws(),
                       acc_debug=torch.empty(m * n - 1, dtype=torch.int32))
    x = torch.zeros(m, k, dtype=torch.bfloat16)
    with pytest.raises(dit.DitError, match="q:"):
        dit.hadamard_quant_int8(x, 64, torch.empty(m, k - 1, dtype=torch.int8), torch.empty(m))
    with pytest.raises(dit.DitError, match="row_scale"):
        dit.hadamard_quant_int8(x, 64, torch.empty(m, k, dtype=torch.int8), torch.empty(m - 1))
    q = dit.alloc_nvfp4(m, k, device="cpu")
    with pytest.raises(dit.DitError, match="sf"):
        dit.hadamard_quant_nvfp4(x, 64, q["codes"], q["sf"][:-1], q["gs"], _ws())
    with pytest.raises(dit.DitError, match="codes"):
        dit.hadamard_quant_nvfp4(x, 64, q["codes"][:-1], q["sf"], q["gs"], _ws())


def test_nvfp4_gemm_operands_are_checked():
    m, n, k = 8, 256, 128
    A, W = dit.alloc_nvfp4(m, k, device="cpu"), dit.alloc_nvfp4(n, k, device="cpu")
    y = torch.empty(m, n, dtype=torch.bfloat16)
    W2 = dit.alloc_nvfp4(n, 2 * k, device="cpu")
    with pytest.raises(dit.DitError, match="same k"):
        dit.qgemm_nvfp4(A["codes"], A["sf"], A["gs"], W2["codes"], W2["sf"], W2["gs"], y, _ws())
    with pytest.raises(dit.DitError, match="b_sf"):
        dit.qgemm_nvfp4(A["codes"], A["sf"], A["gs"], W["codes"], W["sf"][:-16], W["gs"], y, _ws())
    with pytest.raises(dit.DitError, match="bias must be float32"):
        dit.qgemm_nvfp4(A["codes"], A["sf"], A["gs"], W["codes"], W["sf"], W["gs"], y, _ws(),
                        bias=torch.zeros(n, dtype=torch.bfloat16))
    with pytest.raises(dit.DitError, match="bias"):
        dit.qgemm_nvfp4(A["codes"], A["sf"], A["gs"], W["codes"], W["sf"], W["gs"], y, _ws(),
                        bias=torch.zeros(n - 1))
    with pytest.raises(dit.DitError, match="tensor_scale_out"):
        dit.qgemm_nvfp4_amax(A["codes"], A["sf"], A["gs"], W["codes"], W["sf"], W["gs"], y, _ws(), 64,
                             torch.empty(0))


def test_delta_cache_buffers_must_match():
    x = torch.zeros(1024, dtype=torch.bfloat16)
    with pytest.raises(dit.DitError, match="d1"):
        dit.tdc_step(dit.TDC_SKIP, x, _ws(), x_out_skip=torch.empty_like(x), d1=torch.zeros(1023, dtype=torch.bfloat16))
    with pytest.raises(dit.DitError, match="x_out"):
        dit.tdc_step(dit.TDC_COMMIT, x, _ws(), x_out=torch.zeros(1024, dtype=torch.float32),
                     d_new=torch.empty_like(x), gamma=torch.empty(1), sim=torch.empty(1))
    with pytest.raises(dit.DitError, match="same dtype and size"):
        dit.gamma_route(x, torch.zeros(512, dtype=torch.bfloat16), [1.0], [0.0], [0.05], torch.empty(1),
                        torch.empty(1, dtype=torch.int32), _ws())
    with pytest.raises(dit.DitError, match="routes"):
        dit.gamma_route(x, x.clone(), [1.0] * 4, [0.0] * 4, [0.05] * 4, torch.empty(1),
                        torch.empty(3, dtype=torch.int32), _ws())
