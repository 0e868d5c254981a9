"""The workspace-free Gamma/route entry point against the regular one (GPU).

dit_gamma_route_noalloc serves callers that cannot allocate device memory (for example an
inference-engine plugin whose memory is planned by the engine before it runs); its scratch
is a fixed array inside the library that every call reuses.  Two calls in a row, on
different inputs, must each give the same Gamma and routes as dit_gamma_route with a caller
workspace -- so nothing left over from the previous call may leak into the next one; a third,
smaller call checks the same when the grid shrinks.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import int8_mixed_precision_gb300 as dit  # noqa: E402

ALPHA, BETA, THR = [1.0, 0.5, 2.0, 1.0], [0.0, 0.0, 0.0, 0.02], [0.05, 0.05, 0.05, 0.05]


def _pair(n, gam, seed, dtype):
    g = synth.rng(seed)
    xi = g.standard_normal(n).astype(np.float32)
    s = np.where(g.random(n) < 0.5, -1.0, 1.0).astype(np.float32)
    xo = (xi + np.float32(gam) * s * xi).astype(np.float32)
    if dtype == "bf16":
        to = lambda a: torch.from_numpy(synth.to_bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()
    else:
        to = lambda a: torch.from_numpy(a).cuda()
    return to(xi), to(xo)


@pytest.mark.parametrize("dtype,n", [("bf16", 17776 * 1920), ("f32", 256 * 128 + 7)])
def test_noalloc_matches_workspace_entry_point_two_calls(dtype, n):
    """Both entry points run the same kernel with the same grid and the same fixed-order
    reduction, so Gamma must agree bit for bit.  The third call is much smaller (a few CTAs
    instead of hundreds): partial sums left in the array by the larger calls must not reach it."""
    ws = dit.workspace()
    cases = [(n, 0.12, 1), (n, 0.03, 2), (4096 * 10 + 3, 0.07, 3)]
    for call, (size, gam, seed) in enumerate(cases):
        xi, xo = _pair(size, gam, seed, dtype)
        g_ref = torch.empty(1, dtype=torch.float32, device="cuda")
        r_ref = torch.empty(4, dtype=torch.int32, device="cuda")
        dit.gamma_route(xi, xo, ALPHA, BETA, THR, g_ref, r_ref, ws)
        g_na = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
        r_na = torch.full((4,), -1, dtype=torch.int32, device="cuda")
        dit.gamma_route_noalloc(xi, xo, ALPHA, BETA, THR, g_na, r_na)
        torch.cuda.synchronize()
        assert g_na.view(torch.int32).item() == g_ref.view(torch.int32).item(), call
        assert g_na.item() == pytest.approx(gam, rel=1e-2), call
        assert r_na.tolist() == r_ref.tolist(), call
