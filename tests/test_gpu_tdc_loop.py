"""The full delta-cache / PDR loop at the CogVideoX-2B size against the oracle (GPU).

Four chained blocks (block b+1's input is block b's output) run fifty denoising steps at
17776 x 1920 bf16 with the seeded delta recurrence of the TDC workload (Delta_t =
Delta_{t-1} (1 + eps), eps ~ N(0, 0.01), N(0, 0.5) on jump steps).  The device side is what
the library's users run: the C decision state machine fed with the Gamma and similarity the
commit kernel returns, the skip kernel, and PDR routing.  The oracle runs its own chain on
the CPU from the same seeded deltas.  Every skip/compute decision and every compute step's
routes must be identical (a decision or route within 1e-5 relative of its threshold is
counted, not compared), and every step's output is bit-identical, so the two chains never
drift apart.
"""
import numpy as np
import pytest

import synth
from gpu_helpers import dev_bf16, host
from oracle import dmpq as D
from oracle import tdc as T

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import int8_mixed_precision_gb300 as dit  # noqa: E402

M, H, BLOCKS, STEPS, TAU = synth.TOKENS_2B, 1920, 4, 50, 0.05
ALPHA, BETA, THR = [1.0] * 4, [0.0] * 4, [0.05] * 4


@pytest.mark.timeout(1800)
def test_tdc_loop_four_chained_blocks_fifty_steps_full_size():
    ws = dit.workspace()
    gam = torch.zeros(BLOCKS, dtype=torch.float32, device="cuda")
    sim = torch.zeros(BLOCKS, dtype=torch.float32, device="cuda")
    blocks = [dit.DeltaCachedBlock(M * H, torch.bfloat16, TAU, ALPHA, BETA, THR, ws, gam[b:b + 1], sim[b:b + 1])
              for b in range(BLOCKS)]
    oracle = [T.BlockLoop(TAU, ALPHA, BETA, THR, "bf16") for _ in range(BLOCKS)]
    streams = [synth.tdc_delta_stream(STEPS, M, H, seed=900 + b) for b in range(BLOCKS)]
    x0 = synth.activations(M, H, seed=899)
    x0_dev = dev_bf16(x0).reshape(-1)
    bufs = [torch.empty_like(x0_dev), torch.empty_like(x0_dev)]
    decisions = {b: [] for b in range(BLOCKS)}
    borderline = 0
    for t in range(STEPS):
        x_dev, x_host = x0_dev, x0
        for b, blk in enumerate(blocks):
            delta, _ = next(streams[b])
            r = oracle[b].step(x_host, delta)
            x_next = bufs[1] if x_dev is bufs[0] else bufs[0]
            mode = blk.decide()
            got = "skip" if mode == dit.TDC_SKIP else "compute"
            if r["margin"] <= 1e-5:
                borderline += 1
            else:
                assert got == r["decision"], (t, b)
            if mode == dit.TDC_SKIP:
                blk.skip(x_dev, x_next)
            else:
                routes = blk.routes()
                if r["gamma"] is not None and D.route_margin(r["gamma"], ALPHA[0], BETA[0], THR[0]) <= 1e-5:
                    borderline += 1
                else:
                    assert routes == r["routes"], (t, b)
                x_next.copy_((x_dev.float() + dev_bf16(delta).reshape(-1).float()).to(torch.bfloat16))
                blk.commit(x_dev, x_next)
            decisions[b].append(got)
            out = host(x_next).reshape(M, H)
            assert np.array_equal(out, r["out"]), (t, b)
            x_dev, x_host = x_next, r["out"]
        h = torch.stack([gam, sim]).cpu()
        for b, blk in enumerate(blocks):
            blk.absorb(float(h[0, b]), float(h[1, b]))
    torch.cuda.synchronize()
    assert dit.device_status(ws) == 0
    assert borderline <= 2
    for b in range(BLOCKS):   # the workload exercises skips, forced recomputes and PDR refreshes
        assert decisions[b].count("skip") >= 5 and decisions[b].count("compute") >= 5, decisions[b]
