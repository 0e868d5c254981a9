"""One DiT block's tokens split across GPUs (one rank per GPU, torch.distributed).

The path partitions by tokens: quantisation (once the tensor scale is known), the GEMMs
against replicated weights and the delta-cache skip act on a rank's rows alone.  Three
quantities span every token of the block and need one exchange each:

* Gamma (gist.science EN 2.A Mechanism 1): sum|X_out - X_in| / sum|X_in| -- all-reduce SUM
  of two fp64 partials;
* the delta similarity of the delta cache (EN 2.B): sum|Delta - Delta_prev| / sum|Delta_prev|,
  committed together with Gamma -- all-reduce SUM of four fp64 partials;
* the NVFP4 tensor scale (one fp32 scale per tensor): amax / (6 * 448) -- all-reduce MAX of
  one fp32 amax.  The maximum is exact, so every rank's codes equal the one-GPU codes.

Each function enqueues the library's partial kernel on the current stream, all-reduces the
partials with the given process group (NCCL on GPUs), and finishes on the device.  No data
tensor crosses ranks and nothing here uses multicast memory.
"""
from __future__ import annotations

from . import L1_GAMMA, L1_TDC_COMMIT, l1_partials, nvfp4_amax, shard_finish


def _all_reduce(t, op, group):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(t, op=op, group=group)


def gamma_route(x_in, x_out, alpha, beta, thr, gamma, routes, ws, partials, group=None):
    """Gamma of the whole block and the per-layer routes; partials: device float64 [2] scratch."""
    import torch.distributed as dist
    l1_partials(L1_GAMMA, x_in, x_out, partials, ws)
    _all_reduce(partials[:2], dist.ReduceOp.SUM, group)
    shard_finish(partials[:2], None, alpha, beta, thr, gamma=gamma, routes=routes)


def tdc_commit(x_in, x_out, d1, d_new, gamma, sim, ws, partials, group=None):
    """Delta-cache commit of this rank's rows (d_new = x_out - x_in) with Gamma and the delta
    similarity over the whole block; partials: device float64 [4] scratch."""
    import torch.distributed as dist
    l1_partials(L1_TDC_COMMIT, x_in, x_out, partials, ws, d1=d1, d_new=d_new)
    _all_reduce(partials[:4], dist.ReduceOp.SUM, group)
    shard_finish(partials[:4], None, gamma=gamma, sim=sim if d1 is not None else None)


def tensor_scale(x, hblock, scale, ws, amax, group=None):
    """The NVFP4 tensor scale of the whole block input from this rank's rows; amax: device
    float32 [1] scratch.  Pass scale as tensor_scale_in to hadamard_quant_nvfp4."""
    import torch.distributed as dist
    nvfp4_amax(x, hblock, amax, ws)
    _all_reduce(amax, dist.ReduceOp.MAX, group)
    shard_finish(None, amax, tensor_scale=scale)
