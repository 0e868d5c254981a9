"""The token-sharded form on CPU: two gloo ranks split one block's tokens (no GPU).

Each rank holds a ragged half of the rows.  It forms its shard's partials (the L1 sums of
Gamma and of the delta similarity, and the amax of the block-Hadamard-transformed input, all
written out from their definitions in float64 / float32), the ranks all-reduce them (sum and
max) with gloo, and the library's finishing arithmetic (dit_shard_finish_host, the host twin
of the device call) turns them into Gamma, the similarity, the routes and the NVFP4 tensor
scale.  Rank 0 checks them against the oracle run on the whole, unsharded tensors:

* the tensor scale is the same float32 bit for bit (the maximum is exact), so every shard's
  NVFP4 codes and block scales equal the one-GPU encoding row for row;
* Gamma and the similarity, float32 roundings of fp64 ratios whose sums differ from the
  oracle's only in their order, are the oracle's float32 values; the routes and the
  delta-cache decisions of a ten-step sequence (skips, a PDR recompute) are the same.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

ROWS, K, HB, STEPS = 301, 256, 64, 10
ALPHA, BETA, THR, TAU = [1.0, 0.5, 2.0, 1.0], [0.0, 0.0, 0.0, 0.02], [0.05, 0.05, 0.05, 0.05], 0.02


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs():
    """Block input and a delta sequence (bf16 bits), seeded: the same on every rank."""
    import synth
    x = synth.activations(ROWS, K, seed=11)
    deltas, _ = synth.tdc_deltas(STEPS, ROWS, K, seed=12, jump_every=3.0)
    return x, deltas


def _shard(r, world):
    bounds = [0, 150, ROWS][: world + 1] if world == 2 else np.linspace(0, ROWS, world + 1).astype(int)
    return slice(int(bounds[r]), int(bounds[r + 1]))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import int8_mixed_precision_gb300 as dit
    from oracle import dmpq as D
    from oracle import formats as F
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sl = _shard(rank, world)
        x_bits, deltas = _inputs()
        f32 = F.bf16_bits_to_f32
        out = {"steps": []}
        # the NVFP4 tensor scale of the block input from this shard's rows
        amax = torch.tensor([float(np.max(np.abs(D.block_fwht_f32(f32(x_bits[sl]), HB))))], dtype=torch.float32)
        dist.all_reduce(amax, op=dist.ReduceOp.MAX)
        out["tensor_scale"] = dit.shard_finish_host(amax=float(amax.item()))["tensor_scale"]
        # a delta-cache run: every compute step commits with sharded Gamma / similarity
        st = dit.TdcState()
        d_prev = None
        for t in range(STEPS):
            mode = st.decide(TAU)
            if mode == dit.TDC_SKIP:
                st.update(dit.TDC_SKIP)
                out["steps"].append(("skip", None, None, None))
                continue
            routes_in = st.routes(ALPHA, BETA, THR)
            xi = f32(x_bits[sl])
            xo = F.bf16_bits_to_f32(F.f32_to_bf16_bits((xi + f32(deltas[t][sl])).astype(np.float32)))
            diff = (xo - xi).astype(np.float32)
            d_new = f32(F.f32_to_bf16_bits(diff))
            p = torch.zeros(4, dtype=torch.float64)
            p[0] = float(np.sum(np.abs(diff.astype(np.float64))))
            p[1] = float(np.sum(np.abs(xi.astype(np.float64))))
            if d_prev is not None:
                p[2] = float(np.sum(np.abs(d_new.astype(np.float64) - d_prev.astype(np.float64))))
                p[3] = float(np.sum(np.abs(d_prev.astype(np.float64))))
            dist.all_reduce(p, op=dist.ReduceOp.SUM)
            fin = dit.shard_finish_host(p.tolist() if d_prev is not None else p[:2].tolist(), None, ALPHA, BETA, THR)
            st.update(dit.TDC_COMMIT, fin["gamma"], fin.get("sim"))
            out["steps"].append(("compute", routes_in, fin["gamma"], fin.get("sim"), fin["routes"]))
            d_prev = d_new
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def library():
    from int8_mixed_precision_gb300 import _lib, build
    if not os.path.exists(_lib.library_path()):
        try:
            build.build_library()
        except RuntimeError as e:          # no nvcc on this machine
            pytest.skip(str(e))
    return _lib.lib()


@pytest.mark.timeout(600)
def test_two_rank_token_shards_match_the_unsharded_oracle(library):
    from oracle import dmpq as D
    from oracle import formats as F
    from oracle import tdc as T
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=540) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    x_bits, deltas = _inputs()
    f32 = F.bf16_bits_to_f32

    # the tensor scale: one float32, bit for bit on both ranks
    y = D.block_fwht_f32(f32(x_bits), HB)
    want = D.nvfp4_tensor_scale(y)
    for r in range(world):
        assert np.float32(res[r]["tensor_scale"]).view(np.uint32) == np.float32(want).view(np.uint32)
    # hence every shard's encoding equals the unsharded one, row for row
    whole = D.quant_nvfp4(y)
    for r in range(world):
        part = D.quant_nvfp4(y[_shard(r, world)], s_g=np.float32(res[r]["tensor_scale"]))
        assert np.array_equal(part["codes"], whole["codes"][_shard(r, world)])
        assert np.array_equal(part["sf"], whole["sf"][_shard(r, world)])

    # the delta-cache run: decisions, routes, Gamma and similarity against the oracle loop
    ref = T.run_block_loop([x_bits] * STEPS, deltas, TAU, ALPHA, BETA, THR, "bf16")
    assert res[0]["steps"] == res[1]["steps"]
    got = res[0]["steps"]
    assert [s[0] for s in got] == ref["decisions"]
    assert "skip" in ref["decisions"] and ref["decisions"].count("compute") >= 5
    assert any(r == [D.ROUTE_INT8] * 4 for t, r in enumerate(ref["routes"]) if t >= 2 and r)   # a PDR recompute
    d1 = None
    for t, s in enumerate(got):
        if s[0] == "skip":
            continue
        assert s[1] == ref["routes"][t]
        c = T.tdc_commit(x_bits, ref["outs"][t], d1, "bf16")
        assert np.float32(s[2]) == np.float32(c["gamma"])
        assert s[4] == D.route_layers(c["gamma"], ALPHA, BETA, THR)
        if d1 is not None:
            assert np.float32(s[3]) == np.float32(c["d"])
        d1 = c["delta"]
