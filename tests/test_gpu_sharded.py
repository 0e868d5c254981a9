"""The token-sharded form on the GPU: one block's rows split into two shards (GPU).

The partial kernels run on each shard in turn on one GPU; their partials are summed (or
maxed) with torch, which is what the all-reduce of a multi-GPU run computes, and the device
finishing call turns them into Gamma, the similarity, the routes and the tensor scale.  The
results must equal the unsharded library calls (and, through them, the oracle): the tensor
scale and every shard's codes bit for bit, the per-shard deltas bit for bit, Gamma and the
similarity as float32 values (their fp64 sums differ only in order).
"""
import numpy as np
import pytest

import synth
from gpu_helpers import dev_bf16, host
from oracle import dmpq as D
from oracle import formats as F
from oracle import tdc as T

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import int8_mixed_precision_gb300 as dit  # noqa: E402

M, K, HB = synth.TOKENS_2B, 1920, 64
CUT = 70 * 128            # shard boundary on a 128-row block boundary (scale tiles split cleanly)
ALPHA, BETA, THR = [1.0, 0.5, 2.0, 1.0], [0.0, 0.0, 0.0, 0.02], [0.05, 0.05, 0.05, 0.05]


@pytest.fixture(scope="module")
def ws():
    return dit.workspace()


@pytest.fixture(scope="module")
def pair():
    xi = synth.activations(M, K, seed=401)
    xo = synth.gamma_pair(xi, 0.043, seed=402)
    d1 = synth.to_bf16_bits(synth.from_bf16_bits(synth.gamma_pair(xi, 0.05, seed=403)) - synth.from_bf16_bits(xi))
    return xi, xo, d1


def test_sharded_gamma_routes_and_tdc_commit(pair, ws):
    xi, xo, d1 = pair
    Xi, Xo, D1 = (dev_bf16(a).reshape(M, K) for a in (xi, xo, d1))
    shards = [slice(0, CUT), slice(CUT, M)]
    # Gamma and routes
    tot = torch.zeros(2, dtype=torch.float64, device="cuda")
    for sl in shards:
        p = torch.empty(2, dtype=torch.float64, device="cuda")
        dit.l1_partials(dit.L1_GAMMA, Xi[sl], Xo[sl], p, ws)
        tot += p
    g, r = torch.empty(1, device="cuda"), torch.empty(4, dtype=torch.int32, device="cuda")
    dit.shard_finish(tot, None, ALPHA, BETA, THR, gamma=g, routes=r)
    g1, r1 = torch.empty(1, device="cuda"), torch.empty(4, dtype=torch.int32, device="cuda")
    dit.gamma_route(Xi, Xo, ALPHA, BETA, THR, g1, r1, ws)
    torch.cuda.synchronize()
    assert dit.device_status(ws) == 0
    g_ref = D.gamma_rel_l1(F.bf16_bits_to_f32(xi), F.bf16_bits_to_f32(xo))
    assert np.float32(g.item()) == np.float32(g1.item()) == np.float32(g_ref)
    assert r.tolist() == r1.tolist() == D.route_layers(g_ref, ALPHA, BETA, THR)
    # delta-cache commit: per-shard deltas, Gamma and similarity over the whole block
    tot4 = torch.zeros(4, dtype=torch.float64, device="cuda")
    dn = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    for sl in shards:
        p = torch.empty(4, dtype=torch.float64, device="cuda")
        dit.l1_partials(dit.L1_TDC_COMMIT, Xi[sl], Xo[sl], p, ws, d1=D1[sl], d_new=dn[sl])
        tot4 += p
    gs, ss = torch.empty(1, device="cuda"), torch.empty(1, device="cuda")
    dit.shard_finish(tot4, None, gamma=gs, sim=ss)
    dn1 = torch.empty_like(dn)
    gu, su = torch.empty(1, device="cuda"), torch.empty(1, device="cuda")
    dit.tdc_step(dit.TDC_COMMIT, Xi.reshape(-1), ws, x_out=Xo.reshape(-1), d1=D1.reshape(-1), d_new=dn1.reshape(-1),
                 gamma=gu, sim=su)
    torch.cuda.synchronize()
    assert dit.device_status(ws) == 0
    assert torch.equal(dn.view(torch.int16), dn1.view(torch.int16))
    ref = T.tdc_commit(xi, xo, d1, "bf16")
    assert np.array_equal(host(dn), ref["delta"])
    assert np.float32(gs.item()) == np.float32(gu.item()) == np.float32(ref["gamma"])
    assert np.float32(ss.item()) == np.float32(su.item()) == np.float32(ref["d"])
    # the first commit of a block (no previous delta): the similarity partials are zero
    p = torch.full((4,), 7.0, dtype=torch.float64, device="cuda")
    dit.l1_partials(dit.L1_TDC_COMMIT, Xi[:CUT], Xo[:CUT], p, ws, d_new=dn[:CUT])
    torch.cuda.synchronize()
    assert host(p)[2:].tolist() == [0.0, 0.0]


def test_sharded_tensor_scale_gives_the_unsharded_codes(pair, ws):
    xi, _, _ = pair
    X = dev_bf16(xi).reshape(M, K)
    amax = torch.zeros(1, device="cuda")
    for sl in (slice(0, CUT), slice(CUT, M)):
        a = torch.empty(1, device="cuda")
        dit.nvfp4_amax(X[sl], HB, a, ws)
        amax = torch.maximum(amax, a)
    sg = torch.empty(1, device="cuda")
    dit.shard_finish(None, amax, tensor_scale=sg)
    whole = dit.alloc_nvfp4(M, K)
    dit.hadamard_quant_nvfp4(X, HB, whole["codes"], whole["sf"], whole["gs"], ws)
    torch.cuda.synchronize()
    assert sg.view(torch.int32).item() == whole["gs"].view(torch.int32).item()
    want = D.nvfp4_tensor_scale(D.block_fwht_f32(F.bf16_bits_to_f32(xi), HB))
    assert np.float32(sg.item()).view(np.uint32) == np.float32(want).view(np.uint32)
    # each shard quantised with the finished scale: the unsharded codes and block scales
    sf_split = F.sf_padded_shape(CUT, K)[0] * F.sf_padded_shape(CUT, K)[1]
    for sl in (slice(0, CUT), slice(CUT, M)):
        rows = sl.stop - sl.start
        part = dit.alloc_nvfp4(rows, K)
        dit.hadamard_quant_nvfp4(X[sl], HB, part["codes"], part["sf"], part["gs"], ws, tensor_scale_in=sg)
        torch.cuda.synchronize()
        assert torch.equal(part["codes"], whole["codes"][sl])
        ref_sf = whole["sf"][:sf_split] if sl.start == 0 else whole["sf"][sf_split:]
        assert torch.equal(part["sf"], ref_sf)
    assert dit.device_status(ws) == 0
