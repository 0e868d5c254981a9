"""Helpers shared by the GPU parity tests: host<->device moves of seeded inputs and the
comparison rules (bit-exact codes except elements on a rounding boundary)."""
import numpy as np

import synth
from oracle import dmpq as D
from oracle import formats as F

BOUNDARY_REL = 1e-5


def dev_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_f32(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def host(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def as_f32(x, dtype):
    return F.bf16_bits_to_f32(x) if dtype == "bf16" else np.asarray(x, np.float32)


def make_x(rows, k, dtype, seed, dist="normal", mult=50.0):
    x = synth.activations(rows, k, dist=dist, outlier_frac=0.01, outlier_mult=mult, seed=seed, dtype=dtype)
    return x, (dev_bf16(x) if dtype == "bf16" else dev_f32(x))


def check_int8(q_gpu, s_gpu, x_host, dtype, hb):
    """Bit-exact q and scale except elements whose oracle value is on a .5 boundary."""
    y = D.block_fwht_f32(as_f32(x_host, dtype), hb)
    r = D.quant_int8_rows(y)
    assert np.array_equal(s_gpu.view(np.uint32), r["scale"].view(np.uint32)), "row scales differ"
    diff = q_gpu != r["q"]
    exempt = D.int8_rounding_margin(r["v"]) <= BOUNDARY_REL
    bad = diff & ~exempt
    assert not bad.any(), f"{bad.sum()} int8 codes differ (first at {np.argwhere(bad)[:3].tolist()})"
    return int((diff & exempt).sum()), int(exempt.sum())


def check_nvfp4(codes_gpu, sf_gpu, sg_gpu, x_host, dtype, hb, rows, k, s_g=None):
    """Bit-exact codes, scales and tensor scale, except boundary elements / blocks."""
    y = D.block_fwht_f32(as_f32(x_host, dtype), hb)
    r = D.quant_nvfp4(y, s_g=s_g)
    assert np.float32(sg_gpu).view(np.uint32) == np.float32(r["s_g"]).view(np.uint32), \
        f"tensor scale {sg_gpu} vs {r['s_g']}"
    sf_plain = F.sf_from_tiled(sf_gpu, rows, k)
    blk_exempt = F.e4m3_rounding_margin(r["sbf"]) <= BOUNDARY_REL
    sf_bad = (sf_plain != r["sf"]) & ~blk_exempt
    assert not sf_bad.any(), f"{sf_bad.sum()} block scales differ (first {np.argwhere(sf_bad)[:3].tolist()})"
    codes = D.unpack_e2m1(codes_gpu)
    el_exempt = (F.e2m1_rounding_margin(r["v"]) <= BOUNDARY_REL) | blk_exempt.repeat(16, axis=1)
    diff = codes != r["codes"]
    bad = diff & ~el_exempt
    assert not bad.any(), (f"{bad.sum()} E2M1 codes differ (first {np.argwhere(bad)[:3].tolist()}: "
                           f"gpu {codes[tuple(np.argwhere(bad)[0])]} oracle {r['codes'][tuple(np.argwhere(bad)[0])]} "
                           f"v {r['v'][tuple(np.argwhere(bad)[0])]})")
    # rows padded up to 128 carry zero scales
    rp, cp = F.sf_padded_shape(rows, k)
    if rp > rows:
        rr, cc = np.meshgrid(np.arange(rows, rp), np.arange(cp), indexing="ij")
        assert not sf_gpu[F.sf_tiled_offset(rr, cc, rows, k)].any()
    return r, int((diff & el_exempt).sum())


def rel_fro(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))
