"""Seeded synthetic inputs shaped like the CogVideoX-class workloads of 6Bit-Diffusion.

Shared by the tests, the benchmark and the oracle runs.  This module only DRAWS inputs
(numpy PCG64, seeded): it holds none of the method's arithmetic -- no Hadamard, no scale,
no rounding rule of the quantisers, no delta-cache logic.  Activations are delivered as
bf16 bit patterns (uint16) or float32, so every consumer sees bit-identical inputs.

Workloads (the pages evaluate on CogVideoX-2B/5B videos; those models and videos are not
available, these tensors stand in for them):

* ``single_linear``       X fp32 [256 x 128] ~ N(0,1), channels {5,38,71,104} x30;
                          W [512 x 128] ~ N(0,0.02); X_out = X_in + N(0, 0.1).
* ``cogvideox_2b_block``  hidden 1920, 17776 tokens (13x30x45 video + 226 text), bf16,
                          N(0,1) with 1% outlier channels x50; QKV 1920->5760, out
                          1920->1920, FFN 1920->7680->1920.
* ``cogvideox_5b_block``  hidden 3072, Laplace(0,1), 0.5% outlier channels x100.
* ``long_1080p``          hidden 3072, 104746 tokens (13x67x120 + 226), FFN 3072<->12288.
* ``tdc_deltas``          per-block delta recurrence with occasional jumps.
"""
from __future__ import annotations

import numpy as np

TOKENS_2B = 13 * 30 * 45 + 226        # 17776
TOKENS_1080P = 13 * 67 * 120 + 226    # 104746


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Store float32 samples as bf16 (round to nearest even) -- input encoding only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def outlier_channels(k: int, frac: float, seed: int) -> np.ndarray:
    """A fixed seeded subset of floor(frac * k) input channels (at least one)."""
    n = max(1, int(np.floor(frac * k)))
    return np.sort(rng(seed).choice(k, size=n, replace=False))


def activations(rows: int, k: int, *, dist: str = "normal", outlier_frac: float = 0.01,
                outlier_mult: float = 50.0, seed: int = 0, channels=None,
                dtype: str = "bf16") -> np.ndarray:
    """Activation tensor [rows x k] with fixed outlier channels scaled by outlier_mult."""
    g = rng(seed)
    if dist == "normal":
        x = g.standard_normal((rows, k), dtype=np.float32)
    elif dist == "laplace":
        x = g.laplace(0.0, 1.0, size=(rows, k)).astype(np.float32)
    else:
        raise ValueError(dist)
    if channels is None:
        channels = outlier_channels(k, outlier_frac, seed + 7919)
    x[:, channels] *= np.float32(outlier_mult)
    return to_bf16_bits(x) if dtype == "bf16" else x


def weights(n: int, k: int, *, seed: int, std: float = 0.02) -> np.ndarray:
    """Dense weight [n x k] ~ N(0, std), float32."""
    return (rng(seed).standard_normal((n, k), dtype=np.float32) * np.float32(std)).astype(np.float32)


def single_linear(seed: int = 0) -> dict:
    """The 256-token, 128-channel single linear (Hadamard block 16, fp32)."""
    g = rng(seed)
    x = g.standard_normal((256, 128), dtype=np.float32)
    x[:, [5, 38, 71, 104]] *= np.float32(30.0)
    w = (g.standard_normal((512, 128), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    x_out = (x + g.standard_normal((256, 128), dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    return {"x": x, "w": w, "x_out": x_out, "hblock": 16, "alpha": 1.0, "beta": 0.0, "thr": 0.05}


BLOCK_SHAPES = {
    # name: (hidden, ffn, dist, outlier_frac, outlier_mult, hblock)
    "cogvideox_2b": (1920, 7680, "normal", 0.01, 50.0, 64),
    "cogvideox_5b": (3072, 12288, "laplace", 0.005, 100.0, 64),
}


def block_linears(name: str, tokens: int = TOKENS_2B) -> list[tuple[str, int, int]]:
    """(layer, K, N) of the four routed linears of one DiT block."""
    h, f = BLOCK_SHAPES[name][:2]
    return [("qkv", h, 3 * h), ("out", h, h), ("ffn_up", h, f), ("ffn_down", f, h)]


def gamma_pair(x_in_bits: np.ndarray, gamma_target: float, seed: int) -> np.ndarray:
    """X_out = X_in + gamma * S * X_in with random signs S (bf16 in, bf16 out); the relative
    L1 distance of the pair is gamma up to bf16 rounding."""
    xi = from_bf16_bits(x_in_bits)
    s = rng(seed).integers(0, 2, size=xi.shape, dtype=np.int8).astype(np.float32) * 2 - 1
    return to_bf16_bits(xi + np.float32(gamma_target) * s * xi)


def tdc_delta_stream(steps: int, rows: int, k: int, *, seed: int, jump_every: float = 8.0,
                     eps_std: float = 0.01, jump_std: float = 0.5):
    """Per-step true deltas of one block, one step at a time: Delta_0 ~ N(0, sigma), sigma ~
    U(0.02, 0.15); Delta_t = Delta_{t-1} * (1 + eps), eps ~ N(0, 0.01) elementwise, and
    N(0, 0.5) on jump steps (Bernoulli(1/jump_every)).  Yields (bf16 bits, jump) pairs."""
    g = rng(seed)
    sigma = g.uniform(0.02, 0.15)
    d = (g.standard_normal((rows, k), dtype=np.float32) * np.float32(sigma)).astype(np.float32)
    yield to_bf16_bits(d), False
    for _ in range(1, steps):
        jump = bool(g.random() < 1.0 / jump_every)
        std = jump_std if jump else eps_std
        eps = g.standard_normal((rows, k), dtype=np.float32) * np.float32(std)
        d = (d * (np.float32(1.0) + eps)).astype(np.float32)
        yield to_bf16_bits(d), jump


def tdc_deltas(steps: int, rows: int, k: int, *, seed: int, jump_every: float = 8.0,
               eps_std: float = 0.01, jump_std: float = 0.5) -> tuple[list[np.ndarray], list[bool]]:
    """All steps of tdc_delta_stream at once: (list of bf16 bits, list of jump flags)."""
    pairs = list(tdc_delta_stream(steps, rows, k, seed=seed, jump_every=jump_every, eps_std=eps_std,
                                  jump_std=jump_std))
    return [p[0] for p in pairs], [p[1] for p in pairs]
