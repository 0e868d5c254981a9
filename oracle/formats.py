"""Number formats used by the routed quantised linear layer (oracle; test infrastructure only).

* E2M1 -- the 4-bit element format of NVFP4 ("NVFP4 (E2M1)", gist.science/it,
  "3. Contributi Chiave" item 4; gist.science EN "1. Problem Statement", Hardware Gap).
  1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no infinities or NaN.
* E4M3 (the "fn" variant) -- the per-16-element block scale of NVFP4.  1 sign bit, 4
  exponent bits (bias 7), 3 mantissa bits, no infinities, S.1111.111 is NaN, max 448.
* bf16 -- the activation storage type of the CogVideoX-shaped workloads.
* the block-scale tile layout consumed by the block-scaled tensor-core MMA.

Everything is computed from the format definitions in float64 / integers; nothing here
calls a conversion routine of a library (the tests pin these tables against torch).
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------------------
# E2M1
# ----------------------------------------------------------------------------------------


def e2m1_decode_table() -> np.ndarray:
    """Value of each of the 16 E2M1 codes, from the format definition.

    code = s<<3 | e<<1 | m ; e == 0 -> subnormal m * 2^-1 ; else (1 + m/2) * 2^(e-1).
    """
    out = np.zeros(16, dtype=np.float64)
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = m * 0.5 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
        out[code] = -mag if s else mag
    return out


E2M1_VALUES = e2m1_decode_table()
E2M1_MAGNITUDES = E2M1_VALUES[:8]          # codes 0..7: 0, .5, 1, 1.5, 2, 3, 4, 6
E2M1_MAX = 6.0


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even onto the E2M1 grid, saturating at +-6 (the "satfinite" rule).

    Ties go to the code whose mantissa bit is 0 (the even code).  The sign bit is the sign
    of the input, so a negative value that rounds to zero gives code 0x8 (-0): this is the
    sign-magnitude reading of IEEE round-to-nearest for a format that has a signed zero.
    ``v`` is float32 (the precision the quantiser computes in); comparisons are exact in
    float64.
    """
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v).astype(np.float64)
    mags = E2M1_MAGNITUDES
    code = np.zeros(a.shape, dtype=np.uint8)
    # walk the 7 midpoints; each comparison decides one step up the grid
    for i in range(7):
        mid = 0.5 * (mags[i] + mags[i + 1])
        up = a > mid
        tie = a == mid
        # on a tie pick the even code of (i, i+1)
        even_up = (i + 1) % 2 == 0
        step = up | (tie & even_up)
        code = np.where(step & (code == i), np.uint8(i + 1), code)
    sign = np.signbit(v).astype(np.uint8)
    return (code | (sign << 3)).astype(np.uint8)


def e2m1_rounding_margin(v: np.ndarray) -> np.ndarray:
    """Relative distance of |v| to the nearest E2M1 rounding midpoint (float64).

    Used to exempt elements whose pre-rounding value lies within 1e-5 relative of a
    rounding boundary from the bit-exact code comparison.
    """
    a = np.abs(np.asarray(v, dtype=np.float32).astype(np.float64))
    mids = 0.5 * (E2M1_MAGNITUDES[:-1] + E2M1_MAGNITUDES[1:])
    d = np.min(np.abs(a[..., None] - mids) / mids, axis=-1)
    return d


# ----------------------------------------------------------------------------------------
# E4M3 (fn)
# ----------------------------------------------------------------------------------------


def e4m3_decode_table() -> np.ndarray:
    """Value of each of the 256 E4M3 codes (NaN for S.1111.111), from the format definition."""
    out = np.zeros(256, dtype=np.float64)
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            out[code] = np.nan
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        out[code] = -mag if s else mag
    return out


E4M3_VALUES = e4m3_decode_table()
E4M3_MAX = 448.0
_E4M3_POS = E4M3_VALUES[:127]              # codes 0x00..0x7e, increasing, 0 .. 448


def e4m3_encode_nonneg(v: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even of a non-negative float32 onto E4M3, saturating at 448.

    Subnormals are kept (smallest positive value 2^-9).  Ties go to the even code.
    """
    a = np.asarray(v, dtype=np.float32).astype(np.float64)
    if np.any(a < 0) or np.any(np.isnan(a)):
        raise ValueError("block scales are non-negative and finite")
    grid = _E4M3_POS
    mids = 0.5 * (grid[:-1] + grid[1:])
    # index of the first midpoint >= a  == number of midpoints strictly below a
    idx = np.searchsorted(mids, a, side="left")          # a <= mids[idx]
    idx = np.minimum(idx, len(grid) - 1)
    # a exactly on a midpoint: idx points at the lower neighbour (mids[idx] == a)
    on_mid = (idx < len(mids)) & (a == mids[np.minimum(idx, len(mids) - 1)])
    lower = idx
    upper = idx + 1
    pick_upper = on_mid & (upper % 2 == 0)
    code = np.where(pick_upper, upper, lower)
    code = np.where(a >= E4M3_MAX, 126, code)
    return code.astype(np.uint8)


def e4m3_rounding_margin(v: np.ndarray) -> np.ndarray:
    """Relative distance of v (>= 0) to the nearest E4M3 rounding midpoint."""
    a = np.asarray(v, dtype=np.float32).astype(np.float64)
    grid = _E4M3_POS
    mids = 0.5 * (grid[:-1] + grid[1:])
    idx = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    d = np.minimum(np.abs(a - mids[idx]) / mids[idx], np.abs(a - mids[idx - 1]) / mids[idx - 1])
    return d


# ----------------------------------------------------------------------------------------
# bf16
# ----------------------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest even (finite inputs).

    Adding 0x7FFF plus the lowest kept bit to the float32 pattern and dropping the low 16
    bits rounds half to even.  For finite inputs the sum stays below 2^32 (the largest finite
    pattern is 0xFF7FFFFF), so the arithmetic is exact in uint32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u >> np.uint32(16)) & np.uint32(1)
    r += u
    r += np.uint32(0x7FFF)
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> float32 (exact)."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


# ----------------------------------------------------------------------------------------
# block-scale tile layout (128 rows x 4 scale columns per 512-byte atom)
# ----------------------------------------------------------------------------------------


def sf_padded_shape(rows: int, k: int) -> tuple[int, int]:
    """(padded rows, padded scale columns) of a [rows x k] NVFP4 tensor's scale array."""
    kb = k // 16
    return ((rows + 127) // 128) * 128, ((kb + 3) // 4) * 4


def sf_tiled_offset(r: np.ndarray, c: np.ndarray, rows: int, k: int) -> np.ndarray:
    """Byte offset of the scale of (row r, 16-element block c) in the tiled layout.

    The array is cut into atoms of 128 rows x 4 scale columns (512 bytes), atoms ordered
    with the scale-column atom index fastest.  Inside an atom, row ri and column ci sit at
    (ri % 32) * 16 + (ri // 32) * 4 + ci: one 16-byte line holds rows ri, ri+32, ri+64,
    ri+96.  This is the operand layout the block-scaled tensor-core MMA reads its
    per-16-element scales in.
    """
    _, cpad = sf_padded_shape(rows, k)
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    atom = (r // 128) * (cpad // 4) + (c // 4)
    ri = r % 128
    return atom * 512 + (ri % 32) * 16 + (ri // 32) * 4 + (c % 4)


def sf_to_tiled(sf: np.ndarray, rows: int, k: int) -> np.ndarray:
    """Scatter a plain [rows x k/16] scale array into the zero-padded tiled layout."""
    rp, cp = sf_padded_shape(rows, k)
    out = np.zeros(rp * cp, dtype=np.uint8)
    rr, cc = np.meshgrid(np.arange(rows), np.arange(k // 16), indexing="ij")
    out[sf_tiled_offset(rr, cc, rows, k)] = sf
    return out


def sf_from_tiled(buf: np.ndarray, rows: int, k: int) -> np.ndarray:
    """Gather a plain [rows x k/16] scale array out of the tiled layout."""
    rr, cc = np.meshgrid(np.arange(rows), np.arange(k // 16), indexing="ij")
    return np.asarray(buf, dtype=np.uint8)[sf_tiled_offset(rr, cc, rows, k)]
