"""Test-side helpers written independently of the oracle and of the CUDA library.

They restate the number formats from their definitions (OCP E2M1 / E8M0 bit layouts,
IEEE-style bf16) with numpy, so that the oracle can be checked against something other
than itself.
"""
import numpy as np


def e2m1_value_from_bits(code: int) -> float:
    """E2M1 by its bit fields: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0."""
    s = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        return s * 0.5 * m  # subnormal: 0 or 0.5
    return s * (2.0 ** (e - 1)) * (1.0 + 0.5 * m)


def np_mxfp4_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Packed MXFP4 [..., K/2] codes + [..., K/32] E8M0 scales -> float64 [..., K].
    Low nibble of byte j is element 2j, high nibble element 2j+1."""
    codes = np.asarray(codes, dtype=np.uint8)
    lo = codes & 0x0F
    hi = codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (codes.shape[-1] * 2,))
    table = np.array([e2m1_value_from_bits(c) for c in range(16)], dtype=np.float64)
    vals = table[nib]
    sc = np.ldexp(1.0, np.asarray(scales, dtype=np.int64) - 127)
    sc = np.repeat(sc, 32, axis=-1)
    return vals * sc


def bf16_decode(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_neighbors(bits: int):
    """The two finite bf16 values adjacent to `bits` (same sign handling by integer steps)."""
    vals = []
    for d in (-1, 1):
        nb = (int(bits) + d) & 0xFFFF
        vals.append(float(bf16_decode(np.uint16(nb))))
    return vals


def is_nearest_bf16(bits, exact, slack=1e-12) -> np.ndarray:
    """True where bf16 `bits` is (one of) the bf16 value(s) nearest to `exact`.

    `slack` is a relative allowance for the reference's own rounding error, so that a
    value within slack of a tie accepts either neighbour."""
    bits = np.atleast_1d(np.asarray(bits, dtype=np.uint16))
    exact = np.atleast_1d(np.asarray(exact, dtype=np.float64))
    ok = np.empty(bits.shape, dtype=bool)
    for i, (b, x) in enumerate(zip(bits.ravel(), exact.ravel())):
        v = float(bf16_decode(b))
        d = abs(v - x)
        good = np.isfinite(v)
        for n in bf16_neighbors(b):
            if np.isfinite(n) and d > abs(n - x) * (1 + slack) + abs(x) * slack:
                good = False
        ok.ravel()[i] = good
    return ok


def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def quantize_to_nearest_bf16_bits(v) -> np.ndarray:
    """float64 -> bf16 bits, nearest with ties to even, by searching the two candidates
    around the float32 truncation (independent of both the oracle's and torch's routine)."""
    v = np.atleast_1d(np.asarray(v, dtype=np.float64))
    out = np.empty(v.shape, dtype=np.uint16)
    for i, x in enumerate(v.ravel()):
        f = np.float32(x)
        b = int(np.array([f], dtype=np.float32).view(np.uint32)[0] >> 16)
        cands = [(b + d) & 0xFFFF for d in (-1, 0, 1, 2)]
        best = None
        for c in cands:
            cv = float(bf16_decode(np.uint16(c)))
            if not np.isfinite(cv):
                continue
            key = (abs(cv - x), c & 1)  # nearest, then even mantissa
            if best is None or key < best[0]:
                best = (key, c)
        out.ravel()[i] = best[1]
    return out
