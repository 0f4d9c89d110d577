"""Inputs of the cache write on which two readings of "quantise x with the
per-tensor scale s" pick different e4m3 codes: the code nearest to the
exact quotient x / s, and the code of the fp32 product x * fp32(1 / s).  The
two differ only when x / s lies within about 2^-23 (relative) of a midpoint
between two codes, so such inputs are constructed: for a bf16 value x and a
midpoint m, the fp32 numbers s next to x / m are tried.

Both readings are evaluated here with exact rational arithmetic against the
e4m3 values decoded by torch (independent of the oracle's code)."""
from fractions import Fraction

import numpy as np


def e4m3_values():
    """float64[127]: magnitudes of the finite non-negative e4m3 codes 0x00 .. 0x7E."""
    import torch

    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def nearest_code(q: Fraction, mags) -> int:
    """e4m3 code nearest to the rational q, ties to the even code, magnitudes
    beyond 448 saturated; the sign bit from q (q != 0 here)."""
    a = abs(q)
    best = None
    for c, v in enumerate(mags):
        d = abs(Fraction(v) - a)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    code = 0x7E if a >= 448 else best[1]
    return code | (0x80 if q < 0 else 0)


def bf16_bits(x: float) -> np.uint16:
    b = int(np.array([x], dtype=np.float32).view(np.uint32)[0])
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16  # round to nearest even
    return np.uint16(b)


def bits_to_float(bits) -> float:
    return float((np.array([bits], dtype=np.uint32) << 16).view(np.float32)[0])


def distinguishing_cases(n: int, seed: int = 0):
    """n pairs (bf16 bits of x, fp32 s) where the two readings differ."""
    mags = e4m3_values()
    mids = [(mags[i] + mags[i + 1]) / 2 for i in range(8, len(mags) - 1)]
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        xb = bf16_bits(float(rng.standard_normal() * 4))
        x = bits_to_float(xb)
        if x == 0.0:
            continue
        m = mids[int(rng.integers(len(mids)))]
        s = np.float32(abs(x) / m)
        for _ in range(4):
            s = np.nextafter(s, np.float32(np.inf) if rng.integers(2) else np.float32(-np.inf))
            sf = np.float32(s)
            exact = nearest_code(Fraction(x) / Fraction(float(sf)), mags)
            prod = np.float32(np.float32(x) * (np.float32(1.0) / sf))
            recip = nearest_code(Fraction(float(prod)), mags)
            if exact != recip:
                out.append((xb, float(sf)))
                break
    return out
