"""FP8 E4M3 decoding written from the format definition (test infrastructure).

Source: the guijiagi.com "推理优化" tag page, article on quantisation
("FP8量化" format table): E4M3 has 4 exponent bits and 3 mantissa bits and a
range of +-448.  The remaining details are the standard OCP-FP8 E4M3 rules
that this range implies:

* bit 7 is the sign, bits 6..3 the biased exponent (bias 7), bits 2..0 the
  mantissa;
* exponent field 0 encodes subnormals: value = (m / 8) * 2**(1 - 7);
* other exponent fields encode normals: value = (1 + m / 8) * 2**(e - 7);
* there is no infinity; only S.1111.111 (0x7F / 0xFF) is NaN, which is why
  the largest finite magnitude is 1.75 * 2**8 = 448.

Encoding (for the cache write) is rounding to the nearest representable
value, ties to the even code (the one whose mantissa's last bit is 0), with
magnitudes above the largest finite value saturated to 448 (the write
quantises and saturates: TokenSpeed code audit, mlqm.cn/news/403565, section
完整技术清单 > Attention 接入 / KV, fused FP8 KV-pack kernel; the saturation
to +-448 is the reading of "range +-448" for an encoder with no infinity).
A NaN encodes to a NaN code.

Parity: decoding is pinned in tests against torch.float8_e4m3fn (an
independent library decoder) for all 256 codes and against the hand-derived
extreme values; encoding against torch's float8 conversion on in-range
values, and against round trips, midpoints and saturation points derived
by hand.
"""
import numpy as np

_BIAS = 7


def _decode_one(code: int) -> float:
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return float("nan")
    if exp_field == 0:
        return sign * (mant / 8.0) * 2.0 ** (1 - _BIAS)
    return sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - _BIAS)


def e4m3_decode_table() -> np.ndarray:
    """float64[256]: value of every E4M3 byte."""
    return np.array([_decode_one(c) for c in range(256)], dtype=np.float64)


_TABLE = e4m3_decode_table()


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Decode an array of E4M3 bytes (uint8) to float64."""
    codes = np.asarray(codes)
    if codes.dtype != np.uint8:
        raise TypeError("E4M3 codes must be uint8")
    return _TABLE[codes]


# finite non-negative magnitudes, code 0x00 .. 0x7E in increasing order
_MAGS = _TABLE[:0x7F]


def e4m3_encode(x) -> np.ndarray:
    """Encode float values to E4M3 bytes: nearest value, ties to even code,
    |x| > 448 saturated to 448, NaN to 0x7F, the sign bit copied from x
    (so a negative value that rounds to zero gives -0, 0x80)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    flat_x, flat_o = x.reshape(-1), out.reshape(-1)
    for k in range(flat_x.size):
        v = flat_x[k]
        if np.isnan(v):
            flat_o[k] = 0x7F
            continue
        a = abs(v)
        if a >= _MAGS[-1]:
            code = 0x7E
        else:
            lo = int(np.searchsorted(_MAGS, a, side="right")) - 1  # _MAGS[lo] <= a < _MAGS[lo + 1]
            d_lo, d_hi = a - _MAGS[lo], _MAGS[lo + 1] - a
            if d_lo < d_hi:
                code = lo
            elif d_hi < d_lo:
                code = lo + 1
            else:
                code = lo if lo % 2 == 0 else lo + 1
        flat_o[k] = code | (0x80 if np.signbit(v) else 0)
    return out
