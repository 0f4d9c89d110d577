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

Parity: pinned in tests against torch.float8_e4m3fn (an independent library
decoder) for all 256 codes and against the hand-derived extreme values.
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
