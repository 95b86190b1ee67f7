"""Element decoding for the oracle (test infrastructure only).

bfloat16 is the upper half of an IEEE-754 binary32: sign, 8 exponent bits
(bias 127), 7 mantissa bits.  float8_e4m3fn (the "fn" variant named in the
flare_mla_prefill page, Parameters: dtype) has 1 sign bit, 4 exponent bits with
bias 7 and 3 mantissa bits; exponent 0 encodes subnormals 2^-6 * m/8, the code
with all exponent and mantissa bits set is NaN, and there is no infinity, so
the largest finite magnitude is 2^8 * 1.75 = 448.
"""
import numpy as np


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 (exact)."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def _e4m3_table() -> np.ndarray:
    table = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp = (code >> 3) & 0xF
        man = code & 0x7
        if exp == 0xF and man == 0x7:
            table[code] = np.nan
        elif exp == 0:
            table[code] = sign * (man / 8.0) * 2.0 ** (1 - 7)
        else:
            table[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)
    return table


E4M3_VALUES = _e4m3_table()


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """uint8 e4m3fn codes -> float64 (exact)."""
    return E4M3_VALUES[codes.astype(np.intp)]
