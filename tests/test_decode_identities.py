"""Host checks of the fp16 bit identities the INT4 decode relies on (the kernels
apply them to packed halves; here each value is built from its bits with numpy).

A level n in 0..15 ORed into the mantissa of 1024.0 (bits 0x6400) is 1024 + n;
ORed in four bits higher it is 1024 + 16 n. Both decode exactly to the signed
level n - 8: (1024 + n) - 1032, and (1024 + 16 n) / 16 - 72 as one fma."""
import numpy as np


def half_from_bits(bits: int) -> np.float16:
    return np.array([bits], dtype=np.uint16).view(np.float16)[0]


def test_low_nibble_identity():
    for n in range(16):
        x = half_from_bits(0x6400 | n)
        assert float(x) == 1024 + n
        assert float(np.float16(x - half_from_bits(0x6408))) == n - 8   # 0x6408 = 1032


def test_high_nibble_identity():
    sixteenth, minus72 = half_from_bits(0x2C00), half_from_bits(0xD480)
    assert float(sixteenth) == 1 / 16 and float(minus72) == -72
    for n in range(16):
        x = half_from_bits(0x6400 | (n << 4))
        assert float(x) == 1024 + 16 * n
        exact = float(x) * float(sixteenth) + float(minus72)        # what one fma rounds once
        assert exact == n - 8 and float(np.float16(exact)) == exact
