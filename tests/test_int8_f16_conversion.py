"""Host check of the int8 -> f16 conversion the converter warps use (all 256 byte values).

The kernels expand each int8 weight byte v by biasing it to u = v + 128 (v XOR 0x80), placing u
in the low byte of an f16 whose high byte is 0x64 (the f16 1024 + u: 10 mantissa bits hold any
u < 256 exactly) and subtracting the f16 1152 = 1024 + 128.  Two bytes of a 32-bit word become
one f16 pair with a byte permute: selector 0x4140 takes bytes 0 and 1, 0x4342 bytes 2 and 3, each
paired with the constant byte 0x64 of the second permute operand.  This test emulates those
steps bit by bit and checks the result is v exactly for every int8 value, in each byte lane.
"""
import numpy as np


def byte_perm(x: int, y: int, sel: int) -> int:
    """CUDA __byte_perm: result byte i is byte (sel >> 4i) & 7 of the 8-byte value {y, x}."""
    src = x.to_bytes(4, "little") + y.to_bytes(4, "little")
    return int.from_bytes(bytes(src[(sel >> (4 * i)) & 7] for i in range(4)), "little")


def f16_pair_minus_1152(word: int) -> tuple:
    halves = np.array([word & 0xFFFF, word >> 16], dtype=np.uint16).view(np.float16)
    out = halves - np.float16(1152.0)                    # one packed f16 subtraction
    assert out.dtype == np.float16
    return float(out[0]), float(out[1])


def test_constants():
    assert np.array([0x6480], dtype=np.uint16).view(np.float16)[0] == np.float16(1152.0)
    for u in range(256):
        assert float(np.array([0x6400 | u], dtype=np.uint16).view(np.float16)[0]) == 1024.0 + u


def test_every_int8_in_every_byte_lane():
    vals = np.arange(-128, 128)
    for lane in range(4):
        for v in vals:
            others = [(lane * 37 + k * 11) % 256 - 128 for k in range(4)]   # other lanes vary
            lanes = [int(v) if k == lane else others[k] for k in range(4)]
            word = int.from_bytes(bytes((x & 0xFF) for x in lanes), "little")
            biased = word ^ 0x80808080
            lo = f16_pair_minus_1152(byte_perm(biased, 0x64646464, 0x4140))
            hi = f16_pair_minus_1152(byte_perm(biased, 0x64646464, 0x4342))
            got = list(lo) + list(hi)
            assert got == [float(x) for x in lanes], (lane, int(v), got, lanes)
