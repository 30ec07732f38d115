"""Pins for the oracle's bit packing: byte examples worked out by hand for
the LSB-first reading (2/4 bits) and the 32-code group reading (3 bits),
round trips over every code value, and the packed sizes the pages give
(8 values per 3 bytes at 3 bits)."""
import numpy as np
import pytest


def test_worked_examples(orc):
    # 4-bit codes (1, 2): low nibble first
    assert list(orc.pack([1, 2], 4)) == [0x21]
    # 2-bit codes 0..3 -> 0b11100100
    assert list(orc.pack([0, 1, 2, 3], 2)) == [0xE4]
    # 3-bit group of 32: codes 0..7 in the nibbles of W0 (0x76543210), codes
    # 8..23 likewise in W1, W2; code 24+i spreads its bits over the top bit of
    # nibble i of W0, W1, W2.
    codes = [0] * 32
    for i in range(8):
        codes[i] = i
    assert list(orc.pack(codes, 3)) == [0x10, 0x32, 0x54, 0x76] + [0] * 8
    codes = [0] * 32
    codes[24] = 0b101          # bit 0 -> W0 bit 3, bit 2 -> W2 bit 3
    codes[31] = 0b010          # bit 1 -> W1 bit 31
    assert list(orc.pack(codes, 3)) == [0x08, 0, 0, 0, 0, 0, 0, 0x80, 0x08, 0, 0, 0]
    # 8 three-bit values per 3 bytes ("turboquant-plus.md", Background)
    assert orc.pack([7] * 32, 3).size == 12


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
def test_round_trip(orc, bits):
    rng = np.random.default_rng(bits)
    for n in ((32, 64, 128) if bits == 3 else (1, 7, 8, 128, 129)):
        codes = rng.integers(0, 1 << bits, n)
        data = orc.pack(codes, bits)
        assert data.size == (n * bits + 7) // 8
        assert np.array_equal(orc.unpack(data, n, bits), codes)
    every = np.arange(1 << bits).repeat(32 if bits <= 3 else 3)
    assert np.array_equal(orc.unpack(orc.pack(every, bits), every.size, bits), every)


def test_sizes_at_d128(orc):
    assert orc.pack(np.zeros(128, int), 4).size == 64
    assert orc.pack(np.zeros(128, int), 3).size == 48
    assert orc.pack(np.zeros(128, int), 2).size == 32
