"""Pins for the oracle's bit packing: byte examples worked out by hand for
the LSB-first reading, round trips over every code value, and the packed
sizes the pages give (8 values per 3 bytes at 3 bits)."""
import numpy as np
import pytest


def test_worked_examples(orc):
    # 3-bit codes 0..7: sum(i << 3i) = 0xFAC688 -> bytes 88 C6 FA
    assert list(orc.pack(range(8), 3)) == [0x88, 0xC6, 0xFA]
    # 4-bit codes (1, 2): low nibble first
    assert list(orc.pack([1, 2], 4)) == [0x21]
    # 2-bit codes 0..3 -> 0b11100100
    assert list(orc.pack([0, 1, 2, 3], 2)) == [0xE4]
    # 8 three-bit values fill exactly 3 bytes ("turboquant-plus.md", Background)
    assert orc.pack([7] * 8, 3).size == 3


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
def test_round_trip(orc, bits):
    rng = np.random.default_rng(bits)
    for n in (1, 7, 8, 128, 129):
        codes = rng.integers(0, 1 << bits, n)
        data = orc.pack(codes, bits)
        assert data.size == (n * bits + 7) // 8
        assert np.array_equal(orc.unpack(data, n, bits), codes)
    every = np.arange(1 << bits).repeat(3)
    assert np.array_equal(orc.unpack(orc.pack(every, bits), every.size, bits), every)


def test_sizes_at_d128(orc):
    assert orc.pack(np.zeros(128, int), 4).size == 64
    assert orc.pack(np.zeros(128, int), 3).size == 48
    assert orc.pack(np.zeros(128, int), 2).size == 32
