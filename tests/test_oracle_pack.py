"""Pins for the oracle's bit packing: byte examples worked out by hand for
the LSB-first bitstream reading at every width, the 8-codes-per-3-bytes
grouping the pages give for 3-bit data, round trips over every code value,
and the packed sizes at head_dim 128."""
import numpy as np
import pytest


def test_worked_examples(orc):
    # 4-bit codes (1, 2): low nibble first
    assert list(orc.pack([1, 2], 4)) == [0x21]
    # 2-bit codes 0..3 -> 0b11100100
    assert list(orc.pack([0, 1, 2, 3], 2)) == [0xE4]
    # 3-bit codes 0..7, worked by hand: bit stream (LSB first)
    #   000 100 010 110 001 101 011 111  ->  bytes 0b10001000, 0b11000110, 0b11111010
    assert list(orc.pack(list(range(8)), 3)) == [0x88, 0xC6, 0xFA]
    # a code that straddles a byte: code 2 = 0b101 sits in bits 6..8
    assert list(orc.pack([0, 0, 5], 3)) == [0x40, 0x01]


def test_three_bit_groups_of_three_bytes(orc):
    """8 values per 3 bytes ("turboquant-plus.md", Background): every
    3-byte group holds 8 whole codes, so group g depends on codes 8g..8g+7
    only."""
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 8, 128)
    data = orc.pack(codes, 3)
    assert data.size == 48
    for g in range(16):
        alone = orc.pack(codes[8 * g:8 * g + 8], 3)
        assert np.array_equal(data[3 * g:3 * g + 3], alone)


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
def test_round_trip(orc, bits):
    rng = np.random.default_rng(bits)
    for n in (1, 7, 8, 32, 128, 129):
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
