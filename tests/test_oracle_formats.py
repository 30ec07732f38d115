"""Pins for the oracle's scalar formats: fp16 and bf16 against numpy/torch
conversions, FP8 E4M3 exhaustively against torch's float8_e4m3fn cast."""
import numpy as np
import torch


def test_fp16_roundtrip_all_patterns(orc):
    for bits in range(0, 1 << 16, 7):
        v = orc.f16_value(bits)
        ref = float(np.array([bits], np.uint16).view(np.float16)[0])
        if np.isnan(ref):
            assert np.isnan(v)
            continue
        assert v == ref
        if np.isfinite(v) and not (v == 0 and bits == 0x8000):
            assert orc.f16_bits(v) == bits


def test_fp16_rne_matches_numpy(orc):
    rng = np.random.default_rng(5)
    xs = np.concatenate([rng.normal(0, 1, 3000), rng.normal(0, 1e-5, 2000),
                         rng.normal(0, 3e4, 1000), [65519.99, 65520.0, 1e-8, 2.0**-25,
                                                    3 * 2.0**-26, 2.0**-24 * 1.5]])
    for x in xs:
        ref = int(np.array([x], np.float64).astype(np.float16).view(np.uint16)[0])
        assert orc.f16_bits(x) == ref, x


def test_bf16(orc):
    for bits in range(0, 1 << 16, 13):
        t = torch.tensor([bits], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
        ref = float(t.float()[0])
        v = orc.bf16_value(bits)
        assert (np.isnan(ref) and np.isnan(v)) or v == ref


def test_e4m3_exhaustive_over_fp16_inputs(orc):
    """Every finite fp16 value: the oracle's RNE encoder equals torch's cast
    inside the representable range; beyond it the encoder saturates."""
    allf = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    x = allf.astype(np.float32)
    fin = np.isfinite(x)
    ref = torch.from_numpy(x[fin]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([orc.e4m3_encode(float(v)) for v in x[fin]], np.uint8)
    inr = np.abs(x[fin]) < 464.0       # below the first value that rounds past 448
    assert np.array_equal(ours[inr], ref[inr])
    # saturation to +-448 (0x7E / 0xFE) beyond the range
    big = ~inr
    assert np.all((ours[big] & 0x7F) == 0x7E)
    assert np.all((ours[big] >> 7) == (x[fin][big] < 0))


def test_e4m3_decode_encode_identity(orc):
    n = 0
    for b in range(256):
        v = orc.e4m3_decode(b)
        if np.isnan(v):
            assert (b & 0x7F) == 0x7F
            continue
        n += 1
        assert orc.e4m3_encode(v) == b
        ref = float(torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn).float()[0])
        assert v == ref
    assert n == 254
    assert orc.e4m3_decode(0x7E) == 448.0
