"""Pins for the oracle's store: slot layout against the page's 2.6x figure,
the matched-norm identity, bucketize against the midpoint definition,
value quantisation bounds, FP8 keys, and reconstruction error of the
whole encode/decode against the Gaussian quantizer distortion."""
import os

import numpy as np
import pytest

GOLD = os.path.join(os.path.dirname(__file__), "golden")
PRESETS = [0, 1, 2, 3, 4]


def _page_numbers():
    vals = {}
    for line in open(os.path.join(GOLD, "page_numbers.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_slot_sizes(orc):
    sizes = [orc.layout(p)["slot_size_aligned"] for p in PRESETS]
    assert sizes == [196, 134, 118, 102, 70]
    ratio = 2 * 128 * 2 / sizes[0]
    assert round(ratio, 1) == _page_numbers()["k8v4_compression"]
    for p in PRESETS:
        L = orc.layout(p)
        assert L["slot_size_aligned"] % 2 == 0
        assert L["off_v_zero"] + 2 == L["slot_size"]
        assert L["off_v_scale"] + 2 == L["off_v_zero"]


def _setup(orc, preset, D=128):
    L = orc.layout(preset, D)
    s = orc.signs(D, 42)
    if L["key_fp8"]:
        c32, m32 = np.zeros(1, np.float32), np.zeros(1, np.float32)
    else:
        c32, m32 = orc.codebook(D, L["key_bits"])
    return L, s, c32, m32


@pytest.mark.parametrize("preset", [1, 2, 3])
def test_mse_key_bucketize_and_matched_norm(orc, preset):
    rng = np.random.default_rng(preset)
    L, s, c32, m32 = _setup(orc, preset)
    for trial in range(50):
        k = (rng.normal(size=128) * rng.uniform(0.1, 5)).astype(np.float16).astype(np.float32)
        v = rng.normal(size=128).astype(np.float16).astype(np.float32)
        slot, y = orc.store_one(preset, k, v, s, c32, m32)
        idx = orc.unpack(slot[:L["key_data_bytes"]], 128, L["key_bits"])
        # bucketize: m[idx-1] < y <= m[idx]  (value on a midpoint takes the lower code)
        lo = np.concatenate([[-np.inf], m32])[idx]
        hi = np.concatenate([m32, [np.inf]])[idx]
        assert np.all(lo < y) and np.all(y <= hi)
        # y is the rotated, normalised key: unit norm
        assert abs(np.linalg.norm(y.astype(np.float64)) - 1) < 1e-5
        # matched norm: || norm * c[idx] || == ||k|| up to the fp16 rounding of norm
        norm = orc.f16_value(int(slot[L["off_k_norm"]]) | int(slot[L["off_k_norm"] + 1]) << 8)
        recon = norm * np.linalg.norm(c32[idx].astype(np.float64))
        assert abs(recon - np.linalg.norm(k)) <= 2.0**-11 * np.linalg.norm(k) * 1.0001
        # and the correction matters: ||c[idx]|| is not 1
        assert abs(np.linalg.norm(c32[idx]) - 1) > 1e-6


@pytest.mark.parametrize("preset", PRESETS)
def test_value_quantisation(orc, preset):
    rng = np.random.default_rng(10 + preset)
    L, s, c32, m32 = _setup(orc, preset)
    qmax = (1 << L["value_bits"]) - 1
    for trial in range(50):
        v = (rng.normal(size=128) * rng.uniform(0.01, 10)).astype(np.float16).astype(np.float32)
        k = rng.normal(size=128).astype(np.float32)
        slot, _ = orc.store_one(preset, k, v, s, c32, m32)
        codes = orc.unpack(slot[L["off_v_data"]:L["off_v_data"] + L["value_data_bytes"]],
                           128, L["value_bits"])
        u16 = lambda o: int(slot[o]) | int(slot[o + 1]) << 8
        sc, z = orc.f16_value(u16(L["off_v_scale"])), orc.f16_value(u16(L["off_v_zero"]))
        assert z == float(np.float16(v.min()))
        assert abs(sc - (v.max() - v.min()) / qmax) <= 2.0**-11 * sc * 1.0001
        assert codes[np.argmin(v)] == 0
        assert codes[np.argmax(v)] >= qmax - 1 and codes.max() <= qmax
        vh = codes * sc + z
        assert np.max(np.abs(vh - v)) <= sc / 2 + abs(z - v.min()) + 2.0**-10 * sc * qmax
    # constant vector: scale 0, every code 0, v_hat == zero
    v = np.full(128, 0.75, np.float32)
    slot, _ = orc.store_one(preset, np.ones(128, np.float32), v, s, c32, m32)
    kh, vh = orc.dequant_slot(preset, slot, s, c32)
    assert np.all(vh == 0.75)


def test_fp8_keys(orc):
    rng = np.random.default_rng(3)
    L, s, c32, m32 = _setup(orc, 0)
    k = (rng.normal(size=128) * 3).astype(np.float16).astype(np.float32)
    slot, _ = orc.store_one(0, k, k, s, c32, m32)
    assert [int(b) for b in slot[:128]] == [orc.e4m3_encode(float(x)) for x in k]
    kh, _ = orc.dequant_slot(0, slot, s, c32)
    assert np.all(np.abs(kh - k) <= np.maximum(np.abs(k) * 2.0**-4, 2.0**-10))


@pytest.mark.parametrize("preset,distortion", [(1, 0.009497), (2, 0.03454), (3, 0.03454)])
def test_reconstruction_error_is_lloyd_max_distortion(orc, preset, distortion):
    """Random keys rotated to N(0, 1/d) coordinates: the relative squared
    error of k_hat is the Gaussian quantizer's distortion (Max, 1960:
    0.009497 at 4 bits, 0.03454 at 3 bits), here within 25%.  A wrong sign,
    index or transpose anywhere in store or dequant breaks this."""
    rng = np.random.default_rng(7)
    L, s, c32, m32 = _setup(orc, preset)
    errs = []
    for _ in range(200):
        k = rng.normal(size=128).astype(np.float32)
        slot, _ = orc.store_one(preset, k, k, s, c32, m32)
        kh, _ = orc.dequant_slot(preset, slot, s, c32)
        errs.append(np.sum((kh - k) ** 2) / np.sum(k.astype(np.float64) ** 2))
    assert abs(np.mean(errs) / distortion - 1) < 0.25


def test_zero_key(orc):
    L, s, c32, m32 = _setup(orc, 1)
    slot, y = orc.store_one(1, np.zeros(128, np.float32), np.zeros(128, np.float32), s, c32, m32)
    assert np.all(y == 0)
    assert slot[L["off_k_norm"]] == 0 and slot[L["off_k_norm"] + 1] == 0
    kh, vh = orc.dequant_slot(1, slot, s, c32)
    assert np.all(kh == 0) and np.all(vh == 0)


def test_store_paging_and_padding(orc):
    rng = np.random.default_rng(11)
    preset, Hk, bs, nb = 2, 2, 16, 5
    L, s, c32, m32 = _setup(orc, preset)
    S = L["slot_size_aligned"]
    N = 20
    key = rng.normal(size=(N, Hk, 128)).astype(np.float32)
    val = rng.normal(size=(N, Hk, 128)).astype(np.float32)
    sm = rng.permutation(nb * bs)[:N].astype(np.int64)
    sm[3] = -1
    cache = np.full((nb, bs, Hk, S), 0xAB, np.uint8)
    orc.store(preset, key, val, sm, cache, bs, s, c32, m32)
    flat = cache.reshape(nb * bs, Hk, S)
    for t in range(N):
        for h in range(Hk):
            if sm[t] < 0:
                continue
            ref, _ = orc.store_one(preset, key[t, h], val[t, h], s, c32, m32)
            assert np.array_equal(flat[sm[t], h], ref)
    untouched = np.setdiff1d(np.arange(nb * bs), sm[sm >= 0])
    assert np.all(flat[untouched] == 0xAB)


@pytest.mark.parametrize("preset", PRESETS)
def test_soa_store_is_a_rearrangement(orc, preset):
    """The oracle's SoA store writes the same slot bytes as its AoS store, in
    the places the SoA definition gives (an independent numpy re-arrangement),
    and its decode reads them back to the same attention."""
    from _helpers import aos_to_soa
    rng = np.random.default_rng(5150 + preset)
    D, Hk, bs, N = 128, 3, 16, 40
    L = orc.layout(preset)
    s = orc.signs(D, 42)
    c32, m32 = (np.zeros(1, np.float32),) * 2 if L["key_fp8"] else orc.codebook(D, L["key_bits"])
    k = rng.normal(size=(N, Hk, D)).astype(np.float32)
    v = rng.normal(size=(N, Hk, D)).astype(np.float32)
    sm = rng.permutation(3 * bs)[:N].astype(np.int64)
    aos = np.zeros((3, bs, Hk, L["slot_size_aligned"]), np.uint8)
    soa = np.zeros_like(aos)
    orc.store(preset, k, v, sm, aos, bs, s, c32, m32)
    orc.store(preset | orc.LAYOUT_SOA, k, v, sm, soa, bs, s, c32, m32)
    assert np.array_equal(soa, aos_to_soa(orc, preset, aos))
    q = rng.normal(size=(1, 2 * Hk, D)).astype(np.float32)
    bt = np.array([[0, 1, 2]], np.int32)
    sl = np.array([3 * bs], np.int32)
    o1, l1 = orc.decode_dense(preset, q, aos, bt, sl, Hk, bs, s, c32)
    o2, l2 = orc.decode_dense(preset | orc.LAYOUT_SOA, q, soa, bt, sl, Hk, bs, s, c32)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("preset,qmax", [(1, 15), (3, 7), (4, 3)])
def test_value_code_ties_round_half_even(orc, preset, qmax):
    """Exact half-integer quotients round to the even code (reading R9,
    round-half-even): with min 0 and max qmax the fp16 scale is exactly 1
    and the zero 0, so v itself is the quotient.  Worked by hand: 0.5 -> 0,
    1.5 -> 2, 2.5 -> 2, and qmax - 0.5 -> the even neighbour; a round-half-up
    rule would give 1, 2, 3 and qmax there."""
    L, s, c32, m32 = _setup(orc, preset)
    v = np.zeros(128, np.float32)
    v[1] = qmax
    ties = {2: 0.5, 3: 1.5, 4: 2.5, 5: qmax - 0.5}
    for i, x in ties.items():
        v[i] = x
    k = np.random.default_rng(0).normal(size=128).astype(np.float32)
    slot, _ = orc.store_one(preset, k, v, s, c32, m32)
    u16 = lambda o: int(slot[o]) | int(slot[o + 1]) << 8
    assert orc.f16_value(u16(L["off_v_scale"])) == 1.0
    assert orc.f16_value(u16(L["off_v_zero"])) == 0.0
    codes = orc.unpack(slot[L["off_v_data"]:L["off_v_data"] + L["value_data_bytes"]], 128,
                       L["value_bits"])
    even = lambda x: int(np.floor(x)) if int(np.floor(x)) % 2 == 0 else int(np.floor(x)) + 1
    assert codes[1] == qmax
    for i, x in ties.items():
        assert codes[i] == even(x), (i, x, codes[i])
    assert [codes[i] for i in (2, 3, 4)] == [0, 2, 2]


def test_value_code_ties_scaled(orc):
    """The same rule through a non-unit scale: 4-bit values on [0, 7.5] give
    scale 0.5 (exact in fp16), so v = 1.25 and 1.75 are quotients 2.5 and
    3.5 and take codes 2 and 4."""
    L, s, c32, m32 = _setup(orc, 1)
    v = np.zeros(128, np.float32)
    v[1], v[2], v[3] = 7.5, 1.25, 1.75
    slot, _ = orc.store_one(1, np.ones(128, np.float32), v, s, c32, m32)
    codes = orc.unpack(slot[L["off_v_data"]:L["off_v_data"] + 64], 128, 4)
    assert list(codes[1:4]) == [15, 2, 4]
