"""GPU parity of the fused store (through the C ABI) against the oracle:
slot bytes bit-exact except counted boundary ties, norms within 1 fp16 ulp,
untouched slots left alone, padding tokens skipped."""
import math

import numpy as np
import pytest
import torch

import quantized_kv_cache_04_gb300 as tq
from _helpers import TIE_FRACTION, codebook, compare_store, to_f32

pytestmark = pytest.mark.gpu
PRESETS = [0, 1, 2, 3, 4]
SENTINEL = 0x5A


def _run_store(orc, preset, K, V, slot_mapping, num_blocks, bs, key_view=None, value_view=None):
    N, Hk, D = K.shape
    L = tq.tq_get_layout(preset)
    dev = torch.device("cuda")
    s = orc.signs(D, 42)
    c32, m32 = codebook(orc, preset)
    cache = torch.full((num_blocks, bs, Hk, L["slot_size_aligned"]), SENTINEL, dtype=torch.uint8,
                       device=dev)
    kd = (key_view if key_view is not None else K).to(dev)
    vd = (value_view if value_view is not None else V).to(dev)
    if key_view is not None:
        kd = key_view
        vd = value_view
    sm = torch.from_numpy(slot_mapping).to(dev)
    sg = torch.from_numpy(s).to(dev)
    cc = torch.from_numpy(c32).to(dev) if not L["key_fp8"] else None
    mm = torch.from_numpy(m32).to(dev) if not L["key_fp8"] else None
    tq.store(preset, kd, vd, sm, cache, bs, sg, cc, mm)
    torch.cuda.synchronize()
    return cache.cpu().numpy(), s, c32, m32


def _check(orc, preset, K, V, slot_mapping, cache, s, c32, m32, bs, bound_fraction=True):
    N, Hk, D = K.shape
    flat = cache.reshape(-1, Hk, cache.shape[-1])
    live = slot_mapping >= 0
    rows = flat[slot_mapping[live]].reshape(-1, cache.shape[-1])
    kf = to_f32(K)[live].reshape(-1, D)
    vf = to_f32(V)[live].reshape(-1, D)
    flips, codes = compare_store(orc, preset, rows, kf, vf, s, c32, m32)
    if bound_fraction:
        assert flips <= max(1, math.ceil(TIE_FRACTION * codes)), (flips, codes)
    untouched = np.setdiff1d(np.arange(flat.shape[0]), slot_mapping[live])
    assert np.all(flat[untouched] == SENTINEL)
    return flips, codes


@pytest.mark.parametrize("preset", PRESETS)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("Hk,N,bs", [(8, 300, 16), (2, 77, 128), (3, 50, 32), (1, 1, 64),
                                     (32, 9, 16)])
def test_store_parity(orc, preset, dtype, Hk, N, bs):
    rng = np.random.default_rng(preset * 1000 + Hk * 10 + bs)
    K = torch.from_numpy(rng.normal(size=(N, Hk, 128)) * rng.uniform(0.2, 3.0)).to(dtype)
    V = torch.from_numpy(rng.normal(size=(N, Hk, 128)) * rng.uniform(0.2, 3.0)).to(dtype)
    K[..., 5] *= 8
    V[..., 17] *= 8
    num_blocks = (N + bs - 1) // bs + 2
    sm = rng.permutation(num_blocks * bs)[:N].astype(np.int64)
    if N > 3:
        sm[rng.choice(N, max(1, N // 10), replace=False)] = -1
    cache, s, c32, m32 = _run_store(orc, preset, K, V, sm, num_blocks, bs)
    _check(orc, preset, K, V, sm, cache, s, c32, m32, bs)


@pytest.mark.parametrize("preset", PRESETS)
def test_store_edge_values(orc, preset):
    """Zero and constant vectors, tiny and large magnitudes (fp8 saturation),
    one-hot keys, and a strided (non-contiguous token stride) input view.
    Structured keys put many rotated coordinates exactly on a decision
    boundary (e.g. Hadamard cancellation to 0 against the middle midpoint),
    so every flip must still be an adjacent code at a tie, but the 1e-4
    fraction (a bar for random data) is not applied here."""
    Hk, D, bs = 4, 128, 16
    rows = [np.zeros(D), np.full(D, 3.0), np.full(D, -1e-6), np.eye(D)[7] * 5,
            np.linspace(-600, 600, D), np.linspace(-1, 1, D) * 1e-4,
            np.r_[np.full(64, 2.0), np.full(64, -2.0)], np.arange(D) % 3 - 1.0]
    N = len(rows)
    base = np.stack([np.stack([r * (h + 1) for h in range(Hk)]) for r in rows])
    for dtype in (torch.float16, torch.bfloat16):
        K = torch.from_numpy(base).to(dtype)
        V = torch.from_numpy(base[::-1].copy()).to(dtype)
        # strided views: tokens 3*Hk*D apart inside a larger qkv-like buffer
        big = torch.zeros((N, 3, Hk, D), dtype=dtype)
        big[:, 0] = K
        big[:, 2] = V
        bigd = big.cuda()
        kview, vview = bigd[:, 0], bigd[:, 2]
        sm = np.arange(N, dtype=np.int64) * 3 + 1
        cache, s, c32, m32 = _run_store(orc, preset, K, V, sm, (3 * N) // bs + 2, bs,
                                        key_view=kview, value_view=vview)
        _check(orc, preset, K, V, sm, cache, s, c32, m32, bs, bound_fraction=False)


@pytest.mark.parametrize("preset", PRESETS)
def test_store_value_code_ties(orc, preset):
    """Value rows whose quotients (v - zero) / scale are exact half-integers
    (scale 1 and 0.25, exact in fp16) or lie within fp16 rounding of one
    (scale 0.3): the codes must round half to even exactly as the oracle's
    correctly rounded fp32 division does, bit for bit."""
    L = tq.tq_get_layout(preset)
    qmax = 2 ** L["value_bits"] - 1
    rng = np.random.default_rng(9900 + preset)
    Hk, D, bs = 2, 128, 16
    rows = []
    for lo, step in ((0.0, 1.0), (-3.0, 0.25), (0.0, 0.3), (7.0, 0.3)):
        half = lo + (np.arange(D) % qmax + 0.5) * step
        half[0], half[1] = lo, lo + qmax * step          # fix the min and the max
        rows.append(half)
    rows.append(rng.permutation(rows[1]))
    N = len(rows)
    V = torch.from_numpy(np.stack([np.stack([r] * Hk) for r in rows])).to(torch.float16)
    for dtype in (torch.float16, torch.bfloat16):
        Vd = V.to(dtype)
        K = torch.from_numpy(rng.normal(size=(N, Hk, D))).to(dtype)
        sm = np.arange(N, dtype=np.int64) * 2
        cache, s, c32, m32 = _run_store(orc, preset, K, Vd, sm, (2 * N) // bs + 2, bs)
        _check(orc, preset, K, Vd, sm, cache, s, c32, m32, bs, bound_fraction=False)


@pytest.mark.parametrize("preset", PRESETS)
def test_store_unaligned_rows(orc, preset):
    """Input rows that are only 2-byte aligned (a view starting one element
    into a buffer whose token stride is not a multiple of 4 elements): the
    store reads them element by element and writes the same slots as for
    contiguous inputs."""
    rng = np.random.default_rng(9100 + preset)
    N, Hk, D, bs = 45, 8, 128, 16
    K = torch.from_numpy(rng.normal(size=(N, Hk, D))).to(torch.float16)
    V = torch.from_numpy(rng.normal(size=(N, Hk, D))).to(torch.float16)
    row = Hk * D + 6
    kb = torch.zeros((N, row), dtype=torch.float16)
    vb = torch.zeros((N, row), dtype=torch.float16)
    kb[:, 1:1 + Hk * D] = K.reshape(N, -1)
    vb[:, 3:3 + Hk * D] = V.reshape(N, -1)
    kbd, vbd = kb.cuda(), vb.cuda()
    kview = kbd[:, 1:1 + Hk * D].view(N, Hk, D)
    vview = vbd[:, 3:3 + Hk * D].view(N, Hk, D)
    assert kview.data_ptr() % 8 == 2 and kview.stride(0) % 4 == 2
    num_blocks = (N + bs - 1) // bs + 1
    sm = rng.permutation(num_blocks * bs)[:N].astype(np.int64)
    cache_u, s, c32, m32 = _run_store(orc, preset, K, V, sm, num_blocks, bs,
                                      key_view=kview, value_view=vview)
    cache_c, _, _, _ = _run_store(orc, preset, K, V, sm, num_blocks, bs)
    assert np.array_equal(cache_u, cache_c)
    _check(orc, preset, K, V, sm, cache_u, s, c32, m32, bs)


def test_store_padding_only_and_large_batch(orc):
    """All-padding slot mapping writes nothing; a 16384-token store over 8
    heads matches the oracle on a sample of tokens."""
    preset, Hk, bs = 2, 8, 32
    K = torch.randn(16, Hk, 128, dtype=torch.float16)
    sm = np.full(16, -1, np.int64)
    cache, *_ = _run_store(orc, preset, K, K, sm, 4, bs)
    assert np.all(cache == SENTINEL)

    rng = np.random.default_rng(9)
    N = 16384
    g = torch.Generator().manual_seed(3)
    K = torch.randn(N, Hk, 128, generator=g).to(torch.float16)
    V = torch.randn(N, Hk, 128, generator=g).to(torch.float16)
    nb = N // bs + 1
    sm = rng.permutation(nb * bs)[:N].astype(np.int64)
    cache, s, c32, m32 = _run_store(orc, preset, K, V, sm, nb, bs)
    pick = rng.choice(N, 512, replace=False)
    flat = cache.reshape(-1, Hk, cache.shape[-1])
    rows = flat[sm[pick]].reshape(-1, cache.shape[-1])
    flips, codes = compare_store(orc, preset, rows, to_f32(K[pick]).reshape(-1, 128),
                                 to_f32(V[pick]).reshape(-1, 128), s, c32, m32)
    assert flips <= max(1, math.ceil(TIE_FRACTION * codes))


@pytest.mark.parametrize("preset", PRESETS)
@pytest.mark.parametrize("Hk,bs", [(8, 16), (3, 32), (1, 64)])
def test_store_soa_is_the_aos_rearranged(orc, preset, Hk, bs):
    """The SoA store (TQ_LAYOUT_SOA) writes, from the same inputs, exactly the
    bytes of the AoS store re-arranged per the SoA definition (blocks never
    written keep their contents in both)."""
    from _helpers import aos_to_soa
    rng = np.random.default_rng(6200 + 10 * preset + Hk)
    N, nb = 150, 12
    K = torch.from_numpy(rng.normal(size=(N, Hk, 128))).to(torch.float16)
    V = torch.from_numpy(rng.normal(size=(N, Hk, 128))).to(torch.float16)
    sm = rng.permutation(nb * bs)[:N].astype(np.int64)
    sm[::17] = -1
    aos, *_ = _run_store(orc, preset, K, V, sm, nb, bs)
    soa, *_ = _run_store(orc, preset | tq.TQ_LAYOUT_SOA, K, V, sm, nb, bs)
    touched = np.unique(sm[sm >= 0] // bs)
    assert np.array_equal(soa[touched], aos_to_soa(orc, preset, aos[touched]))
    rest = np.setdiff1d(np.arange(nb), touched)
    assert np.all(soa[rest] == SENTINEL)


@pytest.mark.parametrize("preset", PRESETS)
def test_store_skips_slots_outside_the_cache(orc, preset):
    """Slots at or past num_blocks * block_size (and negative ones) are not
    written.  The cache handed to the store is a view of the first num_blocks
    blocks of a larger buffer, so the slots past it still name memory this
    process owns: the two blocks after the view must keep the sentinel."""
    rng = np.random.default_rng(9800 + preset)
    N, Hk, bs, num_blocks = 96, 4, 16, 4
    L = tq.tq_get_layout(preset)
    dev = torch.device("cuda")
    K = torch.from_numpy(rng.normal(size=(N, Hk, 128))).to(torch.float16)
    V = torch.from_numpy(rng.normal(size=(N, Hk, 128))).to(torch.float16)
    nslots = num_blocks * bs
    sm = np.concatenate([rng.permutation(nslots)[:N - 32],
                         nslots + rng.permutation(2 * bs)[:24], [-1] * 8]).astype(np.int64)
    rng.shuffle(sm)
    big = torch.full((num_blocks + 2, bs, Hk, L["slot_size_aligned"]), SENTINEL, dtype=torch.uint8,
                     device=dev)
    cache = big[:num_blocks]
    s = orc.signs(128, 42)
    c32, m32 = codebook(orc, preset)
    cc = torch.from_numpy(c32).to(dev) if not L["key_fp8"] else None
    mm = torch.from_numpy(m32).to(dev) if not L["key_fp8"] else None
    tq.store(preset, K.to(dev), V.to(dev), torch.from_numpy(sm).to(dev), cache, bs,
             torch.from_numpy(s).to(dev), cc, mm)
    torch.cuda.synchronize()
    out = big.cpu().numpy()
    assert np.all(out[num_blocks:] == SENTINEL)
    live = (sm >= 0) & (sm < nslots)
    lt = torch.from_numpy(live)
    _check(orc, preset, K[lt], V[lt], sm[live], out[:num_blocks], s, c32, m32, bs)
