"""Pins for the oracle's decode attention: the dense definition against an
independent numpy softmax over dequantised slots (its own paging), the
split-K/LUT form against the dense form, and closed-form special cases."""
import numpy as np
import pytest

PRESETS = [0, 1, 2, 3, 4]


def _cache(orc, preset, seq_lens, Hk, bs, rng, scale_k=1.0, kind="normal"):
    D = 128
    L = orc.layout(preset)
    s = orc.signs(D, 42)
    if L["key_fp8"]:
        c32, m32 = np.zeros(1, np.float32), np.zeros(1, np.float32)
    else:
        c32, m32 = orc.codebook(D, L["key_bits"])
    nblk = [(n + bs - 1) // bs for n in seq_lens]
    total = sum(nblk)
    perm = rng.permutation(total)
    width = max(1, max(nblk))
    bt = np.full((len(seq_lens), width), total, np.int32)
    cache = np.zeros((total + 1, bs, Hk, L["slot_size_aligned"]), np.uint8)
    pos = 0
    for b, n in enumerate(seq_lens):
        bt[b, :nblk[b]] = perm[pos:pos + nblk[b]]
        pos += nblk[b]
        if n == 0:
            continue
        k = (rng.normal(size=(n, Hk, D)) * scale_k).astype(np.float16).astype(np.float32)
        v = rng.normal(size=(n, Hk, D)).astype(np.float16).astype(np.float32)
        if kind == "equal_keys":
            k[:] = k[0]
        t = np.arange(n)
        sm = bt[b, t // bs].astype(np.int64) * bs + t % bs
        orc.store(preset, k, v, sm, cache, bs, s, c32, m32)
    return cache, bt, s, c32


def _numpy_attention(orc, preset, q, cache, bt, seq_lens, Hk, bs, s, c32):
    """Dequantise every slot with dequant_slot, then softmax with numpy."""
    B, Hq, D = q.shape
    G = Hq // Hk
    out = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -np.inf)
    flat = cache.reshape(-1, Hk, cache.shape[-1])
    for b in range(B):
        n = seq_lens[b]
        if n == 0:
            continue
        for hq in range(Hq):
            h = hq // G
            K = np.zeros((n, D)); V = np.zeros((n, D))
            for t in range(n):
                row = bt[b, t // bs] * bs + t % bs
                K[t], V[t] = orc.dequant_slot(preset, flat[row, h], s, c32)
            logit = K @ q[b, hq].astype(np.float64) / np.sqrt(D)
            m = logit.max()
            p = np.exp(logit - m)
            out[b, hq] = (p / p.sum()) @ V
            lse[b, hq] = m + np.log(p.sum())
    return out, lse


@pytest.mark.parametrize("preset", PRESETS)
def test_dense_equals_numpy_softmax(orc, preset):
    rng = np.random.default_rng(100 + preset)
    seq_lens = np.array([37, 5, 16], np.int32)
    Hk, Hq, bs = 2, 8, 16
    cache, bt, s, c32 = _cache(orc, preset, seq_lens, Hk, bs, rng)
    q = rng.normal(size=(3, Hq, 128)).astype(np.float32)
    o, l = orc.decode_dense(preset, q, cache, bt, seq_lens, Hk, bs, s, c32)
    o2, l2 = _numpy_attention(orc, preset, q, cache, bt, seq_lens, Hk, bs, s, c32)
    assert np.max(np.abs(o - o2)) < 1e-12 and np.max(np.abs(l - l2)) < 1e-12


@pytest.mark.parametrize("preset", PRESETS)
@pytest.mark.parametrize("splits", [1, 3, 8, 64])
def test_split_lut_equals_dense(orc, preset, splits):
    rng = np.random.default_rng(200 + preset)
    seq_lens = np.array([100, 1, 0, 33], np.int32)
    Hk, Hq, bs = 2, 4, 16
    cache, bt, s, c32 = _cache(orc, preset, seq_lens, Hk, bs, rng, scale_k=2.0)
    q = rng.normal(size=(4, Hq, 128)).astype(np.float32) * 2
    o, l = orc.decode_dense(preset, q, cache, bt, seq_lens, Hk, bs, s, c32)
    o2, l2 = orc.decode_split(preset, q, cache, bt, seq_lens, Hk, bs, s, c32, splits)
    assert np.max(np.abs(o - o2)) < 1e-10
    fin = np.isfinite(l)
    assert np.max(np.abs(l[fin] - l2[fin])) < 1e-10
    assert np.array_equal(fin, np.isfinite(l2))
    # empty sequence: zero output, -inf lse
    assert np.all(o[2] == 0) and np.all(np.isneginf(l[2]))


@pytest.mark.parametrize("preset", PRESETS)
def test_single_token_and_equal_keys(orc, preset):
    rng = np.random.default_rng(300 + preset)
    Hk, Hq, bs = 2, 4, 16
    # one token: out = v_hat_0, lse = logit_0
    cache, bt, s, c32 = _cache(orc, preset, np.array([1], np.int32), Hk, bs, rng)
    q = rng.normal(size=(1, Hq, 128)).astype(np.float32)
    o, l = orc.decode_dense(preset, q, cache, bt, np.array([1], np.int32), Hk, bs, s, c32)
    for hq in range(Hq):
        kh, vh = orc.dequant_slot(preset, cache[bt[0, 0], 0, hq // 2], s, c32)
        assert np.max(np.abs(o[0, hq] - vh)) < 1e-12
        assert abs(l[0, hq] - kh @ q[0, hq] / np.sqrt(128)) < 1e-12
    # equal keys: out = mean of v_hat, lse = logit + ln n
    n = 40
    cache, bt, s, c32 = _cache(orc, preset, np.array([n], np.int32), Hk, bs, rng,
                               kind="equal_keys")
    o, l = orc.decode_split(preset, q, cache, bt, np.array([n], np.int32), Hk, bs, s, c32, 3)
    flat = cache.reshape(-1, Hk, cache.shape[-1])
    for hq in range(Hq):
        rows = [bt[0, t // bs] * bs + t % bs for t in range(n)]
        V = np.array([orc.dequant_slot(preset, flat[r, hq // 2], s, c32)[1] for r in rows])
        kh, _ = orc.dequant_slot(preset, flat[rows[0], hq // 2], s, c32)
        assert np.max(np.abs(o[0, hq] - V.mean(0))) < 1e-10
        assert abs(l[0, hq] - (kh @ q[0, hq] / np.sqrt(128) + np.log(n))) < 1e-9


def _numpy_sparse_bound(orc, preset, q, cache, bt, seq_lens, Hk, bs, s, c32, tau):
    """The sparse-V bound by its definition, with numpy over dequantised slots."""
    B, Hq, D = q.shape
    G = Hq // Hk
    bound = np.zeros((B, Hq, D))
    mass = np.zeros((B, Hq))
    flat = cache.reshape(-1, Hk, cache.shape[-1])
    for b in range(B):
        n = seq_lens[b]
        for hq in range(Hq):
            h = hq // G
            K = np.zeros((n, D)); V = np.zeros((n, D))
            for t in range(n):
                row = bt[b, t // bs] * bs + t % bs
                K[t], V[t] = orc.dequant_slot(preset, flat[row, h], s, c32)
            e = np.exp(K @ q[b, hq].astype(np.float64) / np.sqrt(D) - (K @ q[b, hq] / np.sqrt(D)).max())
            drop = e <= tau
            bound[b, hq] = (e[drop, None] * np.abs(V[drop])).sum(0) / e.sum()
            mass[b, hq] = e[drop].sum() / e.sum()
    return bound, mass


@pytest.mark.parametrize("preset", [0, 3])
def test_sparse_v_bound(orc, preset):
    """orc_sparse_v_bound against its definition written with numpy; tau = 0
    drops nothing; tau just above 1 drops every row, so the bound is the
    weighted mean of |v|, which is >= |o| of the dense attention."""
    rng = np.random.default_rng(4400 + preset)
    seq_lens, Hk, bs = [40, 17], 2, 16
    cache, bt, s, c32 = _cache(orc, preset, seq_lens, Hk, bs, rng, scale_k=3.0)
    q = rng.normal(size=(2, 4, 128)).astype(np.float32)
    for tau in (1e-3, 0.05):
        bd, ms = orc.sparse_v_bound(preset, q, cache, bt, np.array(seq_lens, np.int32), Hk, bs, s,
                                    c32, tau)
        rb, rm = _numpy_sparse_bound(orc, preset, q, cache, bt, seq_lens, Hk, bs, s, c32, tau)
        assert np.allclose(bd, rb, rtol=1e-9, atol=1e-12) and np.allclose(ms, rm, rtol=1e-9, atol=1e-12)
        assert ms.max() > 0                              # keys scaled x3: some rows below tau
    bd, ms = orc.sparse_v_bound(preset, q, cache, bt, np.array(seq_lens, np.int32), Hk, bs, s, c32, 0.0)
    assert not bd.any() and not ms.any()
    bd, ms = orc.sparse_v_bound(preset, q, cache, bt, np.array(seq_lens, np.int32), Hk, bs, s, c32,
                                1.0 + 1e-12)
    out, _ = orc.decode_dense(preset, q, cache, bt, np.array(seq_lens, np.int32), Hk, bs, s, c32)
    assert np.allclose(ms, 1.0) and np.all(bd >= np.abs(out) - 1e-12)
