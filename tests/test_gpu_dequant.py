"""GPU dequantisation (tq_dequant) against the oracle's per-slot dequantisation.

The oracle restates the inverse of the store in fp64: k = k_norm * s . (H c[idx])
with the explicit Sylvester matrix (FP8 keys decoded as they are) and
v = code * v_scale + v_zero.  Bars:
  - values: bit-exact in fp32 (code * scale is exact in fp32 and the single
    rounding of + zero is the fp32 rounding of the exact value); within one
    ulp of the output type for fp16 / bf16 (the GPU rounds its fp32 result);
  - keys: fp32 max-abs error <= 4e-6 * ||k||_2 per row: the fast transform in
    fp32 takes 7 butterfly levels, each adding at most 2^-24 relative error
    of its operands, about 4.2e-7 ||k|| in all (10x margin); fp16 / bf16
    outputs within one ulp of the output type on top of that;
  - padding slots (negative, or past the cache) give zero rows.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import quantized_kv_cache_04_gb300 as tq
from _helpers import paged_problem, to_f32

pytestmark = pytest.mark.gpu

K_REL = 4e-6


def _ulp(x, dtype):
    """One ulp of the output type at |x| (normal range; subnormals use the minimum)."""
    x = np.abs(np.asarray(x, np.float64))
    mant, emin = {torch.float16: (10, -14), torch.bfloat16: (7, -126)}[dtype]
    e = np.floor(np.log2(np.maximum(x, 2.0 ** emin)))
    return 2.0 ** (e - mant)


def _gpu_dequant(preset, cache_np, slots, Hk, bs, signs, c32, out_dtype):
    dev = torch.device("cuda")
    L = tq.tq_get_layout(preset)
    cache = torch.from_numpy(cache_np).to(dev)
    sm = torch.from_numpy(np.asarray(slots, np.int64)).to(dev)
    sg = torch.from_numpy(signs).to(dev)
    cc = torch.from_numpy(c32).to(dev) if not L["key_fp8"] else None
    N = len(slots)
    k = torch.full((N, Hk, 128), float("nan"), dtype=out_dtype, device=dev)
    v = torch.full((N, Hk, 128), float("nan"), dtype=out_dtype, device=dev)
    tq.dequant(preset, sm, cache, Hk, bs, sg, cc, k, v)
    torch.cuda.synchronize()
    return to_f32(k), to_f32(v)


def _check_rows(orc, preset, cache_np, slots, Hk, bs, signs, c32, k, v, out_dtype, rows=None):
    L = orc.layout(preset)
    S = L["slot_size_aligned"]
    flat = cache_np.reshape(-1, S)
    nslots = cache_np.shape[0] * bs
    idx = range(len(slots)) if rows is None else rows
    for n in idx:
        sl = int(slots[n])
        for h in range(Hk):
            if sl < 0 or sl >= nslots:
                assert not k[n, h].any() and not v[n, h].any(), f"padding row {n} not zero"
                continue
            kh, vh = orc.dequant_slot(preset, flat[sl * Hk + h], signs, c32)
            kerr = np.abs(k[n, h].astype(np.float64) - kh)
            bound = K_REL * np.linalg.norm(kh) + 1e-30
            if out_dtype == torch.float32:
                assert kerr.max() <= bound, f"row {n} head {h}: key error {kerr.max()} > {bound}"
                assert np.array_equal(v[n, h], vh.astype(np.float32)), f"row {n} head {h}: values"
            else:
                assert np.all(kerr <= bound + _ulp(kh, out_dtype)), f"row {n} head {h}: key"
                verr = np.abs(v[n, h].astype(np.float64) - vh)
                assert np.all(verr <= _ulp(vh, out_dtype)), f"row {n} head {h}: values"


@pytest.mark.parametrize("preset", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("Hk,bs", [(1, 16), (8, 64), (3, 32)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_dequant_on_oracle_cache(orc, preset, Hk, bs, out_dtype):
    rng = np.random.default_rng(7000 + 100 * preset + 10 * Hk + bs)
    seq_lens = [37, 100]
    pb = paged_problem(orc, preset, seq_lens, Hk, bs, rng)
    slots = []
    for b, n in enumerate(seq_lens):
        t = np.arange(n)
        slots.append(pb["bt"][b, t // bs].astype(np.int64) * bs + t % bs)
    slots = np.concatenate(slots)
    rng.shuffle(slots)
    nslots = pb["cache"].shape[0] * bs
    slots = np.concatenate([slots[:50], [-1], slots[50:], [nslots, nslots + 7, -5]])
    k, v = _gpu_dequant(preset, pb["cache"], slots, Hk, bs, pb["signs"], pb["c32"], out_dtype)
    _check_rows(orc, preset, pb["cache"], slots, Hk, bs, pb["signs"], pb["c32"], k, v, out_dtype)


@pytest.mark.parametrize("preset", [0, 1, 2, 3, 4])
def test_dequant_inverts_store_up_to_quantisation(orc, preset):
    """A property that holds at any size: FP8 keys come back within E4M3
    rounding of the stored bf16-exact inputs; MSE keys keep the input norm
    within fp16 rounding (matched norm); values within half a quantisation
    step (plus fp16 rounding of scale and zero)."""
    dev = torch.device("cuda")
    rng = np.random.default_rng(8100 + preset)
    N, Hk, bs = 300, 8, 16
    L = tq.tq_get_layout(preset)
    K = torch.from_numpy(rng.normal(size=(N, Hk, 128))).to(torch.float16).to(dev)
    V = torch.from_numpy(rng.normal(size=(N, Hk, 128))).to(torch.float16).to(dev)
    c = tq.TQCache(preset, (N + bs - 1) // bs, bs, Hk, device=dev)
    sm = torch.arange(N, dtype=torch.int64, device=dev)
    c.store(K, V, sm)
    ko = torch.empty((N, Hk, 128), dtype=torch.float32, device=dev)
    vo = torch.empty_like(ko)
    c.dequant(sm, ko, vo)
    torch.cuda.synchronize()
    k, v, k0, v0 = to_f32(ko), to_f32(vo), to_f32(K), to_f32(V)
    if L["key_fp8"]:
        assert np.all(np.abs(k - k0) <= np.abs(k0) * 2.0 ** -4 + 2.0 ** -10)
    else:
        nk, n0 = np.linalg.norm(k, axis=-1), np.linalg.norm(k0, axis=-1)
        assert np.all(np.abs(nk - n0) <= n0 * 2.0 ** -10)
    # |v - v0| <= scale/2 when scale and zero are exact; their fp16 rounding
    # adds up to (2^b - 1) half-ulps of the scale and half an ulp of the zero
    lv = 2 ** L["value_bits"] - 1
    step = (v0.max(-1) - v0.min(-1)) / lv
    bound = (0.5 * step + lv * 0.5 * _ulp(step, torch.float16)
             + 0.5 * _ulp(v0.min(-1), torch.float16) + 1e-6)
    assert np.all(np.abs(v - v0) <= bound[..., None])


def test_dequant_full_size_sampled(orc):
    """Llama-3-8B-shaped cache (32 x 8192 tokens, 8 kv heads, k8v4 and
    3bit_nc) written by the GPU store, dequantised whole (fp16 out); sampled
    rows are checked against the oracle's dequantisation of the same slot
    bytes."""
    from quantized_kv_cache_04_gb300 import workloads as wl
    dev = torch.device("cuda")
    for preset_name in ("turboquant_k8v4", "turboquant_3bit_nc"):
        w = wl.make("llama3_8b", preset=preset_name)
        c = tq.TQCache(w.preset, w.num_blocks, w.block_size, w.Hk, device=dev)
        sms = []
        for b in range(w.B):
            n = int(w.seq_lens[b])
            K, V = wl.gen_kv(w, b, 0, n, dev)
            sm = torch.from_numpy(w.slot_mapping(b, np.arange(n))).to(dev)
            c.store(K, V, sm)
            sms.append(sm)
        sm = torch.cat(sms)
        N = sm.numel()
        ko = torch.empty((N, w.Hk, 128), dtype=torch.float16, device=dev)
        vo = torch.empty_like(ko)
        c.dequant(sm, ko, vo)
        torch.cuda.synchronize()
        rng = np.random.default_rng(8200)
        rows = np.sort(rng.choice(N, 64, replace=False))
        cache_np = c.cache.cpu().numpy()
        signs = c.signs.cpu().numpy()
        c32 = c.centroids.cpu().numpy() if c.centroids is not None else np.zeros(1, np.float32)
        k = to_f32(ko[torch.from_numpy(rows).to(dev)])
        v = to_f32(vo[torch.from_numpy(rows).to(dev)])
        slots = sm.cpu().numpy()[rows]
        _check_rows(orc, w.preset_id, cache_np, slots, w.Hk, w.block_size, signs, c32, k, v,
                    torch.float16, rows=range(len(rows)))
        del c, ko, vo
        torch.cuda.empty_cache()


@pytest.mark.parametrize("preset", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("Hk,bs", [(8, 16), (3, 64)])
def test_dequant_soa_cache(orc, preset, Hk, bs):
    """Dequantisation of a cache in the SoA block convention equals the
    oracle's dequantisation of the same slots in AoS form."""
    from _helpers import aos_to_soa
    rng = np.random.default_rng(7500 + 10 * preset + Hk)
    seq_lens = [60, 33]
    pb = paged_problem(orc, preset, seq_lens, Hk, bs, rng)
    slots = np.concatenate([pb["bt"][b, np.arange(n) // bs].astype(np.int64) * bs + np.arange(n) % bs
                            for b, n in enumerate(seq_lens)] + [np.array([-1], np.int64)])
    soa = aos_to_soa(orc, preset, pb["cache"])
    k, v = _gpu_dequant(preset | tq.TQ_LAYOUT_SOA, soa, slots, Hk, bs, pb["signs"], pb["c32"],
                        torch.float32)
    _check_rows(orc, preset, pb["cache"], slots, Hk, bs, pb["signs"], pb["c32"], k, v,
                torch.float32)
