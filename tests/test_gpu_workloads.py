"""Full-size parity at the workload configurations, in the launch
configuration the benchmark times (bench.Problem: the same cache shape,
paging, block tables, sequence lengths, split count and step).

The whole batch runs on the GPU.  A few sampled sequences get their K/V (and
the step's new token) from the seeded generators run on the CPU and uploaded,
so that the oracle can build its own cache for them from the same values:
the oracle stores the first and the last kv head of those sequences and
decodes the query heads of those kv heads (dense attention over its
dequantised cache), and the GPU's output rows and LSEs for them must meet the
decode tolerances.  The other sequences keep the benchmark's device-generated
inputs.  The store configuration (16,384 new tokens of 16 sequences) is
checked slot by slot on sampled (token, kv head) pairs against the oracle's
store of the same inputs, and the decode over its cache like the others.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import quantized_kv_cache_04_gb300 as tq
from quantized_kv_cache_04_gb300 import workloads as wl
from _helpers import check_decode, codebook, compare_store, TIE_FRACTION, to_f32

pytestmark = pytest.mark.gpu

CHUNK = 32768


def _sampled(w):
    """Sequences checked against the oracle: the shortest and the longest
    (the first and the last when all have the same length)."""
    order = np.argsort(w.seq_lens, kind="stable")
    return sorted({int(order[0]), int(order[-1])})


DECODE_CASES = [("tiny", None), ("llama3_8b", None), ("qwen3_32b", None), ("long", None)] + [
    ("store_mixed", p) for p in ("turboquant_k8v4", "turboquant_4bit_nc", "turboquant_k3v4_nc",
                                 "turboquant_3bit_nc", "turboquant_2bit_nc")]


@pytest.mark.parametrize("name,preset", DECODE_CASES)
def test_decode_full_size_sampled(orc, name, preset):
    """Every decode workload, and the decode (32 query heads) over the mixed
    16-sequence cache of the store workload in every preset."""
    import bench
    dev = torch.device("cuda")
    w = wl.make(name, preset=preset)
    p = bench.Problem(w, dev, None)
    L = orc.layout(w.preset_id)
    signs = orc.signs(128, 42)
    c32, m32 = codebook(orc, w.preset_id)
    # the library's rotation signs and codebook are the oracle's
    assert np.array_equal(p.c.signs.cpu().numpy(), signs)
    if not L["key_fp8"]:
        assert np.array_equal(p.c.centroids.cpu().numpy(), c32)

    q_cpu = wl.gen_q(w, "cpu")
    p.q.copy_(q_cpu.to(dev))
    samples = _sampled(w)
    G = w.Hq // w.Hk
    kv = sorted({0, w.Hk - 1})                          # sampled kv heads
    qh = np.concatenate([np.arange(h * G, (h + 1) * G) for h in kv])
    oracle = {}
    for b in samples:
        n = int(w.seq_lens[b])
        nblk = (n + w.block_size - 1) // w.block_size
        cache_o = np.zeros((nblk, w.block_size, len(kv), L["slot_size_aligned"]), np.uint8)
        for t0 in range(0, n, CHUNK):
            t1 = min(n, t0 + CHUNK)
            K, V = wl.gen_kv(w, b, t0, t1, "cpu")
            sm = torch.from_numpy(w.slot_mapping(b, np.arange(t0, t1))).to(dev)
            p.c.store(K.to(dev), V.to(dev), sm)
            orc.store(w.preset_id, to_f32(K[:, kv]), to_f32(V[:, kv]),
                      np.arange(t0, t1, dtype=np.int64), cache_o, w.block_size, signs, c32, m32)
        Kn, Vn = wl.gen_kv(w, b, n - 1, n, "cpu")       # the step's new token
        p.new_k[b].copy_(Kn[0].to(dev))
        p.new_v[b].copy_(Vn[0].to(dev))
        bt_o = np.arange(nblk, dtype=np.int32)[None, :]
        oracle[b] = orc.decode_dense(w.preset_id, to_f32(q_cpu[b:b + 1, qh]), cache_o, bt_o,
                                     np.array([n], np.int32), len(kv), w.block_size, signs, c32)

    # one benchmark step (store of the new tokens + decode), then the same
    # decode with an fp32 output
    p.store()
    p.decode()
    out32 = torch.empty(p.out.shape, dtype=torch.float32, device=dev)
    lse32 = torch.empty_like(p.lse)
    p.c.decode(p.q, p.bt, p.sl, p.max_len, out32, lse32, p.ws, num_splits=p.S)
    torch.cuda.synchronize()
    o32, l32 = to_f32(out32), to_f32(lse32)
    o_b, l_b = to_f32(p.out), to_f32(p.lse)
    assert np.array_equal(l_b, l32)
    for b in samples:
        ref_o, ref_l = oracle[b]
        check_decode(o32[b:b + 1, qh], l32[b:b + 1, qh], ref_o, ref_l, f"{name} sequence {b}")
        # the benchmark's own output (query dtype): the fp32 result rounded once
        r16 = torch.from_numpy(o32[b]).to(p.out.dtype).float().numpy()
        assert np.array_equal(o_b[b], r16), f"{name} sequence {b}: output rounding"
    assert np.all(np.isfinite(o32)) and np.all(np.isfinite(l32))


@pytest.mark.parametrize("preset", ["turboquant_k8v4", "turboquant_4bit_nc", "turboquant_k3v4_nc",
                                    "turboquant_3bit_nc", "turboquant_2bit_nc"])
def test_store_mixed_full_size_sampled(orc, preset):
    """The chunked-prefill store (16,384 tokens of 16 sequences, bs 32, 8 kv
    heads) in one call, as the benchmark's store run issues it; 256 sampled
    (token, kv head) slots against the oracle's store of the same inputs."""
    dev = torch.device("cuda")
    w = wl.make("store_mixed", preset=preset)
    c = tq.TQCache(w.preset_id, w.num_blocks, w.block_size, w.Hk, device=dev)
    Ks, Vs, sms = [], [], []
    for b in range(w.B):
        n = int(w.seq_lens[b])
        K, V = wl.gen_kv(w, b, 0, n, "cpu")
        Ks.append(K)
        Vs.append(V)
        sms.append(w.slot_mapping(b, np.arange(n)))
    K, V = torch.cat(Ks), torch.cat(Vs)
    sm = np.concatenate(sms).astype(np.int64)
    c.store(K.to(dev), V.to(dev), torch.from_numpy(sm).to(dev))
    torch.cuda.synchronize()
    cache = c.cache.cpu().numpy()
    S = cache.shape[-1]
    rng = np.random.default_rng(9300)
    pick = rng.choice(K.shape[0] * w.Hk, 256, replace=False)
    tok, head = pick // w.Hk, pick % w.Hk
    flat = cache.reshape(-1, w.Hk, S)
    rows = flat[sm[tok], head]
    kf = to_f32(K)[tok, head]
    vf = to_f32(V)[tok, head]
    signs = orc.signs(128, 42)
    c32, m32 = codebook(orc, w.preset_id)
    flips, codes = compare_store(orc, w.preset_id, rows, kf, vf, signs, c32, m32)
    assert flips <= max(1, int(np.ceil(TIE_FRACTION * codes))), (flips, codes)
