"""A cache larger than 2 GiB: byte offsets past 2^31 in the store (slot
index x row bytes), the decode (page x block bytes) and the dequantisation.

Two sequences of 4096 tokens have their pages at the end of a ~2.5 GB cache
(past byte 2^31) and across the 2^31 boundary.  The store writes them in one
call; the slots are checked against the oracle's store of the same inputs
(sampled rows for the Lloyd-Max preset, whose codes may flip at counted
ties), the decode against the oracle's dense attention over its own cache,
and the dequantised rows against the oracle's per-slot dequantisation.
Every block outside the two sequences stays zero, so no offset wrapped.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import quantized_kv_cache_04_gb300 as tq
from quantized_kv_cache_04_gb300 import workloads as wl
from _helpers import check_decode, codebook, compare_store, to_f32, TIE_FRACTION

pytestmark = pytest.mark.gpu

TWO_GIB = 2 ** 31


@pytest.mark.parametrize("preset", ["turboquant_k8v4", "turboquant_k3v4_nc"])
def test_cache_past_two_gib(orc, preset):
    dev = torch.device("cuda")
    pid = wl.PRESET_IDS[preset]
    L = orc.layout(pid)
    Hk, bs, Hq, n = 8, 16, 32, 4096
    S = L["slot_size_aligned"]
    block_bytes = bs * Hk * S
    cross = TWO_GIB // block_bytes                        # the block holding byte 2^31
    num_blocks = int(2.5e9) // block_bytes
    nblk = n // bs
    starts = [num_blocks - nblk - 1, cross - nblk // 2]   # past 2^31, and across it
    assert (starts[0] * block_bytes) > TWO_GIB and starts[1] * block_bytes < TWO_GIB
    bt = np.stack([np.arange(s0, s0 + nblk, dtype=np.int32) for s0 in starts])
    cache = torch.zeros((num_blocks, bs, Hk, S), dtype=torch.uint8, device=dev)
    assert cache.numel() > TWO_GIB + block_bytes * nblk

    w = wl.make("sweep", preset=preset, ctx=n, batch=2)   # value recipe of the Llama shape
    signs = orc.signs(128, 42)
    c32, m32 = codebook(orc, pid)
    sg = torch.from_numpy(signs).to(dev)
    cc = None if L["key_fp8"] else torch.from_numpy(c32).to(dev)
    mm = None if L["key_fp8"] else torch.from_numpy(m32).to(dev)
    Ks, Vs, sms = [], [], []
    for b in range(2):
        K, V = wl.gen_kv(w, b, 0, n, "cpu")
        Ks.append(K)
        Vs.append(V)
        t = np.arange(n)
        sms.append(bt[b, t // bs].astype(np.int64) * bs + t % bs)
    K, V = torch.cat(Ks), torch.cat(Vs)
    sm = np.concatenate(sms)
    assert sm.max() * Hk * S > TWO_GIB
    tq.store(pid, K.to(dev), V.to(dev), torch.from_numpy(sm).to(dev), cache, bs, sg, cc, mm)
    torch.cuda.synchronize()

    # nothing outside the two sequences' blocks was written
    inside = sum(int(torch.count_nonzero(cache[s0:s0 + nblk])) for s0 in starts)
    assert inside > 0 and int(torch.count_nonzero(cache)) == inside

    # the slots against the oracle's store of the same inputs
    flat = cache.view(-1, Hk, S)
    rng = np.random.default_rng(31)
    pick = rng.choice(2 * n * Hk, 512, replace=False)
    tok, head = pick // Hk, pick % Hk
    rows = flat[torch.from_numpy(sm[tok]).to(dev), torch.from_numpy(head).to(dev)].cpu().numpy()
    flips, codes = compare_store(orc, pid, rows, to_f32(K)[tok, head], to_f32(V)[tok, head],
                                 signs, c32, m32)
    assert flips <= max(1, int(np.ceil(TIE_FRACTION * codes))), (flips, codes)

    # decode over the large cache against the oracle's own cache of the same tokens
    q = wl.gen_q(w, "cpu")
    out = torch.empty((2, Hq, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((2, Hq), dtype=torch.float32, device=dev)
    S_ = tq.tq_decode_pick_splits(pid, 128, 2, Hq, Hk, n)
    ws = torch.empty(tq.tq_decode_workspace_bytes(2, Hq, S_, 128), dtype=torch.uint8, device=dev)
    tq.decode_attention(pid, q.to(dev), cache, torch.from_numpy(bt).to(dev),
                        torch.full((2,), n, dtype=torch.int32, device=dev), n, Hk, bs, sg, cc,
                        out, lse, ws, num_splits=S_)
    torch.cuda.synchronize()
    for b in range(2):
        cache_o = np.zeros((nblk, bs, Hk, S), np.uint8)
        orc.store(pid, to_f32(K[b * n:(b + 1) * n]), to_f32(V[b * n:(b + 1) * n]),
                  np.arange(n, dtype=np.int64), cache_o, bs, signs, c32, m32)
        ref_o, ref_l = orc.decode_dense(pid, to_f32(q[b:b + 1]), cache_o,
                                        np.arange(nblk, dtype=np.int32)[None, :],
                                        np.array([n], np.int32), Hk, bs, signs, c32)
        check_decode(to_f32(out[b:b + 1]), to_f32(lse[b:b + 1]), ref_o, ref_l, f"sequence {b}")

    # dequantisation of sampled slots past 2^31 against the oracle's, from the GPU's own bytes
    sel = np.sort(rng.choice(2 * n, 64, replace=False))
    ko = torch.empty((sel.size, Hk, 128), dtype=torch.float32, device=dev)
    vo = torch.empty_like(ko)
    tq.dequant(pid, torch.from_numpy(sm[sel]).to(dev), cache, Hk, bs, sg, cc, ko, vo)
    torch.cuda.synchronize()
    kg, vg = to_f32(ko), to_f32(vo)
    for i, t in enumerate(sel):
        for h in (0, Hk - 1):
            slot = flat[int(sm[t]), h].cpu().numpy()
            kh, vh = orc.dequant_slot(pid, slot, signs, c32)
            assert np.abs(kg[i, h] - kh).max() <= 4e-6 * np.linalg.norm(kh) + 1e-30
            assert np.array_equal(vg[i, h], vh.astype(np.float32))
