"""Seeded randomized parity sweep of decode attention.

Each case draws at random:
- the preset;
- the kv-head count and the group size (1-16 query heads per kv head);
- the block size;
- ragged sequence lengths (empty ones and multiples of the 32-token tile
  included);
- the split count (the library's pick or a fixed one);
- the query dtype;
- the block convention (AoS or SoA);
- a sparse-V threshold (mostly 0).

The GPU runs through the C ABI on a cache the oracle built, and its fp32
output and LSE must meet the decode tolerances against the oracle's dense
attention. With a sparse-V threshold, the output must instead stay within
the oracle's bound of the dense attention plus the dense tolerance, with
the dense LSE. The seed fixes the cases, so a failure names a case that
reproduces.
"""
import numpy as np
import pytest
import torch

import quantized_kv_cache_04_gb300 as tq
from _helpers import LSE_ABS, OUT_MAX_ABS, aos_to_soa, check_decode, paged_problem, to_f32

pytestmark = pytest.mark.gpu

N_CASES = 256
MAX_SLOTS = 12000          # tokens x kv heads per case (the oracle's store is the slow part)


def _draw(i):
    rng = np.random.default_rng(77000 + i)
    preset = int(rng.integers(0, 5))
    Hk = int(rng.choice([1, 2, 3, 4, 6, 8, 12]))
    G = int(rng.integers(1, 17))
    bs = int(rng.choice([16, 32, 64, 128]))
    B = int(rng.integers(1, 5))
    cap = max(1, MAX_SLOTS // (Hk * B))
    kind = rng.integers(0, 4, size=B)
    lens = []
    for k in kind:
        if k == 0:
            lens.append(0 if rng.random() < 0.5 else int(rng.integers(1, 8)))
        elif k == 1:
            lens.append(32 * int(rng.integers(1, max(2, cap // 32))))
        else:
            lens.append(int(rng.integers(1, cap + 1)))
    lens = [min(n, cap) for n in lens]
    splits = 0 if rng.random() < 0.5 else int(rng.integers(1, 49))
    qdtype = torch.float16 if rng.random() < 0.5 else torch.bfloat16
    soa = bool(rng.random() < 0.25)
    tau = 1e-3 if rng.random() < 0.15 else 0.0
    return dict(preset=preset, Hk=Hk, G=G, bs=bs, lens=lens, splits=splits, qdtype=qdtype, soa=soa,
                tau=tau, rng=rng)


def _decode(preset, q, cache_np, bt, seq_lens, Hk, bs, signs, c32, num_splits, v_threshold):
    dev = torch.device("cuda")
    B, Hq, D = q.shape
    cache = torch.from_numpy(cache_np).to(dev)
    btd = torch.from_numpy(np.ascontiguousarray(bt)).to(dev)
    sl = torch.from_numpy(np.asarray(seq_lens, np.int32)).to(dev)
    L = tq.tq_get_layout(preset & 0xFF)
    sg = torch.from_numpy(signs).to(dev)
    cc = torch.from_numpy(c32).to(dev) if not L["key_fp8"] else None
    maxlen = int(max(seq_lens))
    S = num_splits or tq.tq_decode_pick_splits(preset, D, B, Hq, Hk, maxlen)
    ws = torch.empty(max(16, tq.tq_decode_workspace_bytes(B, Hq, S, D)), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    tq.decode_attention(preset, q.to(dev).contiguous(), cache, btd, sl, maxlen, Hk, bs, sg, cc,
                        out, lse, ws, num_splits=S, v_threshold=v_threshold)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("i", range(N_CASES))
def test_decode_random_case(orc, i):
    c = _draw(i)
    preset, Hk, G, bs, lens, rng = c["preset"], c["Hk"], c["G"], c["bs"], c["lens"], c["rng"]
    what = (f"case {i}: preset {preset} Hk {Hk} G {G} bs {bs} lens {lens} splits {c['splits']} "
            f"{c['qdtype']} {'soa' if c['soa'] else 'aos'} tau {c['tau']} "
            f"kind {tq.tq_decode_kernel_kind(preset, 128, G * Hk, Hk)}")
    pb = paged_problem(orc, preset, lens, Hk, bs, rng, kscale=2.0 if c["tau"] > 0 else 1.0,
                       dtype="bfloat16" if c["qdtype"] == torch.bfloat16 else "float16")
    q = torch.from_numpy(rng.normal(size=(len(lens), G * Hk, 128)) * 1.5).to(c["qdtype"])
    sl = np.asarray(lens, np.int32)
    ref_o, ref_l = orc.decode_dense(preset, to_f32(q), pb["cache"], pb["bt"], sl, Hk, bs,
                                    pb["signs"], pb["c32"])
    cache = aos_to_soa(orc, preset, pb["cache"]) if c["soa"] else pb["cache"]
    p = preset | (tq.TQ_LAYOUT_SOA if c["soa"] else 0)
    o, l = _decode(p, q, cache, pb["bt"], lens, Hk, bs, pb["signs"], pb["c32"], c["splits"], c["tau"])
    if c["tau"] == 0.0:
        check_decode(o, l, ref_o, ref_l, what)
        return
    bound, _ = orc.sparse_v_bound(preset, to_f32(q), pb["cache"], pb["bt"], sl, Hk, bs,
                                  pb["signs"], pb["c32"], c["tau"])
    assert np.all(np.isfinite(o)), what
    err = np.abs(o.astype(np.float64) - ref_o)
    assert np.all(err <= bound + OUT_MAX_ABS), f"{what}: {(err - bound).max()}"
    ninf = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(l), ninf), what
    if (~ninf).any():
        assert np.abs(l[~ninf] - ref_l[~ninf]).max() <= LSE_ABS, what
