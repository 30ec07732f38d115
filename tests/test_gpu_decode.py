"""GPU parity of split-K decode attention (through the C ABI) against the
oracle's dense attention over the oracle's cache, and end to end (GPU store
+ GPU decode against oracle store + oracle decode)."""
import numpy as np
import pytest
import torch

import quantized_kv_cache_04_gb300 as tq
from _helpers import (LSE_ABS, OUT_MAX_ABS, check_decode, codebook, expected_kernel_kind, paged_problem,
                      to_f32)

pytestmark = pytest.mark.gpu
PRESETS = [0, 1, 2, 3, 4]


def _gpu_decode(preset, q, cache_np, bt, seq_lens, Hk, bs, signs, c32, num_splits=0,
                out_dtype=torch.float32, cache_dev=None, v_threshold=0.0):
    dev = torch.device("cuda")
    B, Hq, D = q.shape
    cache = cache_dev if cache_dev is not None else torch.from_numpy(cache_np).to(dev)
    btd = torch.from_numpy(np.ascontiguousarray(bt)).to(dev)
    sl = torch.from_numpy(np.asarray(seq_lens, np.int32)).to(dev)
    L = tq.tq_get_layout(preset)
    sg = torch.from_numpy(signs).to(dev)
    cc = torch.from_numpy(c32).to(dev) if not L["key_fp8"] else None
    maxlen = int(max(seq_lens)) if len(seq_lens) else 0
    S = num_splits or tq.tq_decode_pick_splits(preset, D, B, Hq, Hk, maxlen)
    ws = torch.empty(max(16, tq.tq_decode_workspace_bytes(B, Hq, S, D)), dtype=torch.uint8,
                     device=dev)
    out = torch.empty((B, Hq, D), dtype=out_dtype, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    tq.decode_attention(preset, q.to(dev).contiguous(), cache, btd, sl, maxlen, Hk, bs, sg, cc,
                        out, lse, ws, num_splits=num_splits, v_threshold=v_threshold)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


CASES = [  # (G, Hk, bs, seq_lens, splits): CUDA-core and tensor-core stage 1 shapes
    (4, 2, 16, [512], 0),
    (8, 2, 64, [1000, 1, 0, 130], 7),
    (1, 4, 32, [65, 300], 1),
    (16, 1, 128, [1500], 64),
    (6, 2, 16, [33, 200], 3),
    (4, 8, 32, [17, 0, 256, 97, 5], 0),
    (8, 8, 64, [700, 65, 1], 3),
    (4, 8, 16, [1024, 31], 0),
    (1, 8, 32, [129, 16], 2),
    (2, 8, 128, [1000], 64),
    (6, 8, 16, [250, 0], 5),
    (5, 16, 32, [90, 333], 0),
    (16, 8, 16, [200], 2),
    (2, 1, 32, [300, 45], 0),
    (4, 3, 16, [77, 400], 0),
    (4, 8, 16, [16500, 200], 0),   # a 16K-token sequence next to a short one
    (3, 3, 32, [700, 33], 5),      # 3 kv heads: Lloyd-Max rows of 2 mod 4 bytes (CUDA cores)
]


def _expected_kind(preset, G, Hk):
    return expected_kernel_kind(preset, G, Hk)


@pytest.mark.parametrize("preset", PRESETS)
@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("qdtype", [torch.float16, torch.bfloat16])
def test_decode_on_oracle_cache(orc, preset, case, qdtype):
    G, Hk, bs, seq_lens, S = CASES[case]
    assert tq.tq_decode_kernel_kind(preset, 128, G * Hk, Hk) == _expected_kind(preset, G, Hk)
    rng = np.random.default_rng(1000 * preset + 10 * case + (qdtype == torch.bfloat16))
    pb = paged_problem(orc, preset, seq_lens, Hk, bs, rng,
                       dtype="bfloat16" if qdtype == torch.bfloat16 else "float16")
    B = len(seq_lens)
    q = torch.from_numpy(rng.normal(size=(B, G * Hk, 128)) * 1.5).to(qdtype)
    ref_o, ref_l = orc.decode_dense(preset, to_f32(q), pb["cache"], pb["bt"],
                                    np.asarray(seq_lens, np.int32), Hk, bs, pb["signs"],
                                    pb["c32"])
    o, l = _gpu_decode(preset, q, pb["cache"], pb["bt"], seq_lens, Hk, bs, pb["signs"],
                       pb["c32"], S)
    check_decode(o, l, ref_o, ref_l, f"preset {preset} case {case}")
    # output in the query dtype: within one ulp of the exact result rounded once
    # (plus the fp32 path's own error, far below the 2e-3 bar, for tiny values)
    o16, _ = _gpu_decode(preset, q, pb["cache"], pb["bt"], seq_lens, Hk, bs, pb["signs"],
                         pb["c32"], S, out_dtype=qdtype)
    ref16 = torch.from_numpy(ref_o).to(qdtype).float().numpy()
    eps = 2.0 ** -10 if qdtype == torch.float16 else 2.0 ** -7
    ulp = eps * np.maximum(2.0 ** np.floor(np.log2(np.maximum(np.abs(ref16), 2.0 ** -14))),
                           2.0 ** -14)
    assert np.all(np.abs(o16 - ref16) <= ulp * 1.0001 + 2e-5)


@pytest.mark.parametrize("preset", [1, 2, 3, 4])
@pytest.mark.parametrize("G,Hk,bs,seq_lens", [(4, 8, 16, [300, 77]), (8, 8, 64, [400]),
                                              (4, 2, 32, [129])])
def test_decode_custom_codebook(orc, preset, G, Hk, bs, seq_lens):
    """A codebook other than the library's Lloyd-Max one (entries moved by up
    to 2%, no longer symmetric): the decode picks its own centroid scale for
    the fp16 + E4M3 score split and still meets the tolerances."""
    L = orc.layout(preset)
    rng = np.random.default_rng(4200 + 10 * preset + G)
    c, _ = codebook(orc, preset)
    c = np.sort(c.astype(np.float64) * (1.0 + 0.02 * rng.uniform(-1, 1, c.shape))).astype(np.float32)
    m = ((c[1:].astype(np.float64) + c[:-1]) / 2).astype(np.float32)
    pb = paged_problem(orc, preset, seq_lens, Hk, bs, rng, book=(c, m))
    q = torch.from_numpy(rng.normal(size=(len(seq_lens), G * Hk, 128)) * 2.0).to(torch.float16)
    ref_o, ref_l = orc.decode_dense(preset, to_f32(q), pb["cache"], pb["bt"],
                                    np.asarray(seq_lens, np.int32), Hk, bs, pb["signs"], c)
    o, l = _gpu_decode(preset, q, pb["cache"], pb["bt"], seq_lens, Hk, bs, pb["signs"], c)
    check_decode(o, l, ref_o, ref_l, f"preset {preset} custom codebook")


@pytest.mark.parametrize("preset", [0, 2])
@pytest.mark.parametrize("B", [512, 520])
def test_decode_large_varlen_batch(orc, preset, B):
    """Many short sequences of mixed lengths (0..70 tokens): CTA rows take
    the sequences longest first up to 512 sequences and in index order
    beyond; both give the oracle's result."""
    rng = np.random.default_rng(9700 + B + preset)
    Hk, G, bs = 8, 4, 16
    seq_lens = rng.integers(0, 71, size=B)
    pb = paged_problem(orc, preset, seq_lens, Hk, bs, rng)
    q = torch.from_numpy(rng.normal(size=(B, G * Hk, 128))).to(torch.float16)
    ref_o, ref_l = orc.decode_dense(preset, to_f32(q), pb["cache"], pb["bt"],
                                    np.asarray(seq_lens, np.int32), Hk, bs, pb["signs"], pb["c32"])
    o, l = _gpu_decode(preset, q, pb["cache"], pb["bt"], seq_lens, Hk, bs, pb["signs"], pb["c32"], 3)
    check_decode(o, l, ref_o, ref_l, f"preset {preset} B {B}")


@pytest.mark.parametrize("preset", PRESETS)
def test_split_count_invariance(orc, preset):
    """Results do not depend on the split count beyond rounding."""
    rng = np.random.default_rng(77 + preset)
    seq_lens, Hk, bs = [3000, 45], 2, 32
    pb = paged_problem(orc, preset, seq_lens, Hk, bs, rng)
    q = torch.from_numpy(rng.normal(size=(2, 8, 128))).to(torch.float16)
    base = _gpu_decode(preset, q, pb["cache"], pb["bt"], seq_lens, Hk, bs, pb["signs"], pb["c32"], 1)
    for S in (2, 5, 64, 256):
        o, l = _gpu_decode(preset, q, pb["cache"], pb["bt"], seq_lens, Hk, bs, pb["signs"],
                           pb["c32"], S)
        assert np.max(np.abs(o - base[0])) < 1e-4
        assert np.max(np.abs(l - base[1])) < 1e-5


@pytest.mark.parametrize("preset", PRESETS)
def test_end_to_end_store_then_decode(orc, preset):
    """GPU store + GPU decode against oracle store + oracle decode."""
    rng = np.random.default_rng(500 + preset)
    seq_lens, Hk, G, bs = [700, 33, 1], 4, 4, 16
    dev = torch.device("cuda")
    pb = paged_problem(orc, preset, seq_lens, Hk, bs, rng)   # oracle cache + inputs
    L = tq.tq_get_layout(preset)
    cache = torch.zeros(pb["cache"].shape, dtype=torch.uint8, device=dev)
    cache[pb["guard"]] = 0xFF
    sg = torch.from_numpy(pb["signs"]).to(dev)
    cc = torch.from_numpy(pb["c32"]).to(dev) if not L["key_fp8"] else None
    mm = torch.from_numpy(pb["m32"]).to(dev) if not L["key_fp8"] else None
    for b, n in enumerate(seq_lens):
        t = np.arange(n)
        sm = torch.from_numpy(pb["bt"][b, t // bs].astype(np.int64) * bs + t % bs).to(dev)
        tq.store(preset, pb["K"][b].to(dev), pb["V"][b].to(dev), sm, cache, bs, sg, cc, mm)
    q = torch.from_numpy(rng.normal(size=(len(seq_lens), G * Hk, 128))).to(torch.float16)
    ref_o, ref_l = orc.decode_dense(preset, to_f32(q), pb["cache"], pb["bt"],
                                    np.asarray(seq_lens, np.int32), Hk, bs, pb["signs"], pb["c32"])
    o, l = _gpu_decode(preset, q, None, pb["bt"], seq_lens, Hk, bs, pb["signs"], pb["c32"],
                       cache_dev=cache)
    check_decode(o, l, ref_o, ref_l, f"e2e preset {preset}")


@pytest.mark.parametrize("preset,Hk", [(3, 2), (3, 8), (2, 8), (0, 8)])
def test_planted_key_peaked_softmax(orc, preset, Hk):
    """A key aligned with the query (logit ~ 12) dominates each split: the
    LSE merge of peaked partials stays within 1e-4 (this is where fp16
    rounding of centroids or q alone would miss the bar)."""
    rng = np.random.default_rng(4 + preset + Hk)
    G, bs, n = 4, 128, 8192 if Hk == 2 else 4096
    pb = paged_problem(orc, preset, [n], Hk, bs, rng, dtype="bfloat16")
    q = torch.from_numpy(rng.normal(size=(1, G * Hk, 128)) * 1.2).to(torch.bfloat16)
    # plant keys aligned with head-0 queries every 1024 tokens, re-store with the oracle
    K = pb["K"][0].clone()
    for t in range(512, n, 1024):
        for h in range(Hk):
            d = to_f32(q[0, h * G]).astype(np.float64)
            K[t, h] = torch.from_numpy(1.1 * np.sqrt(128) * d / np.linalg.norm(d)).to(torch.bfloat16)
    tt = np.arange(n)
    sm = pb["bt"][0, tt // bs].astype(np.int64) * bs + tt % bs
    orc.store(preset, to_f32(K), to_f32(pb["V"][0]), sm, pb["cache"], bs, pb["signs"],
              pb["c32"], pb["m32"])
    ref_o, ref_l = orc.decode_dense(preset, to_f32(q), pb["cache"], pb["bt"],
                                    np.array([n], np.int32), Hk, bs, pb["signs"], pb["c32"])
    assert ref_l.max() > 8
    for S in (1, 8, 64):
        o, l = _gpu_decode(preset, q, pb["cache"], pb["bt"], [n], Hk, bs, pb["signs"], pb["c32"], S)
        check_decode(o, l, ref_o, ref_l, f"planted S={S}")


@pytest.mark.parametrize("preset", PRESETS)
def test_continuation_prefill_as_decode_rows(orc, preset):
    """A continuation chunk of q_len new tokens attends causally to the cached
    prefix by running each query row as a decode request with its own
    sequence length (cached_len + i + 1) over one shared block-table row
    (block_table_stride = 0), the decode-kernel path of the API page's
    `_prefill_attention` for short continuations."""
    rng = np.random.default_rng(900 + preset)
    Hk, G, bs, seq_len, q_len = 8, 4, 32, 700, 13
    cached = seq_len - q_len
    pb = paged_problem(orc, preset, [seq_len], Hk, bs, rng)
    dev = torch.device("cuda")
    L = tq.tq_get_layout(preset)
    seq_lens = np.arange(cached + 1, seq_len + 1, dtype=np.int32)          # causal per row
    q = torch.from_numpy(rng.normal(size=(q_len, G * Hk, 128))).to(torch.float16)
    bt_oracle = np.repeat(pb["bt"][:1], q_len, axis=0)                    # same row for every query
    ref_o, ref_l = orc.decode_dense(preset, to_f32(q), pb["cache"], bt_oracle, seq_lens, Hk, bs,
                                    pb["signs"], pb["c32"])
    cache = torch.from_numpy(pb["cache"]).to(dev)
    bt_row = torch.from_numpy(np.ascontiguousarray(pb["bt"][0])).to(dev)   # one row, stride 0
    sl = torch.from_numpy(seq_lens).to(dev)
    sg = torch.from_numpy(pb["signs"]).to(dev)
    cc = torch.from_numpy(pb["c32"]).to(dev) if not L["key_fp8"] else None
    S = tq.tq_decode_pick_splits(preset, 128, q_len, G * Hk, Hk, seq_len)
    ws = torch.empty(tq.tq_decode_workspace_bytes(q_len, G * Hk, S, 128), dtype=torch.uint8, device=dev)
    out = torch.empty((q_len, G * Hk, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((q_len, G * Hk), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    rc = tq.tq_decode_attention(preset, 128, q_len, G * Hk, Hk, bs, tq.TQ_F16, q.to(dev).data_ptr(),
                                cache.data_ptr(), cache.shape[0], bt_row.data_ptr(), 0, sl.data_ptr(),
                                seq_len, 128 ** -0.5, S, sg.data_ptr(), 0 if cc is None else cc.data_ptr(),
                                out.data_ptr(), tq.TQ_F32, lse.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    assert rc == 0, tq.tq_status_string(rc)
    torch.cuda.synchronize()
    check_decode(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, f"continuation preset {preset}")


@pytest.mark.parametrize("preset", PRESETS)
@pytest.mark.parametrize("G,Hk,bs", [(4, 8, 16), (8, 8, 64), (4, 2, 32)])
def test_sparse_v_within_bound(orc, preset, G, Hk, bs):
    """Sparse V (rows with exp(logit - running max) <= tau leave the value
    sum): the output stays within the oracle's bound of the dense attention
    (sum over rows with exp(logit - max) <= tau of p |v| / sum p, plus the
    dense tolerance), the LSE is the dense one, tau = 0 is the plain decode
    bit for bit, and rows do drop (the output moves) when the bound says
    some may.  Keys scaled x4 make the softmax peaked."""
    rng = np.random.default_rng(9100 + 10 * preset + Hk)
    seq_lens = [700, 129]
    pb = paged_problem(orc, preset, seq_lens, Hk, bs, rng, kscale=4.0)
    B = len(seq_lens)
    q = torch.from_numpy(rng.normal(size=(B, G * Hk, 128)) * 1.5).to(torch.float16)
    sl = np.asarray(seq_lens, np.int32)
    ref_o, ref_l = orc.decode_dense(preset, to_f32(q), pb["cache"], pb["bt"], sl, Hk, bs,
                                    pb["signs"], pb["c32"])
    args = (preset, q, pb["cache"], pb["bt"], seq_lens, Hk, bs, pb["signs"], pb["c32"])
    o0, l0 = _gpu_decode(*args)
    o0s, l0s = _gpu_decode(*args, v_threshold=0.0)
    assert np.array_equal(o0, o0s) and np.array_equal(l0, l0s)
    for tau in (1e-3, 0.02):
        bound, mass = orc.sparse_v_bound(preset, to_f32(q), pb["cache"], pb["bt"], sl, Hk, bs,
                                         pb["signs"], pb["c32"], tau)
        o, l = _gpu_decode(*args, v_threshold=tau)
        err = np.abs(o.astype(np.float64) - ref_o)
        assert np.all(err <= bound + OUT_MAX_ABS), f"tau {tau}: {(err - bound).max()}"
        assert np.abs(l - ref_l).max() <= LSE_ABS
        if mass.max() > 1e-6:
            assert not np.array_equal(o, o0), f"tau {tau}: nothing dropped"



@pytest.mark.parametrize("preset", PRESETS)
@pytest.mark.parametrize("G,Hk,bs,seq_lens", [(4, 8, 16, [300, 77]), (8, 8, 64, [500, 1]),
                                               (4, 2, 32, [129, 40]), (2, 16, 16, [90])])
def test_decode_soa_cache(orc, preset, G, Hk, bs, seq_lens):
    """Decode over a cache in the SoA block convention (the oracle's cache
    re-arranged per the SoA definition) matches the oracle's attention."""
    from _helpers import aos_to_soa
    rng = np.random.default_rng(6300 + 10 * preset + Hk)
    pb = paged_problem(orc, preset, seq_lens, Hk, bs, rng)
    B = len(seq_lens)
    q = torch.from_numpy(rng.normal(size=(B, G * Hk, 128)) * 1.5).to(torch.float16)
    ref_o, ref_l = orc.decode_dense(preset, to_f32(q), pb["cache"], pb["bt"],
                                    np.asarray(seq_lens, np.int32), Hk, bs, pb["signs"], pb["c32"])
    soa = aos_to_soa(orc, preset, pb["cache"])
    out, lse = _gpu_decode(preset | tq.TQ_LAYOUT_SOA, q, soa, pb["bt"], seq_lens, Hk, bs,
                           pb["signs"], pb["c32"])
    check_decode(out, lse, ref_o, ref_l, f"soa preset {preset} G {G} Hk {Hk}")
