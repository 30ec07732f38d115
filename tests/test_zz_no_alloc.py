"""The decode entry point that allocates nothing.

Some callers cannot allocate device memory (an engine that has handed the
GPU's memory to its own KV-cache pool, or a latency-critical loop that must
not take cudaMalloc's device-wide synchronisation).  tq_decode_attention_noalloc
serves them by keeping the split partials in a fixed array that the library
declares in device memory.  This test calls it through the C ABI twice in a
row, on different inputs, and checks each result against the regular entry
point that takes a caller-owned workspace.  It lives in its own file that
pytest collects last, and it needs nothing from the other tests.
"""
import numpy as np
import pytest
import torch

import quantized_kv_cache_04_gb300 as tq
from quantized_kv_cache_04_gb300 import _lib

pytestmark = pytest.mark.gpu


def _problem(seed, preset, B, Hq, Hk, bs, ctx, dtype, on_device=False):
    """A paged cache of B sequences of ctx tokens.  Inputs are drawn on the
    CPU, or on the GPU for the large shapes (on_device)."""
    dev = torch.device("cuda")
    g = torch.Generator(device="cpu").manual_seed(seed)
    gk = torch.Generator(device=dev).manual_seed(seed) if on_device else g
    L = tq.tq_get_layout(preset)
    nblk = (ctx + bs - 1) // bs
    nb = B * nblk
    cache = torch.zeros((nb, bs, Hk, L["slot_size_aligned"]), dtype=torch.uint8, device=dev)
    perm = torch.randperm(nb, generator=g).to(torch.int32)
    bt = perm.view(B, nblk).contiguous().to(dev)
    signs = torch.from_numpy(tq.tq_make_signs(128, 42)).to(dev)
    cent = mids = None
    if not L["key_fp8"]:
        c, m = tq.tq_build_codebook(128, L["key_bits"])
        cent, mids = torch.from_numpy(c).to(dev), torch.from_numpy(m).to(dev)
    kv_dev = dev if on_device else "cpu"
    for b in range(B):
        K = torch.randn((ctx, Hk, 128), generator=gk, device=kv_dev).to(dtype).to(dev)
        V = torch.randn((ctx, Hk, 128), generator=gk, device=kv_dev).to(dtype).to(dev)
        t = torch.arange(ctx)
        sm = (bt[b].cpu()[t // bs].long() * bs + t % bs).to(dev)
        tq.store(preset, K, V, sm, cache, bs, signs, cent, mids)
    q = torch.randn((B, Hq, 128), generator=g).to(dtype).to(dev)
    sl = torch.full((B,), ctx, dtype=torch.int32, device=dev)
    return dict(preset=preset, B=B, Hq=Hq, Hk=Hk, bs=bs, ctx=ctx, q=q, cache=cache, bt=bt, sl=sl,
                signs=signs, cent=cent)


def _args(p, num_splits, out, lse):
    stream = torch.cuda.current_stream().cuda_stream
    return (p["preset"], 128, p["B"], p["Hq"], p["Hk"], p["bs"], tq.TQ_F16 if p["q"].dtype == torch.float16
            else tq.TQ_BF16, p["q"].data_ptr(), p["cache"].data_ptr(), p["cache"].shape[0],
            p["bt"].data_ptr(), p["bt"].stride(0), p["sl"].data_ptr(), p["ctx"], 128 ** -0.5,
            num_splits, p["signs"].data_ptr(), 0 if p["cent"] is None else p["cent"].data_ptr(),
            out.data_ptr(), tq.TQ_F32, lse.data_ptr(), stream)


def _with_workspace(p, num_splits):
    S = num_splits or tq.tq_decode_pick_splits(p["preset"], 128, p["B"], p["Hq"], p["Hk"], p["ctx"])
    ws = torch.empty(tq.tq_decode_workspace_bytes(p["B"], p["Hq"], S, 128), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((p["B"], p["Hq"], 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((p["B"], p["Hq"]), dtype=torch.float32, device="cuda")
    args = _args(p, S, out, lse)
    rc = tq.tq_decode_attention(*args[:-1], ws.data_ptr(), ws.numel(), args[-1])
    assert rc == 0, tq.tq_status_string(rc)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def _no_alloc(p, num_splits):
    out = torch.full((p["B"], p["Hq"], 128), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((p["B"], p["Hq"]), float("nan"), dtype=torch.float32, device="cuda")
    rc = _lib.tq_decode_attention_noalloc(*_args(p, num_splits, out, lse))
    assert rc == 0, tq.tq_status_string(rc)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def _close(a, b):
    (o1, l1), (o2, l2) = a, b
    assert np.all(np.isfinite(o2)) and np.all(np.isfinite(l2))
    assert np.max(np.abs(o1 - o2)) <= 2e-3
    assert np.linalg.norm(o1 - o2) <= 1e-3 * np.linalg.norm(o1)
    assert np.max(np.abs(l1 - l2)) <= 1e-4


def test_no_alloc_matches_workspace_entry_point_twice():
    first = _problem(11, tq.TQ_K8V4, B=4, Hq=32, Hk=8, bs=16, ctx=3000, dtype=torch.bfloat16)
    second = _problem(12, tq.TQ_K3V4_NC, B=3, Hq=16, Hk=2, bs=64, ctx=1500, dtype=torch.float16)
    # two calls in a row, different shapes and inputs, explicit split counts
    _close(_with_workspace(first, 6), _no_alloc(first, 6))
    _close(_with_workspace(second, 5), _no_alloc(second, 5))
    # library-chosen split count (fits the array for these shapes)
    _close(_with_workspace(first, 0), _no_alloc(first, 0))


def test_no_alloc_rejects_partials_beyond_its_array():
    p = _problem(13, tq.TQ_K8V4, B=4, Hq=64, Hk=8, bs=16, ctx=64, dtype=torch.float16)
    per_split = tq.tq_decode_workspace_bytes(p["B"], p["Hq"], 1, 128)
    too_many = _lib.TQ_NOALLOC_SCRATCH_BYTES // per_split + 1
    assert too_many <= _lib.TQ_MAX_SPLITS
    out = torch.empty((p["B"], p["Hq"], 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((p["B"], p["Hq"]), dtype=torch.float32, device="cuda")
    assert _lib.tq_decode_attention_noalloc(*_args(p, too_many, out, lse)) == _lib.TQ_ERR_WORKSPACE


def test_no_alloc_lowers_the_library_split_count_to_fit():
    """With num_splits = 0 and a shape whose library-chosen split count
    would not fit the array (B = 64 sequences x 64 query heads: about 2.1 MB
    of partials per split, so at most 7 splits fit), the call runs with the
    largest count that fits, and gives exactly what the workspace entry
    point gives with that count."""
    B, Hq, Hk = 64, 64, 8
    per_split = tq.tq_decode_workspace_bytes(B, Hq, 1, 128)
    fit = _lib.TQ_NOALLOC_SCRATCH_BYTES // per_split
    ctx = next((c for c in (8192, 16384, 32768)
                if tq.tq_decode_pick_splits(tq.TQ_K3V4_NC, 128, B, Hq, Hk, c) > fit), None)
    assert ctx is not None, "no context length where the library picks more splits than fit"
    p = _problem(14, tq.TQ_K3V4_NC, B=B, Hq=Hq, Hk=Hk, bs=64, ctx=ctx, dtype=torch.float16,
                 on_device=True)
    o1, l1 = _with_workspace(p, fit)
    o2, l2 = _no_alloc(p, 0)
    assert np.all(np.isfinite(o2)) and np.all(np.isfinite(l2))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
