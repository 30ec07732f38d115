"""The tensor-core stage 1 gives up on a stage whose copies never complete,
without a fault or a hang: its mbarrier waits are bounded.

tq_test_decode_wait_expiry announces one tile (split 0, sequence 0, kv-head
group 0) to its mbarrier as 16 bytes longer than the copies that fill it,
with a short poll limit.  Every copy lands, but the stage never completes:
the CTA's warps give up, drain their other requests with the same limit and
give their heads a NaN lse for that split.  The test checks that exactly
those query heads of sequence 0 come out NaN, that every other output and
lse equals the clean decode bit for bit, and that the context still decodes
correctly afterwards.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import quantized_kv_cache_04_gb300 as tq
from quantized_kv_cache_04_gb300 import _lib
from quantized_kv_cache_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _args(p, out, lse, ws):
    c, w = p.c, p.w
    return (c.preset, 128, w.B, w.Hq, w.Hk, w.block_size, _lib._dtype_code(p.q), p.q.data_ptr(),
            c.cache.data_ptr(), c.cache.shape[0], p.bt.data_ptr(), p.bt.stride(0), p.sl.data_ptr(),
            p.max_len, 128 ** -0.5, p.S, c.signs.data_ptr(),
            0 if c.centroids is None else c.centroids.data_ptr(), out.data_ptr(), tq.TQ_F32,
            lse.data_ptr(), ws.data_ptr(), ws.numel())


def _clean(p):
    out = torch.empty((p.w.B, p.w.Hq, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((p.w.B, p.w.Hq), dtype=torch.float32, device="cuda")
    rc = tq.tq_decode_attention(*_args(p, out, lse, p.ws), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, tq.tq_status_string(rc)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def _stuck(p, tile, polls):
    out = torch.empty((p.w.B, p.w.Hq, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((p.w.B, p.w.Hq), dtype=torch.float32, device="cuda")
    rc = _lib.tq_test_decode_wait_expiry(*_args(p, out, lse, p.ws), tile, polls,
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == 0, tq.tq_status_string(rc)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("preset,q_heads", [("turboquant_k8v4", 32), ("turboquant_k3v4_nc", 32),
                                            ("turboquant_k3v4_nc", 64)])
def test_bounded_wait_runs_out_and_marks_the_split(preset, q_heads):
    """Groups of 4 and of 8 query heads; with 8 and Lloyd-Max keys the CTA
    also frees its tensor-memory q columns on the way out."""
    import bench
    w = wl.make("sweep", preset=preset, ctx=2048, batch=3, q_heads=q_heads)
    p = bench.Problem(w, torch.device("cuda"), 2)         # 2 splits of 32 tiles
    assert tq.tq_decode_kernel_kind(p.c.preset, 128, w.Hq, w.Hk) == 1
    o0, l0 = _clean(p)
    o1, l1 = _stuck(p, tile=1, polls=1000)
    G = w.Hq // w.Hk
    hpc = 4 if preset == "turboquant_k8v4" else w.Hk       # kv heads per CTA of the tensor-core stage 1
    hit = np.zeros((w.B, w.Hq), bool)
    hit[0, :hpc * G] = True
    assert np.all(np.isnan(l1[hit])) and np.all(np.isnan(o1[hit]))
    assert np.array_equal(l1[~hit], l0[~hit]) and np.array_equal(o1[~hit], o0[~hit])
    # a tile past the split's end is never requested: nothing changes
    o2, l2 = _stuck(p, tile=10_000, polls=1000)
    assert np.array_equal(l2, l0) and np.array_equal(o2, o0)
    # the context is still usable and decodes as before
    o3, l3 = _clean(p)
    assert np.array_equal(l3, l0) and np.array_equal(o3, o0)
    assert np.all(np.isfinite(l0)) and np.all(np.isfinite(o0))


def test_wait_expiry_rejects_the_cuda_core_path():
    import bench
    # one kv head with 3-bit keys: 118-byte token rows, the CUDA-core stage 1
    w = wl.make("sweep", preset="turboquant_k3v4_nc", ctx=512, batch=1, q_heads=4, kv_heads=1)
    p = bench.Problem(w, torch.device("cuda"), 4)
    assert tq.tq_decode_kernel_kind(p.c.preset, 128, w.Hq, w.Hk) == 0
    out = torch.empty((w.B, w.Hq, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    rc = _lib.tq_test_decode_wait_expiry(*_args(p, out, lse, p.ws), 0, 1000,
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.TQ_ERR_UNSUPPORTED
