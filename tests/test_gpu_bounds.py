"""Block-table entries outside the cache.

An entry that the decode would read and that lies outside [0, num_blocks)
is a caller error.  Both stage-1 kernels check every page they read against
num_blocks before touching it; such a page is not read, and every query
head of that sequence comes out NaN (output and LSE), while the other
sequences of the batch keep the exact result of a clean table.

The out-of-range entries used here (-1 and num_blocks .. num_blocks + 2)
still point into the test's device allocation: the cache handed to the
library is a view that starts one block into a larger buffer and ends three
blocks before its end, so even an unchecked read would stay inside memory
this process owns.
"""
import numpy as np
import pytest
import torch

import quantized_kv_cache_04_gb300 as tq
from _helpers import expected_kernel_kind, paged_problem

pytestmark = pytest.mark.gpu


def _decode(preset, q, cache, bt, seq_lens, Hk, bs, signs, c32, num_splits):
    dev = torch.device("cuda")
    B, Hq, D = q.shape
    L = tq.tq_get_layout(preset)
    btd = torch.from_numpy(np.ascontiguousarray(bt)).to(dev)
    sl = torch.from_numpy(np.asarray(seq_lens, np.int32)).to(dev)
    sg = torch.from_numpy(signs).to(dev)
    cc = torch.from_numpy(c32).to(dev) if not L["key_fp8"] else None
    maxlen = int(max(seq_lens))
    ws = torch.empty(tq.tq_decode_workspace_bytes(B, Hq, num_splits, D), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    tq.decode_attention(preset, q.to(dev).contiguous(), cache, btd, sl, maxlen, Hk, bs, sg, cc,
                        out, lse, ws, num_splits=num_splits)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("preset", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("G,Hk,bs,splits", [(4, 2, 16, 3), (4, 8, 32, 2), (16, 1, 16, 3), (2, 1, 16, 3),
                                             (1, 16, 16, 3)])
def test_out_of_range_pages_give_nan_rows(orc, preset, G, Hk, bs, splits):
    dev = torch.device("cuda")
    rng = np.random.default_rng(9700 + 10 * preset + Hk)
    seq_lens = [300, 200, 150, 90]
    pb = paged_problem(orc, preset, seq_lens, Hk, bs, rng)
    cache_np, bt = pb["cache"], pb["bt"]
    nb = cache_np.shape[0]
    big = torch.zeros((nb + 4,) + cache_np.shape[1:], dtype=torch.uint8, device=dev)
    big[1:nb + 1] = torch.from_numpy(cache_np).to(dev)
    cache = big[1:nb + 1]                      # num_blocks = nb
    assert cache.shape[0] == nb and cache.is_contiguous()
    q = torch.from_numpy(rng.normal(size=(len(seq_lens), G * Hk, 128))).to(torch.float16)
    # both stage-1 kernels: one kv head with Lloyd-Max keys (rows not
    # 4-byte aligned) and 16 kv heads of 3- or 4-bit keys (rows too large for
    # the tensor-core ring) take the CUDA-core stage 1
    kind = tq.tq_decode_kernel_kind(preset, 128, G * Hk, Hk)
    assert kind == expected_kernel_kind(preset, G, Hk)

    ref_o, ref_l = _decode(preset, q, cache, bt, seq_lens, Hk, bs, pb["signs"], pb["c32"], splits)
    assert np.all(np.isfinite(ref_o)) and np.all(np.isfinite(ref_l))

    bad = bt.copy()
    nblk = [(n + bs - 1) // bs for n in seq_lens]
    bad[1, nblk[1] // 2] = -1                  # a middle page
    bad[2, nblk[2] - 1] = nb                   # the last page
    bad[3, 0] = nb + 1                         # the first page
    o, l = _decode(preset, q, cache, bad, seq_lens, Hk, bs, pb["signs"], pb["c32"], splits)
    assert np.array_equal(o[0], ref_o[0]) and np.array_equal(l[0], ref_l[0])
    for b in (1, 2, 3):
        assert np.all(np.isnan(l[b])), f"sequence {b}: lse {l[b]}"
        assert np.all(np.isnan(o[b])), f"sequence {b}: output not NaN"

    # entries past the sequence's last page are never read, in range or not
    tail = bt.copy()
    for b, n in enumerate(nblk):
        tail[b, n:] = -1 if b % 2 else nb + 2
    o, l = _decode(preset, q, cache, tail, seq_lens, Hk, bs, pb["signs"], pb["c32"], splits)
    assert np.array_equal(o, ref_o) and np.array_equal(l, ref_l)
