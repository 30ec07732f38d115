"""CPU checks of the C-ABI library: it loads, exports every symbol the
header declares, and its host logic (layout, codebook, signs, sizing,
argument validation) agrees with the oracle and the header.  No call here
reaches the GPU: every device entry point is called only with arguments
that the host-side validation rejects, or with empty sizes."""
import ctypes
import os
import re

import numpy as np
import pytest

import quantized_kv_cache_04_gb300 as tq
from quantized_kv_cache_04_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    txt = open(os.path.join(ROOT, "include", "tq.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z_0-9]+)\s*\(", txt)))


def test_library_exports_every_declared_symbol():
    L = _lib.load()
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert tq.tq_version() >= 100


def test_layout_matches_oracle(orc):
    for p in range(5):
        a = tq.tq_get_layout(p, 128)
        b = orc.layout(p, 128)
        for k in ("key_fp8", "key_bits", "value_bits", "norm_correction", "key_data_bytes",
                  "off_v_data", "value_data_bytes", "off_v_scale", "off_v_zero", "slot_size",
                  "slot_size_aligned"):
            assert a[k] == b[k], (p, k)
        assert a["off_k_norm"] == b["off_k_norm"]
    assert [tq.tq_get_layout(p)["slot_size_aligned"] for p in range(5)] == [196, 134, 118, 102, 70]
    with pytest.raises(tq.TQError):
        tq.tq_get_layout(7, 128)
    with pytest.raises(tq.TQError):
        tq.tq_get_layout(1, 100)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("d", [64, 128])
def test_codebook_matches_oracle(orc, bits, d):
    c, m = tq.tq_build_codebook(d, bits)
    _, c32, m32, _ = orc.lloyd_max(d, bits)
    assert np.array_equal(c, c32)
    assert np.array_equal(m, m32)


def test_signs_match_oracle(orc):
    for seed in (0, 42, 42 + 1337, 2**63 + 5):
        assert np.array_equal(tq.tq_make_signs(128, seed), orc.signs(128, seed))


def test_sizing():
    assert tq.tq_decode_workspace_bytes(32, 32, 16, 128) == 32 * 32 * 16 * 129 * 4
    assert tq.tq_decode_workspace_bytes(0, 32, 16, 128) == 0
    for preset in range(5):
        for B, Hk, L in [(1, 2, 512), (32, 8, 8192), (4, 8, 262144), (64, 8, 32768), (1, 1, 1),
                         (0, 8, 100), (3, 8, 0)]:
            s = tq.tq_decode_pick_splits(preset, 128, B, Hk * 4, Hk, L)
            assert 1 <= s <= _lib.TQ_MAX_SPLITS
            assert s <= max(1, (L + 127) // 128)          # splits of at least 128 tokens
    for bad in [(7, 128, 1, 8, 2, 64), (0, 128, 1, 6, 4, 64), (0, 128, 1, 8, 0, 64)]:
        with pytest.raises(tq.TQError):
            tq.tq_decode_pick_splits(*bad)
    assert tq.tq_status_string(0) == "ok"
    assert "workspace" in tq.tq_status_string(-3)


def test_device_calls_rejected_on_host():
    """Invalid arguments never reach a launch: these return without a GPU."""
    z = 0
    # head_dim 64 unsupported
    rc = tq.tq_store(1, 64, 10, 8, 16, 0, 1, 1, 512, 512, 1, 16, 1, 1, 1, 1, None)
    assert rc == _lib.TQ_ERR_UNSUPPORTED
    # block size 8 unsupported
    rc = tq.tq_store(1, 128, 10, 8, 8, 0, 1, 1, 1024, 1024, 1, 16, 1, 1, 1, 1, None)
    assert rc == _lib.TQ_ERR_UNSUPPORTED
    # fp32 inputs unsupported
    rc = tq.tq_store(1, 128, 10, 8, 16, 2, 1, 1, 1024, 1024, 1, 16, 1, 1, 1, 1, None)
    assert rc == _lib.TQ_ERR_UNSUPPORTED
    # zero tokens is a no-op
    assert tq.tq_store(1, 128, 0, 8, 16, 0, z, z, 1024, 1024, z, z, 0, z, z, z, None) == 0
    # null key pointer
    rc = tq.tq_store(1, 128, 10, 8, 16, 0, z, 1, 1024, 1024, 1, 16, 1, 1, 1, 1, None)
    assert rc == _lib.TQ_ERR_INVALID_ARG
    # token stride smaller than a token row
    rc = tq.tq_store(1, 128, 10, 8, 16, 0, 1, 1, 100, 1024, 1, 16, 1, 1, 1, 1, None)
    assert rc == _lib.TQ_ERR_INVALID_ARG
    # misaligned cache
    rc = tq.tq_store(1, 128, 10, 8, 16, 0, 1, 1, 1024, 1024, 1, 17, 1, 1, 1, 1, None)
    assert rc == _lib.TQ_ERR_INVALID_ARG
    # decode: workspace too small
    rc = tq.tq_decode_attention(1, 128, 2, 8, 2, 16, 0, 1, 1, 4, 1, 4, 1, 64, 0.1, 4, 1, 1, 1,
                                2, 0, 16, 10, None)
    assert rc == _lib.TQ_ERR_WORKSPACE
    # decode: Hq not a multiple of Hk
    rc = tq.tq_decode_attention(1, 128, 2, 9, 2, 16, 0, 1, 1, 4, 1, 4, 1, 64, 0.1, 4, 1, 1, 1,
                                2, 0, 16, 1 << 30, None)
    assert rc == _lib.TQ_ERR_INVALID_ARG
    # decode: group of 32 query heads per kv head unsupported
    rc = tq.tq_decode_attention(1, 128, 2, 64, 2, 16, 0, 1, 1, 4, 1, 4, 1, 64, 0.1, 4, 1, 1, 1,
                                2, 0, 16, 1 << 30, None)
    assert rc == _lib.TQ_ERR_UNSUPPORTED
    # decode: too many splits
    rc = tq.tq_decode_attention(1, 128, 2, 8, 2, 16, 0, 1, 1, 4, 1, 4, 1, 64, 0.1, 999, 1, 1, 1,
                                2, 0, 16, 1 << 30, None)
    assert rc == _lib.TQ_ERR_INVALID_ARG
    # decode: empty batch is a no-op
    assert tq.tq_decode_attention(1, 128, 0, 8, 2, 16, 0, z, z, 0, z, 0, z, 0, 0.1, 0, z, z, z,
                                  2, z, z, 0, None) == 0


def test_dequant_rejected_on_host():
    """tq_dequant validates its arguments before any launch."""
    z, a = 0, 1 << 20                       # a: a 16-byte aligned fake address
    args = dict(preset=1, hd=128, n=10, hk=8, bs=16, cache=a, nb=4, sm=a, sg=a, c=a, k=a, v=a,
                dt=0, ks=1024, vs=1024)

    def call(**kw):
        x = dict(args, **kw)
        return tq.tq_dequant(x["preset"], x["hd"], x["n"], x["hk"], x["bs"], x["cache"], x["nb"],
                             x["sm"], x["sg"], x["c"], x["k"], x["v"], x["dt"], x["ks"], x["vs"], None)

    assert call(hd=64) == _lib.TQ_ERR_UNSUPPORTED          # head_dim
    assert call(bs=8) == _lib.TQ_ERR_UNSUPPORTED           # block size
    assert call(dt=5) == _lib.TQ_ERR_UNSUPPORTED           # output dtype
    assert call(preset=9) == _lib.TQ_ERR_UNSUPPORTED       # preset
    assert call(n=0, cache=z, sm=z, k=z, v=z) == 0         # no tokens: no-op
    assert call(n=-1) == _lib.TQ_ERR_INVALID_ARG
    assert call(hk=0) == _lib.TQ_ERR_INVALID_ARG
    assert call(sm=z) == _lib.TQ_ERR_INVALID_ARG            # null slot mapping
    assert call(c=z) == _lib.TQ_ERR_INVALID_ARG             # MSE keys need centroids
    assert call(ks=1000) == _lib.TQ_ERR_INVALID_ARG         # stride below a token row
    assert call(vs=1028) == _lib.TQ_ERR_INVALID_ARG         # stride not a multiple of 8
    assert call(k=a + 8) == _lib.TQ_ERR_INVALID_ARG         # output not 16-byte aligned
    assert call(cache=a + 2) == _lib.TQ_ERR_INVALID_ARG     # cache not 16-byte aligned


def test_sparse_v_threshold_checked_on_host():
    """tq_decode_attention_sparse_v takes thresholds in [0, 1) only."""
    for tau in (1.5, -0.1, float("nan")):
        rc = tq.tq_decode_attention_sparse_v(1, 128, 2, 8, 2, 16, 0, 1, 1, 4, 1, 4, 1, 64, 0.1, 4,
                                             1, 1, 1, 2, 0, 16, 1 << 30, tau, None)
        assert rc == _lib.TQ_ERR_INVALID_ARG


def test_kernel_kind_follows_the_documented_rule():
    """tq_decode_kernel_kind (host only) against the rule restated in the
    test helpers, over every preset, 1-16 kv heads and groups of 1-20: the
    tensor-core stage 1 for groups up to 16 whose copied row parts are whole
    16-byte units (or whole rows of a multiple of 4 bytes) and fit its ring,
    the CUDA-core one for the other groups up to 16, unsupported above."""
    from _helpers import expected_kernel_kind
    for preset in range(5):
        for hk in range(1, 17):
            for g in range(1, 21):
                kind = tq.tq_decode_kernel_kind(preset, 128, g * hk, hk)
                want = -1 if g > 16 else expected_kernel_kind(preset, g, hk)
                assert kind == want, (preset, hk, g, kind, want)
    assert tq.tq_decode_kernel_kind(2, 64, 8, 2) == -1          # head_dim 128 only
    assert tq.tq_decode_kernel_kind(2, 128, 9, 2) == -1         # q heads not a multiple
