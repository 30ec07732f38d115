"""ctypes binding of the TurboQuant C ABI (include/tq.h).

Argument marshalling only: every step of the store and the decode runs in the
CUDA kernels of libtq_gb300.so.  The raw functions keep the C names and take
plain ints / addresses; the helpers below them take torch tensors and pass
their data pointers and the current CUDA stream.  If the library cannot be
loaded, every call raises: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

TQ_K8V4, TQ_4BIT_NC, TQ_K3V4_NC, TQ_3BIT_NC, TQ_2BIT_NC = 0, 1, 2, 3, 4
TQ_F16, TQ_BF16, TQ_F32 = 0, 1, 2
TQ_LAYOUT_SOA = 0x100       # OR-ed into a preset: SoA byte convention inside cache blocks
TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_WORKSPACE, TQ_ERR_CUDA = 0, -1, -2, -3, -4
TQ_MAX_SPLITS = 256
PRESETS = {"turboquant_k8v4": TQ_K8V4, "turboquant_4bit_nc": TQ_4BIT_NC,
           "turboquant_k3v4_nc": TQ_K3V4_NC, "turboquant_3bit_nc": TQ_3BIT_NC,
           "turboquant_2bit_nc": TQ_2BIT_NC}

_c_int, _c_ll, _c_sz, _c_vp = ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t, ctypes.c_void_p


class TQLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "key_fp8", "key_bits", "value_bits", "norm_correction", "n_centroids",
        "key_data_bytes", "key_packed_size", "value_data_bytes", "value_packed_size",
        "slot_size", "slot_size_aligned", "off_k_norm", "off_v_data", "off_v_scale",
        "off_v_zero")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class TQError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {tq_status_string(status)} ({status})")
        self.status = status


_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libtq_gb300.so (building it from source if it is absent)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise OSError(f"TurboQuant CUDA library not built: {path}")
        _build.build()
    L = ctypes.CDLL(path)
    L.tq_get_layout.argtypes = [_c_int, _c_int, ctypes.POINTER(TQLayout)]
    L.tq_build_codebook.argtypes = [_c_int, _c_int, _c_vp, _c_vp]
    L.tq_make_signs.argtypes = [_c_int, ctypes.c_uint64, _c_vp]
    L.tq_store.argtypes = ([_c_int] * 6 + [_c_vp, _c_vp, _c_ll, _c_ll, _c_vp, _c_vp, _c_ll]
                           + [_c_vp] * 4)
    L.tq_decode_pick_splits.argtypes = [_c_int] * 6
    L.tq_decode_workspace_bytes.argtypes = [_c_int] * 4
    L.tq_decode_workspace_bytes.restype = _c_sz
    L.tq_decode_attention.argtypes = ([_c_int] * 7 + [_c_vp, _c_vp, _c_ll, _c_vp, _c_int, _c_vp,
                                                      _c_int, ctypes.c_float, _c_int, _c_vp,
                                                      _c_vp, _c_vp, _c_int, _c_vp, _c_vp, _c_sz,
                                                      _c_vp])
    L.tq_decode_kernel_kind.argtypes = [_c_int] * 4
    L.tq_decode_attention_sparse_v.argtypes = ([_c_int] * 7 + [_c_vp, _c_vp, _c_ll, _c_vp, _c_int,
                                                               _c_vp, _c_int, ctypes.c_float, _c_int,
                                                               _c_vp, _c_vp, _c_vp, _c_int, _c_vp,
                                                               _c_vp, _c_sz, ctypes.c_float, _c_vp])
    L.tq_dequant.argtypes = ([_c_int] * 5 + [_c_vp, _c_ll, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int,
                                             _c_ll, _c_ll, _c_vp])
    L.tq_status_string.argtypes = [_c_int]
    L.tq_status_string.restype = ctypes.c_char_p
    L.tq_version.restype = _c_int
    _lib = L
    return L


# ------------------------------------------------------------------ raw C names
def tq_status_string(status: int) -> str:
    return load().tq_status_string(int(status)).decode()


def tq_version() -> int:
    return load().tq_version()


def tq_get_layout(preset: int, head_dim: int = 128) -> dict:
    out = TQLayout()
    rc = load().tq_get_layout(int(preset), int(head_dim), ctypes.byref(out))
    if rc:
        raise TQError("tq_get_layout", rc)
    return out.as_dict()


def tq_build_codebook(head_dim: int, bits: int):
    """Host Lloyd-Max codebook -> (centroids, midpoints) as numpy float32."""
    import numpy as np
    c = np.zeros(1 << bits, np.float32)
    m = np.zeros(max(1, (1 << bits) - 1), np.float32)
    rc = load().tq_build_codebook(int(head_dim), int(bits), c.ctypes.data, m.ctypes.data)
    if rc:
        raise TQError("tq_build_codebook", rc)
    return c, m[: (1 << bits) - 1]


def tq_make_signs(head_dim: int, seed: int = 42):
    import numpy as np
    s = np.zeros(head_dim, np.int8)
    rc = load().tq_make_signs(int(head_dim), ctypes.c_uint64(seed & (2**64 - 1)), s.ctypes.data)
    if rc:
        raise TQError("tq_make_signs", rc)
    return s


def tq_decode_pick_splits(preset: int, head_dim: int, batch: int, num_q_heads: int,
                          num_kv_heads: int, max_seq_len: int) -> int:
    s = load().tq_decode_pick_splits(int(preset), int(head_dim), int(batch), int(num_q_heads),
                                     int(num_kv_heads), int(max_seq_len))
    if s < 0:
        raise TQError("tq_decode_pick_splits", s)
    return s


def tq_decode_kernel_kind(preset: int, head_dim: int, num_q_heads: int, num_kv_heads: int) -> int:
    """1 = tensor-core stage 1, 0 = CUDA-core stage 1, -1 = unsupported shape."""
    return load().tq_decode_kernel_kind(int(preset), int(head_dim), int(num_q_heads),
                                        int(num_kv_heads))


def tq_decode_workspace_bytes(batch: int, num_q_heads: int, num_splits: int, head_dim: int = 128) -> int:
    return int(load().tq_decode_workspace_bytes(int(batch), int(num_q_heads), int(num_splits),
                                                int(head_dim)))


def tq_store(*args) -> int:
    """Raw C call; arguments exactly as in include/tq.h.  Returns the status."""
    return load().tq_store(*args)


def tq_decode_attention(*args) -> int:
    """Raw C call; arguments exactly as in include/tq.h.  Returns the status."""
    return load().tq_decode_attention(*args)


def tq_decode_attention_sparse_v(*args) -> int:
    """Raw C call; arguments exactly as in include/tq.h.  Returns the status."""
    return load().tq_decode_attention_sparse_v(*args)


def tq_dequant(*args) -> int:
    """Raw C call; arguments exactly as in include/tq.h.  Returns the status."""
    return load().tq_dequant(*args)


# ------------------------------------------------------------------ torch helpers
def _dtype_code(t) -> int:
    import torch
    return {torch.float16: TQ_F16, torch.bfloat16: TQ_BF16, torch.float32: TQ_F32}[t.dtype]


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def store(preset: int, key, value, slot_mapping, kv_cache, block_size: int, signs,
          centroids=None, midpoints=None, stream=None) -> None:
    """tq_store on torch tensors.  key/value (N, Hk, D) with unit inner strides."""
    N, Hk, D = key.shape
    assert key.stride(2) == 1 and key.stride(1) == D and value.stride(2) == 1 and value.stride(1) == D
    rc = tq_store(int(preset), D, N, Hk, int(block_size), _dtype_code(key), _ptr(key), _ptr(value),
                  key.stride(0), value.stride(0), _ptr(slot_mapping), _ptr(kv_cache),
                  kv_cache.shape[0], _ptr(signs), _ptr(centroids), _ptr(midpoints),
                  _stream_ptr(stream))
    if rc:
        raise TQError("tq_store", rc)


def dequant(preset: int, slot_mapping, kv_cache, num_kv_heads: int, block_size: int, signs,
            centroids, key_out, value_out, stream=None) -> None:
    """tq_dequant on torch tensors: key_out/value_out (N, Hk, D) with unit inner strides."""
    N, Hk, D = key_out.shape
    assert key_out.stride(2) == 1 and key_out.stride(1) == D
    assert value_out.stride(2) == 1 and value_out.stride(1) == D and value_out.dtype == key_out.dtype
    rc = tq_dequant(int(preset), D, N, int(num_kv_heads), int(block_size), _ptr(kv_cache),
                    kv_cache.shape[0], _ptr(slot_mapping), _ptr(signs), _ptr(centroids),
                    _ptr(key_out), _ptr(value_out), _dtype_code(key_out), key_out.stride(0),
                    value_out.stride(0), _stream_ptr(stream))
    if rc:
        raise TQError("tq_dequant", rc)


def decode_attention(preset: int, query, kv_cache, block_table, seq_lens, max_seq_len: int,
                     num_kv_heads: int, block_size: int, signs, centroids, out, lse, workspace,
                     num_splits: int = 0, softmax_scale: float | None = None, stream=None,
                     v_threshold: float = 0.0) -> None:
    """tq_decode_attention (or, with v_threshold > 0, the sparse-V form) on
    torch tensors.  query (B, Hq, D) contiguous."""
    B, Hq, D = query.shape
    assert query.is_contiguous() and out.is_contiguous()
    scale = D ** -0.5 if softmax_scale is None else float(softmax_scale)
    args = (int(preset), D, B, Hq, int(num_kv_heads), int(block_size),
            _dtype_code(query), _ptr(query), _ptr(kv_cache), kv_cache.shape[0],
            _ptr(block_table), block_table.stride(0), _ptr(seq_lens),
            int(max_seq_len), scale, int(num_splits), _ptr(signs),
            _ptr(centroids), _ptr(out), _dtype_code(out), _ptr(lse),
            _ptr(workspace), workspace.numel() * workspace.element_size())
    if v_threshold:
        rc = tq_decode_attention_sparse_v(*args, float(v_threshold), _stream_ptr(stream))
        if rc:
            raise TQError("tq_decode_attention_sparse_v", rc)
        return
    rc = tq_decode_attention(*args, _stream_ptr(stream))
    if rc:
        raise TQError("tq_decode_attention", rc)


TQ_NOALLOC_SCRATCH_BYTES = 16 << 20


def tq_decode_attention_noalloc(*args) -> int:
    """Raw C call of the decode entry point that allocates nothing (arguments
    as tq_decode_attention without workspace and workspace_bytes).  For
    callers that cannot allocate device memory: the split partials live in a
    fixed 16 MiB array the library declares in device memory, shared by all
    calls, so calls that overlap on the GPU race.  Returns the status."""
    L = load()
    fn = L.tq_decode_attention_noalloc
    if fn.argtypes is None:
        fn.argtypes = ([_c_int] * 7 + [_c_vp, _c_vp, _c_ll, _c_vp, _c_int, _c_vp, _c_int,
                                       ctypes.c_float, _c_int, _c_vp, _c_vp, _c_vp, _c_int, _c_vp,
                                       _c_vp])
    return fn(*args)


def tq_test_decode_wait_expiry(*args) -> int:
    """Raw C call of the wait-expiry test entry point (arguments as
    tq_decode_attention, then stuck_tile, wait_polls, stream): one stage of
    split 0 of sequence 0 never completes, its bounded waits run out, and
    those heads come out NaN.  Returns the status."""
    L = load()
    fn = L.tq_test_decode_wait_expiry
    if fn.argtypes is None:
        fn.argtypes = ([_c_int] * 7 + [_c_vp, _c_vp, _c_ll, _c_vp, _c_int, _c_vp, _c_int,
                                       ctypes.c_float, _c_int, _c_vp, _c_vp, _c_vp, _c_int, _c_vp,
                                       _c_vp, _c_sz, _c_int, ctypes.c_uint, _c_vp])
    return fn(*args)
