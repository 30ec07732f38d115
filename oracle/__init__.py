"""CPU oracle for the TurboQuant KV-cache hot path (test infrastructure).

This package is TEST INFRASTRUCTURE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  The product library never links, imports or calls it; the
two share no code.  The arithmetic lives in ``tq_oracle.c`` (plain C,
compiled with ``-ffp-contract=off``); this module only marshals numpy
arrays into it.

Every function documented in ``tq_oracle.h`` is exposed here with numpy
arguments.  Parity of each oracle function is pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_HDR = os.path.join(_HERE, "tq_oracle.h")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")

K8V4, TQ4_NC, K3V4_NC, TQ3_NC, TQ2_NC = 0, 1, 2, 3, 4
LAYOUT_SOA = 0x100          # OR-ed into a preset: SoA byte convention inside cache blocks
PRESETS = {"turboquant_k8v4": K8V4, "turboquant_4bit_nc": TQ4_NC,
           "turboquant_k3v4_nc": K3V4_NC, "turboquant_3bit_nc": TQ3_NC,
           "turboquant_2bit_nc": TQ2_NC}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no GPU needed).  Returns the .so path."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < newest:
        os.makedirs(os.path.dirname(_OUT), exist_ok=True)
        tmp = _OUT + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _OUT)
    return _OUT


class _Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "key_fp8", "key_bits", "value_bits", "norm_correction", "key_data_bytes",
        "off_k_norm", "off_v_data", "value_data_bytes", "off_v_scale", "off_v_zero",
        "slot_size", "slot_size_aligned")]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        L = _lib
        L.orc_double_to_f16.restype = ctypes.c_uint16
        L.orc_double_to_f16.argtypes = [ctypes.c_double]
        L.orc_f16_to_double.restype = ctypes.c_double
        L.orc_f16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_float.restype = ctypes.c_float
        L.orc_bf16_to_float.argtypes = [ctypes.c_uint16]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_double]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_lloyd_max.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p]
        L.orc_signs.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_void_p]
        L.orc_hadamard.argtypes = [ctypes.c_int, ctypes.c_void_p]
        L.orc_pack.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        L.orc_unpack.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        L.orc_get_layout.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(_Layout)]
        L.orc_store_one.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 7
        L.orc_store.argtypes = ([ctypes.c_int] * 5 + [ctypes.c_void_p] * 4 + [ctypes.c_int64]
                                + [ctypes.c_void_p] * 3)
        L.orc_dequant_slot.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 5
        common = ([ctypes.c_int] * 6 + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                        ctypes.c_double])
        L.orc_decode_dense.argtypes = common + [ctypes.c_void_p] * 4
        L.orc_decode_split.argtypes = common + [ctypes.c_int] + [ctypes.c_void_p] * 4
        L.orc_sparse_v_bound.argtypes = common + [ctypes.c_double] + [ctypes.c_void_p] * 4
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- scalars
def f16_bits(x: float) -> int:
    return int(lib().orc_double_to_f16(float(x)))


def f16_value(bits: int) -> float:
    return float(lib().orc_f16_to_double(int(bits)))


def bf16_value(bits: int) -> float:
    return float(lib().orc_bf16_to_float(int(bits)))


def e4m3_encode(x: float) -> int:
    return int(lib().orc_e4m3_encode(float(x)))


def e4m3_decode(b: int) -> float:
    return float(lib().orc_e4m3_decode(int(b)))


# ---------------------------------------------------------------- layout
def layout(preset: int, head_dim: int = 128) -> dict:
    L = _Layout()
    if lib().orc_get_layout(int(preset), int(head_dim), ctypes.byref(L)):
        raise ValueError("bad preset / head_dim")
    return {n: getattr(L, n) for n, _ in _Layout._fields_}


# ---------------------------------------------------------------- codebook
def lloyd_max(d: int, bits: int, trapz_n: int = 200, max_iter: int = 200, tol: float = 1e-10):
    """Returns (centroids as float64 iterate, fp32 centroids, fp32 midpoints, iterations)."""
    n = 1 << bits
    c64 = np.zeros(n, np.float64)
    c32 = np.zeros(n, np.float32)
    m32 = np.zeros(n - 1, np.float32)
    it = lib().orc_lloyd_max(d, bits, trapz_n, max_iter, tol, _p(c64), _p(c32), _p(m32))
    if it < 0:
        raise ValueError("bad arguments")
    return c64, c32, m32, it


def codebook(head_dim: int, bits: int):
    """fp32 centroids and fp32 midpoints with the page's defaults."""
    _, c32, m32, _ = lloyd_max(head_dim, bits)
    return c32, m32


# ---------------------------------------------------------------- rotation
def signs(head_dim: int, seed: int = 42) -> np.ndarray:
    s = np.zeros(head_dim, np.int8)
    lib().orc_signs(head_dim, ctypes.c_uint64(seed & (2**64 - 1)), _p(s))
    return s


def hadamard(D: int) -> np.ndarray:
    H = np.zeros((D, D), np.float64)
    lib().orc_hadamard(D, _p(H))
    return H


# ---------------------------------------------------------------- packing
def pack(codes, bits: int) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, np.int32))
    out = np.zeros((c.size * bits + 7) // 8, np.uint8)
    lib().orc_pack(_p(c), c.size, bits, _p(out))
    return out


def unpack(data, n: int, bits: int) -> np.ndarray:
    d = np.ascontiguousarray(np.asarray(data, np.uint8))
    out = np.zeros(n, np.int32)
    lib().orc_unpack(_p(d), n, bits, _p(out))
    return out


# ---------------------------------------------------------------- store
def store_one(preset, k, v, signs_, c32, m32):
    """Returns (slot bytes, fp32 pre-quantisation coordinates)."""
    k = np.ascontiguousarray(k, np.float32)
    v = np.ascontiguousarray(v, np.float32)
    D = k.size
    lay = layout(preset, D)
    slot = np.zeros(lay["slot_size_aligned"], np.uint8)
    y = np.zeros(D, np.float32)
    s = np.ascontiguousarray(signs_, np.int8)
    c = np.ascontiguousarray(c32, np.float32)
    m = np.ascontiguousarray(m32, np.float32)
    rc = lib().orc_store_one(preset, D, _p(k), _p(v), _p(s), _p(c), _p(m), _p(slot), _p(y))
    if rc:
        raise ValueError(rc)
    return slot, y


def store(preset, key, value, slot_mapping, cache, block_size, signs_, c32, m32):
    """key/value (N, Hk, D) float32; cache (num_blocks, bs, Hk, slot) uint8, updated in place."""
    key = np.ascontiguousarray(key, np.float32)
    value = np.ascontiguousarray(value, np.float32)
    sm = np.ascontiguousarray(slot_mapping, np.int64)
    N, Hk, D = key.shape
    assert cache.flags["C_CONTIGUOUS"] and cache.dtype == np.uint8
    s = np.ascontiguousarray(signs_, np.int8)
    c = np.ascontiguousarray(c32, np.float32)
    m = np.ascontiguousarray(m32, np.float32)
    rc = lib().orc_store(preset, D, N, Hk, block_size, _p(key), _p(value), _p(sm), _p(cache),
                         cache.shape[0], _p(s), _p(c), _p(m))
    if rc:
        raise ValueError(rc)
    return cache


def dequant_slot(preset, slot, signs_, c32, head_dim=128):
    slot = np.ascontiguousarray(slot, np.uint8)
    kh = np.zeros(head_dim, np.float64)
    vh = np.zeros(head_dim, np.float64)
    s = np.ascontiguousarray(signs_, np.int8)
    c = np.ascontiguousarray(c32 if c32 is not None else np.zeros(16, np.float32), np.float32)
    rc = lib().orc_dequant_slot(preset, head_dim, _p(slot), _p(s), _p(c), _p(kh), _p(vh))
    if rc:
        raise ValueError(rc)
    return kh, vh


# ---------------------------------------------------------------- decode
def _decode(fn, preset, q, cache, block_table, seq_lens, Hk, block_size, signs_, c32,
            scale, extra):
    q = np.ascontiguousarray(q, np.float32)
    B, Hq, D = q.shape
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    s = np.ascontiguousarray(signs_, np.int8)
    c = np.ascontiguousarray(c32 if c32 is not None else np.zeros(16, np.float32), np.float32)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    args = [preset, D, B, Hq, Hk, block_size, _p(q), _p(cache), cache.shape[0], _p(bt),
            bt.shape[1] if bt.ndim == 2 else 0, _p(sl), float(scale)] + extra + \
           [_p(s), _p(c), _p(out), _p(lse)]
    rc = fn(*args)
    if rc:
        raise ValueError(rc)
    return out, lse


def decode_dense(preset, q, cache, block_table, seq_lens, Hk, block_size, signs_, c32,
                 scale=None):
    """Dense softmax attention over the dequantised cache.  Returns (out, lse) float64."""
    return _decode(lib().orc_decode_dense, preset, q, cache, block_table, seq_lens, Hk,
                   block_size, signs_, c32, scale, [])


def decode_split(preset, q, cache, block_table, seq_lens, Hk, block_size, signs_, c32,
                 num_splits, scale=None):
    """Rotated-q, LUT-score, split-K + log-sum-exp merge form.  Returns (out, lse)."""
    return _decode(lib().orc_decode_split, preset, q, cache, block_table, seq_lens, Hk,
                   block_size, signs_, c32, scale, [int(num_splits)])


def sparse_v_bound(preset, q, cache, block_table, seq_lens, Hk, block_size, signs_, c32, tau,
                   scale=None):
    """Per-dimension bound on how far the sparse-V output may move from the
    dense one when rows with exp(logit - max) <= tau drop out of the value
    sum, and the weight of those rows.  Returns (bound (B,Hq,D), mass (B,Hq))."""
    return _decode(lib().orc_sparse_v_bound, preset, q, cache, block_table, seq_lens, Hk,
                   block_size, signs_, c32, scale, [float(tau)])
