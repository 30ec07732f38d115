"""Seeded synthetic workloads for the TurboQuant KV-cache store and decode.

This module only draws random inputs (shapes, values, paging metadata).  It
holds none of the method's arithmetic, so the CUDA path and the CPU oracle
can both take their inputs from it.

The shapes follow the workloads the pages talk about: GQA heads with
head_dim 128, paged caches with block sizes 16-128 ("get_supported_kernel_
block_sizes" in the vLLM backend), contexts from 512 to 256K tokens, and the
four cache presets.  Value distributions stand in for real activations
(normal with outlier channels, per-channel scales, heavy tails, planted
high-similarity keys); no model weights or datasets are involved.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

PRESET_IDS = {"turboquant_k8v4": 0, "turboquant_4bit_nc": 1,
              "turboquant_k3v4_nc": 2, "turboquant_3bit_nc": 3, "turboquant_2bit_nc": 4}
PRESET_NAMES = {v: k for k, v in PRESET_IDS.items()}
SIGN_SEED = 42


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hk: int
    D: int
    block_size: int
    preset: str
    dtype: str                  # "float16" | "bfloat16"
    seq_lens: np.ndarray        # (B,) int32
    block_table: np.ndarray     # (B, max_blocks) int32, unused entries -> guard block
    num_blocks: int             # includes the trailing guard block
    num_splits: int             # 0 = library picks
    seed: int
    values: str                 # value-distribution recipe name
    chan_scale_k: np.ndarray | None = None   # (Hk, D) per-channel scale for K and Q
    chan_scale_v: np.ndarray | None = None   # (Hk, D) per-channel scale for V
    outlier_channels: np.ndarray | None = None
    plant_every: int = 0

    @property
    def guard_block(self) -> int:
        return self.num_blocks - 1

    @property
    def preset_id(self) -> int:
        return PRESET_IDS[self.preset]

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.sum())

    def slot_mapping(self, b: int, positions: np.ndarray) -> np.ndarray:
        """Cache slot of each position of sequence b."""
        pos = np.asarray(positions, np.int64)
        blocks = self.block_table[b, pos // self.block_size].astype(np.int64)
        return blocks * self.block_size + pos % self.block_size


def _paging(seq_lens: np.ndarray, bs: int, rng: np.random.Generator, shuffle: bool):
    nblk = [(int(n) + bs - 1) // bs for n in seq_lens]
    total = sum(nblk)
    ids = rng.permutation(total) if shuffle else np.arange(total)
    width = max(1, max(nblk))
    guard = total                      # one extra block, never written
    bt = np.full((len(seq_lens), width), guard, np.int32)
    pos = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = ids[pos:pos + n]
        pos += n
    return bt, total + 1


def make(name: str, preset: str | None = None, seed: int | None = None,
         batch: int | None = None, ctx: int | None = None,
         q_heads: int | None = None, kv_heads: int | None = None) -> Workload:
    """Build the paging metadata and value recipe of a named workload.

    tiny        B=1, Hq=8, Hk=2, ctx 512, bs 16, 4bit_nc, fp16, 4 outlier channels x8
    llama3_8b   B=32, Hq=32, Hk=8, ctx 8192, bs 16, k8v4, bf16, per-channel scale
                log-uniform in [0.25, 4], random block permutation
    qwen3_32b   B=64, Hq=64, Hk=8, ctx ~ U{16384..32768}, bs 64, k3v4_nc, fp16,
                2% of coordinates Student-t(3)
    long        B=4, Hq=32, Hk=8, ctx 262144, bs 128, 3bit_nc, bf16, a planted
                high-similarity key every 4096 tokens, 64 splits
    store_mixed 16 sequences, geometric lengths (mean 1024) rescaled to 16384
                tokens, bs 32, Hk 8, Hq 32, fp16, any preset (default 4bit_nc)
    sweep       like llama3_8b at a given context (B*ctx ~ 1M tokens), any preset;
                q_heads / kv_heads change its head counts (e.g. groups of 16)
    """
    base_seed = {"tiny": 1001, "llama3_8b": 1002, "qwen3_32b": 1003, "long": 1004,
                 "store_mixed": 1005, "sweep": 1006}[name]
    seed = base_seed if seed is None else seed
    rng = np.random.default_rng(seed)
    D = 128
    if name == "tiny":
        B, Hq, Hk, bs, pre, dt = 1, 8, 2, 16, "turboquant_4bit_nc", "float16"
        seq = np.full(B, 512 if ctx is None else ctx, np.int32)
        bt, nb = _paging(seq, bs, rng, shuffle=False)
        w = Workload(name, B, Hq, Hk, D, bs, preset or pre, dt, seq, bt, nb, 0, seed,
                     "outliers")
        w.outlier_channels = np.sort(rng.choice(D, 4, replace=False)).astype(np.int64)
        return w
    if name in ("llama3_8b", "sweep"):
        B, Hq, Hk, bs, pre, dt = 32, 32, 8, 16, "turboquant_k8v4", "bfloat16"
        L = 8192
        if name == "sweep":
            L = ctx or 32768
            B = max(1, (1 << 20) // L)
            Hq, Hk = q_heads or Hq, kv_heads or Hk
        elif ctx is not None:
            L = ctx
        if batch is not None:
            B = batch
        seq = np.full(B, L, np.int32)
        bt, nb = _paging(seq, bs, rng, shuffle=True)
        w = Workload(name, B, Hq, Hk, D, bs, preset or pre, dt, seq, bt, nb, 0, seed,
                     "chanscale")
        w.chan_scale_k = np.exp(rng.uniform(np.log(0.25), np.log(4.0), (Hk, D))).astype(np.float32)
        w.chan_scale_v = np.exp(rng.uniform(np.log(0.25), np.log(4.0), (Hk, D))).astype(np.float32)
        return w
    if name == "qwen3_32b":
        B, Hq, Hk, bs, pre, dt = 64, 64, 8, 64, "turboquant_k3v4_nc", "float16"
        if batch is not None:
            B = batch
        seq = rng.integers(16384, 32768, size=B, endpoint=True).astype(np.int32)
        if ctx is not None:
            seq[:] = ctx
        bt, nb = _paging(seq, bs, rng, shuffle=True)
        return Workload(name, B, Hq, Hk, D, bs, preset or pre, dt, seq, bt, nb, 0, seed,
                        "heavytail")
    if name == "long":
        B, Hq, Hk, bs, pre, dt = 4, 32, 8, 128, "turboquant_3bit_nc", "bfloat16"
        if batch is not None:
            B = batch
        seq = np.full(B, 262144 if ctx is None else ctx, np.int32)
        bt, nb = _paging(seq, bs, rng, shuffle=True)
        w = Workload(name, B, Hq, Hk, D, bs, preset or pre, dt, seq, bt, nb, 64, seed,
                     "planted")
        w.plant_every = 4096
        return w
    if name == "store_mixed":
        Hq, Hk, bs, pre, dt = 32, 8, 32, "turboquant_4bit_nc", "float16"
        B, total = 16, 16384
        raw = rng.geometric(1.0 / 1024.0, size=B).astype(np.float64)
        seq = np.maximum(1, np.floor(raw / raw.sum() * total)).astype(np.int64)
        seq[np.argmax(seq)] += total - seq.sum()        # exact total
        seq = seq.astype(np.int32)
        bt, nb = _paging(seq, bs, rng, shuffle=True)
        return Workload(name, B, Hq, Hk, D, bs, preset or pre, dt, seq, bt, nb, 0, seed,
                        "normal")
    raise KeyError(name)


# ------------------------------------------------------------------ values
def _torch():
    import torch
    return torch


def _gen(device, seed: int):
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def torch_dtype(w: Workload):
    torch = _torch()
    return {"float16": torch.float16, "bfloat16": torch.bfloat16}[w.dtype]


def query_direction(w: Workload, b: int, device="cpu"):
    """Unit direction of the planted keys of sequence b, one per kv head (Hk, D)."""
    torch = _torch()
    g = _gen(device, w.seed * 7919 + 17 + b)
    d = torch.randn((w.Hk, w.D), generator=g, device=device, dtype=torch.float32)
    return d / d.norm(dim=-1, keepdim=True)


def gen_kv(w: Workload, b: int, t0: int, t1: int, device="cpu"):
    """K and V of tokens [t0, t1) of sequence b, each (t1-t0, Hk, D) in w.dtype.

    Draws are keyed by (seed, sequence, 4096-token chunk), so any sub-range
    of a sequence can be regenerated alone.
    """
    torch = _torch()
    n = t1 - t0
    ks, vs = [], []
    CH = 4096
    c0 = t0 // CH
    c1 = (t1 + CH - 1) // CH if n > 0 else c0
    for c in range(c0, c1):
        g = _gen(device, (w.seed * 1_000_003 + b) * 65_537 + c)
        k = torch.randn((CH, w.Hk, w.D), generator=g, device=device, dtype=torch.float32)
        v = torch.randn((CH, w.Hk, w.D), generator=g, device=device, dtype=torch.float32)
        if w.values == "heavytail":
            # 2% of coordinates replaced by Student-t(3) draws: z / sqrt(chi2_3 / 3)
            for x in (k, v):
                m = torch.rand(x.shape, generator=g, device=device) < 0.02
                z = torch.randn(x.shape, generator=g, device=device)
                chi = torch.randn((3,) + tuple(x.shape), generator=g, device=device).pow(2).sum(0)
                t = z / torch.sqrt(chi / 3.0)
                x.copy_(torch.where(m, t, x))
        ks.append(k)
        vs.append(v)
    if n <= 0:
        z = torch.zeros((0, w.Hk, w.D), device=device, dtype=torch_dtype(w))
        return z, z.clone()
    k = torch.cat(ks)[t0 - c0 * CH: t1 - c0 * CH]
    v = torch.cat(vs)[t0 - c0 * CH: t1 - c0 * CH]
    if w.values == "outliers":
        idx = torch.as_tensor(w.outlier_channels, device=device)
        k[:, :, idx] *= 8.0
        v[:, :, idx] *= 8.0
    elif w.values == "chanscale":
        k = k * torch.as_tensor(w.chan_scale_k, device=device)
        v = v * torch.as_tensor(w.chan_scale_v, device=device)
    elif w.values == "planted":
        pos = torch.arange(t0, t1, device=device)
        hit = (pos % w.plant_every) == (w.plant_every // 2)
        if bool(hit.any()):
            # k = alpha * q_dir * ||typical k||: logit ~ alpha*|q|*sqrt(D)/sqrt(D)
            dirs = query_direction(w, b, device)                 # (Hk, D)
            alpha = 1.1
            planted = alpha * math.sqrt(w.D) * dirs
            k[hit] = planted.unsqueeze(0).expand(int(hit.sum()), -1, -1)
    return k.to(torch_dtype(w)), v.to(torch_dtype(w))


def gen_q(w: Workload, device="cpu", step: int = 0):
    """Decode queries (B, Hq, D) in w.dtype."""
    torch = _torch()
    g = _gen(device, w.seed * 104_729 + 991 + step)
    q = torch.randn((w.B, w.Hq, w.D), generator=g, device=device, dtype=torch.float32)
    G = w.Hq // w.Hk
    if w.values == "outliers":
        idx = torch.as_tensor(w.outlier_channels, device=device)
        q[:, :, idx] *= 8.0
    elif w.values == "chanscale":
        sc = torch.as_tensor(w.chan_scale_k, device=device).repeat_interleave(G, dim=0)
        q = q * sc
    elif w.values == "planted":
        # every query head points at its kv head's planted direction, plus noise,
        # with |q| ~ sqrt(D): planted logits land around 10-15
        for b in range(w.B):
            dirs = query_direction(w, b, device).repeat_interleave(G, dim=0)
            q[b] = 0.35 * q[b] + math.sqrt(w.D) * dirs
    return q.to(torch_dtype(w))
