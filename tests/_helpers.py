"""Shared helpers of the parity tests: oracle-side cache construction and the
acceptance checks (store bytes with counted boundary ties, fp16 norms within
one ulp, decode output and LSE tolerances)."""
from __future__ import annotations

import numpy as np

# Acceptance bars (the method's stated tolerances)
TIE_EPS = 1e-5           # |y - midpoint| below this may flip to the adjacent code
TIE_FRACTION = 1e-4      # at most this fraction of key codes may flip
OUT_MAX_ABS = 2e-3
OUT_REL_L2 = 1e-3
LSE_ABS = 1e-4


def f16_ulp(x: np.ndarray) -> np.ndarray:
    x = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0**-14)))
    return 2.0 ** (e - 10)


def to_f32(t) -> np.ndarray:
    """torch tensor (any float dtype, any device) -> exact float32 numpy."""
    return t.detach().float().cpu().numpy()


def codebook(orc, preset, D=128):
    L = orc.layout(preset, D)
    if L["key_fp8"]:
        return np.zeros(1, np.float32), np.zeros(1, np.float32)
    return orc.codebook(D, L["key_bits"])


def compare_store(orc, preset, gpu_rows, keys, values, signs, c32, m32):
    """gpu_rows: (M, slot) uint8 slots written by the GPU for M (token, head)
    pairs whose fp32 inputs are keys[M, D], values[M, D].  Checks each slot
    against the oracle.  Returns (number of flipped codes, number of codes)."""
    L = orc.layout(preset)
    M = gpu_rows.shape[0]
    flips = 0
    kd = L["key_data_bytes"]
    for i in range(M):
        ref, y = orc.store_one(preset, keys[i], values[i], signs, c32, m32)
        got = gpu_rows[i]
        # values, value metadata and padding: bit-exact
        assert np.array_equal(got[L["off_v_data"]:], ref[L["off_v_data"]:]), \
            f"value bytes differ at row {i}"
        if L["key_fp8"]:
            assert np.array_equal(got[:kd], ref[:kd]), f"fp8 key bytes differ at row {i}"
            continue
        cg = orc.unpack(got[:kd], 128, L["key_bits"])
        cr = orc.unpack(ref[:kd], 128, L["key_bits"])
        bad = np.nonzero(cg != cr)[0]
        for j in bad:
            lo = min(cg[j], cr[j])
            assert abs(int(cg[j]) - int(cr[j])) == 1, f"row {i} dim {j}: {cg[j]} vs {cr[j]}"
            assert abs(float(y[j]) - float(m32[lo])) < TIE_EPS, \
                f"row {i} dim {j}: flip away from a boundary ({y[j]} vs {m32[lo]})"
        flips += bad.size
        # norm: within one fp16 ulp of the oracle's, for the codes the GPU chose
        o = L["off_k_norm"]
        ng = orc.f16_value(int(got[o]) | int(got[o + 1]) << 8)
        if bad.size == 0:
            nr = orc.f16_value(int(ref[o]) | int(ref[o + 1]) << 8)
        else:
            kk = keys[i].astype(np.float64)
            nr = float(np.float16(np.linalg.norm(kk) / np.linalg.norm(c32[cg].astype(np.float64))))
        assert abs(ng - nr) <= f16_ulp(nr) * 1.0001, f"row {i}: norm {ng} vs {nr}"
    return flips, M * 128


def check_decode(out, lse, ref_out, ref_lse, what=""):
    """out/lse: GPU fp32 numpy; ref_*: oracle fp64."""
    out = np.asarray(out, np.float64)
    ref_out = np.asarray(ref_out, np.float64)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    err = np.abs(out - ref_out)
    mx = float(err.max()) if err.size else 0.0
    rel = float(np.linalg.norm(out - ref_out) / max(np.linalg.norm(ref_out), 1e-30))
    assert mx <= OUT_MAX_ABS, f"{what}: max-abs {mx}"
    assert rel <= OUT_REL_L2 or np.linalg.norm(ref_out) == 0, f"{what}: rel-L2 {rel}"
    if lse is not None:
        lse = np.asarray(lse, np.float64)
        ninf = np.isneginf(ref_lse)
        assert np.array_equal(np.isneginf(lse), ninf), f"{what}: -inf pattern"
        if (~ninf).any():
            le = float(np.abs(lse[~ninf] - ref_lse[~ninf]).max())
            assert le <= LSE_ABS, f"{what}: lse {le}"
    return mx, rel


def expected_kernel_kind(preset, G, Hk):
    """Which stage-1 kernel the library runs (1 tensor cores, 0 CUDA cores),
    restated from its documented rule: the tensor-core stage 1 serves every
    preset with G <= 16 (CTAs of up to 8 query heads per kv head); a CTA
    takes the token rows of 4 kv heads (FP8 keys, Hk a multiple of 4 above
    4) or of all Hk <= 16 heads; that part of a row must be whole 16-byte
    units, or, when the CTA takes whole rows, a multiple of 4 bytes (copied
    per page segment); and a two-stage ring of 32 such rows must fit in
    ~110 KB of shared memory."""
    slot = [196, 134, 118, 102, 70][preset]
    hpc = 4 if (preset == 0 and Hk % 4 == 0 and Hk > 4) else Hk
    row = hpc * slot
    rows_ok = row % 16 == 0 or (hpc == Hk and row % 4 == 0)
    return int(G <= 16 and hpc <= 16 and rows_ok and 2 * 32 * (row + 16) <= 110 * 1024)


def paged_problem(orc, preset, seq_lens, Hk, bs, rng, dtype="float16", kscale=1.0, book=None):
    """Random paged cache built by the ORACLE (fp16/bf16-exact inputs).
    `book`: (centroids, midpoints) to use instead of the Lloyd-Max codebook.
    Returns dict with cache (with a 0xFF guard block), block_table, K, V."""
    import torch
    D = 128
    L = orc.layout(preset)
    s = orc.signs(D, 42)
    c32, m32 = codebook(orc, preset) if book is None else book
    nblk = [(int(n) + bs - 1) // bs for n in seq_lens]
    total = sum(nblk)
    perm = rng.permutation(total)
    width = max(1, max(nblk)) + 1
    guard = total
    bt = np.full((len(seq_lens), width), guard, np.int32)
    cache = np.zeros((total + 1, bs, Hk, L["slot_size_aligned"]), np.uint8)
    cache[guard] = 0xFF
    tdt = {"float16": torch.float16, "bfloat16": torch.bfloat16}[dtype]
    Ks, Vs = [], []
    pos = 0
    for b, n in enumerate(seq_lens):
        bt[b, :nblk[b]] = perm[pos:pos + nblk[b]]
        pos += nblk[b]
        k = torch.from_numpy(rng.normal(size=(int(n), Hk, D)) * kscale).to(tdt)
        v = torch.from_numpy(rng.normal(size=(int(n), Hk, D))).to(tdt)
        Ks.append(k)
        Vs.append(v)
        if n:
            t = np.arange(int(n))
            sm = bt[b, t // bs].astype(np.int64) * bs + t % bs
            orc.store(preset, to_f32(k), to_f32(v), sm, cache, bs, s, c32, m32)
    return dict(cache=cache, bt=bt, K=Ks, V=Vs, signs=s, c32=c32, m32=m32, guard=guard)


def aos_to_soa(orc, preset, cache):
    """Re-arrange an AoS cache (num_blocks, bs, Hk, slot) into the SoA byte
    convention, written out from its definition: per block, a data region of
    [key data][value data] records, record (t, h) at index t*Hk + h, then a
    metadata region of uint16 [k_norm][v_scale][v_zero] records
    ([v_scale][v_zero] for FP8 keys) in the same order."""
    L = orc.layout(preset & 0xFF)
    nb, bs, Hk, S = cache.shape
    kd, vd = L["key_data_bytes"], L["value_data_bytes"]
    fields = ([L["off_v_scale"], L["off_v_zero"]] if L["key_fp8"]
              else [L["off_k_norm"], L["off_v_scale"], L["off_v_zero"]])
    out = np.zeros_like(cache).reshape(nb, -1)
    rec = cache.reshape(nb, bs * Hk, S)
    data = np.concatenate([rec[:, :, :kd], rec[:, :, L["off_v_data"]:L["off_v_data"] + vd]], axis=2)
    meta = np.concatenate([rec[:, :, f:f + 2] for f in fields], axis=2)
    db, mb = kd + vd, 2 * len(fields)
    out[:, :bs * Hk * db] = data.reshape(nb, -1)
    out[:, bs * Hk * db:bs * Hk * (db + mb)] = meta.reshape(nb, -1)
    return out.reshape(cache.shape)
