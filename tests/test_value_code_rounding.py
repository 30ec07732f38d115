"""The store's value code rint((v - z) / sc) without a division per code.

Warp-per-head kernel: q' = fl(t * fl(1/sc)) (t = fl(v - z)), with a fallback
to the correctly rounded quotient fl(t / sc) only when q' lies within 2^-16
of a half-integer.  Two-heads-per-warp kernel: r = rint(t * fl(1/sc)) of the
exact product (an FMA with 1.5 * 2^23), d = fl(t * fl(1/sc) - r) (an FMA),
and the same fallback when |d| > 1/2 - 2^-16.  For quotients below 16 the
approximations differ from the exact quotient by at most 2^-19, so outside
the window they round to the same integer, and above 16 all clamp to the
top code.  This restates both rules in numpy (float32 IEEE operations with
round-to-nearest-even like the kernel's _rn intrinsics; the exact product of
two float32 values held in float64) and checks them against the exact rule
on random inputs shaped like the store's and next to every half-integer
boundary.
"""
import numpy as np
import pytest

f32 = np.float32


def _exact(t, sc, qmax):
    q = (t / sc).astype(f32)
    return np.clip(np.rint(q), 0, qmax)


def _fast(t, sc, qmax):
    r = (f32(1) / sc).astype(f32)
    q = (t * r).astype(f32)
    near = np.abs(q - (np.floor(q) + f32(0.5))) < f32(2.0 ** -16)
    q = np.where(near, (t / sc).astype(f32), q)
    return np.clip(np.rint(q), 0, qmax), near


def _fast_fma(t, sc, qmax):
    r32 = np.where(sc > 0, f32(1) / np.where(sc > 0, sc, f32(1)), f32(0)).astype(f32)
    p = t.astype(np.float64) * r32.astype(np.float64)       # exact product of two float32
    r = np.rint(p)                                          # the FMA with 1.5 * 2^23: half to even
    d = (p - r).astype(f32)                                 # one rounding of an exact difference
    near = np.abs(d) > f32(0.5) - f32(2.0 ** -16)
    q = np.where(near, np.rint((t / np.where(sc > 0, sc, f32(1))).astype(f32)), r)
    return np.clip(q, 0, qmax), near


RULES = [lambda t, sc, qmax: _fast(t, sc, qmax), _fast_fma]


@pytest.mark.parametrize("rule", [0, 1])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_random_rows_like_the_store(bits, rule):
    qmax = 2 ** bits - 1
    rng = np.random.default_rng(4000 + bits)
    rows = rng.normal(size=(20000, 128)) * rng.uniform(0.01, 100, (20000, 1)) + rng.normal(size=(20000, 1)) * 10
    v = rows.astype(np.float16).astype(f32)
    lo, hi = v.min(1, keepdims=True), v.max(1, keepdims=True)
    sc = ((hi - lo) / f32(qmax)).astype(f32).astype(np.float16).astype(f32)
    z = lo.astype(np.float16).astype(f32)
    ok = (sc > 0)[:, 0]
    t = (v[ok] - z[ok]).astype(f32)
    e = _exact(t, sc[ok], qmax)
    f, _ = RULES[rule](t, sc[ok], qmax)
    assert np.array_equal(e, f)


@pytest.mark.parametrize("rule", [0, 1])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_next_to_every_boundary(bits, rule):
    """t placed a few float32 steps either side of (k + 1/2) * sc for every
    boundary k + 1/2 <= qmax + 1/2 and many fp16 scales: the exact rule and
    the fast rule agree, and the fallback is taken where it must be."""
    qmax = 2 ** bits - 1
    rng = np.random.default_rng(4100 + bits)
    sc = rng.uniform(1e-3, 50, 4000).astype(np.float16).astype(f32)
    sc = sc[sc > 0]
    k = np.arange(qmax + 1, dtype=f32) + f32(0.5)
    base = (k[None, :] * sc[:, None]).astype(f32)                 # (S, K)
    far = 2 ** np.arange(7, 15)
    steps = np.concatenate([np.arange(-40, 41), far, -far]).astype(np.int32)
    t = (base[..., None].view(np.int32) + steps[None, None, :]).view(f32)   # float32 steps from the boundary
    scb = np.broadcast_to(sc[:, None, None], t.shape)
    e = _exact(t, scb, qmax)
    f, near = RULES[rule](t, scb, qmax)
    assert np.array_equal(e, f)
    assert near.any() and not near.all()   # both branches are exercised
