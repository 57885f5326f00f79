"""The split form of fp32 operands used on the tensor cores (kernels_rows.cu
split3_kernel, kernels_tc.cu emit_dlogits_split): x = hi + mid + lo with
hi = bf16(x), mid = bf16(x - hi), lo = bf16(x - hi - mid), all roundings to
nearest even, every difference taken in fp32.

Pinned here on the host (the arithmetic, not the kernel, which the fp32
parity tests check against the fp64 oracle):
  * the three parts reproduce x exactly, and the last remainder needs no
    rounding (it fits bf16's 8 significant bits);
  * the part products the kernels drop (mid.lo, lo.mid, lo.lo) come to at
    most about 2^-23 of |x y|, while each kept small one (hi.lo, lo.hi,
    mid.mid) can reach 2^-16 of it, so none of the six could be dropped.
"""
import numpy as np
import pytest


def bf16_rne(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest, ties to even) -> fp32, by bit operations."""
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def split3(x: np.ndarray):
    x = x.astype(np.float32)
    hi = bf16_rne(x)
    r1 = (x - hi).astype(np.float32)
    mid = bf16_rne(r1)
    r2 = (r1 - mid).astype(np.float32)
    lo = bf16_rne(r2)
    return hi, mid, lo, r2


def _samples(seed, n=200_000):
    g = np.random.default_rng(seed)
    mant = g.uniform(1.0, 2.0, n)
    expo = g.integers(-100, 100, n)
    sign = g.choice([-1.0, 1.0], n)
    return (sign * mant * np.exp2(expo)).astype(np.float32)


@pytest.mark.parametrize("seed", [0, 1])
def test_parts_are_exact(seed):
    x = _samples(seed)
    hi, mid, lo, r2 = split3(x)
    assert np.array_equal(lo, r2), "the last remainder must fit bf16 exactly"
    recon = hi.astype(np.float64) + mid.astype(np.float64) + lo.astype(np.float64)
    assert np.array_equal(recon, x.astype(np.float64))


def test_parts_of_special_values():
    x = np.array([0.0, -0.0, 1.0, -1.0, 3.0, 1e-30, -1e30, 2.0 ** -126, 2.0 ** 127,
                  np.float32(1.0) + np.float32(2.0 ** -23)], dtype=np.float32)
    hi, mid, lo, r2 = split3(x)
    assert np.array_equal(lo, r2)
    recon = hi.astype(np.float64) + mid.astype(np.float64) + lo.astype(np.float64)
    assert np.array_equal(recon, x.astype(np.float64))


def test_dropped_products_bound():
    x, y = _samples(2, 100_000), _samples(3, 100_000)
    xs, ys = split3(x)[:3], split3(y)[:3]
    prod = np.abs(x.astype(np.float64) * y.astype(np.float64))
    dropped = (np.abs(xs[1].astype(np.float64) * ys[2]) + np.abs(xs[2].astype(np.float64) * ys[1])
               + np.abs(xs[2].astype(np.float64) * ys[2]))
    assert float(np.max(dropped / prod)) <= 2.0 ** -23 * 1.01
    # the kept six give x*y to that bound; each of the small kept ones is needed
    kept = sum(xs[i].astype(np.float64) * ys[j] for i, j in
               [(0, 0), (0, 1), (1, 0), (0, 2), (2, 0), (1, 1)])
    assert float(np.max(np.abs(kept - x.astype(np.float64) * y) / prod)) <= 2.0 ** -23 * 1.01
    small_kept = np.maximum.reduce([np.abs(xs[0].astype(np.float64) * ys[2]),
                                    np.abs(xs[2].astype(np.float64) * ys[0]),
                                    np.abs(xs[1].astype(np.float64) * ys[1])])
    assert float(np.max(small_kept / prod)) > 2.0 ** -20


def test_planted_mistake_is_caught():
    """Taking mid without subtracting hi first would not reproduce x."""
    x = _samples(4, 10_000)
    hi = bf16_rne(x)
    mid_wrong = bf16_rne(x)  # the mistake: the remainder is not formed
    lo = bf16_rne((x - hi - mid_wrong).astype(np.float32))
    recon = hi.astype(np.float64) + mid_wrong + lo
    assert not np.array_equal(recon, x.astype(np.float64))
