"""The scan's epilogue evaluates each head-chain step fma(w, max(x, 0), p) as
fma(w / 2, x + |x|, p). These checks pin, in FP32 arithmetic on the host, the facts the
kernel relies on: x + |x| equals 2 max(x, 0) exactly for every finite x (negatives and -0
give +0); halving w is exact for w = 0 and |w| >= 2^-125; so the two forms multiply to the
same exact product and a chain of them gives the plain chain's bits at every step. Below
2^-125 halving can round (the smallest subnormal halves to zero), which is the one place
the forms can differ."""
import numpy as np


def _fma32(a, b, c):
    """fma rounded to FP32: the product of two FP32 values is exact in FP64. Both forms
    below reach this function with the same exact product and addend, so they round the
    same value whatever the emulation's own rounding."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def test_x_plus_abs_x_is_twice_relu():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * np.float32(50),
                        np.array([0.0, -0.0, 1e-30, -1e-30, 1e-45, -1e-45, 3e37, -3e37], np.float32)])
    doubled = (x + np.abs(x)).astype(np.float32)
    plain = np.maximum(x, np.float32(0))
    assert np.array_equal((np.float32(2) * plain).view(np.uint32), doubled.view(np.uint32))
    assert not np.any(np.signbit(doubled))  # never -0


def test_halving_is_exact_from_two_to_the_minus_125():
    rng = np.random.default_rng(2)
    mant = rng.uniform(1.0, 2.0, 50000)
    expo = rng.integers(-125, 127, 50000)
    w = (mant * np.exp2(expo.astype(np.float64))).astype(np.float32) * rng.choice([-1, 1], 50000).astype(np.float32)
    w = np.concatenate([w, np.array([0.0, -0.0, 2.0 ** -125, -(2.0 ** -125), 3.0e38], np.float32)])
    half = (np.float32(0.5) * w).astype(np.float32)
    assert np.array_equal((np.float32(2) * half).view(np.uint32), w.view(np.uint32))
    tiny = np.array([2.0 ** -149], np.float32)  # the smallest subnormal: halving rounds it away
    assert (np.float32(0.5) * tiny)[0] == 0.0


def test_halved_weight_chain_is_the_plain_chain():
    rng = np.random.default_rng(1)
    n, heads = 20000, 8
    w = (rng.standard_normal((heads, n)) / 8).astype(np.float32)
    x = (rng.standard_normal((heads, n)) * 11).astype(np.float32)
    w[:, :4] = np.array([0.0, -0.0, 2.0 ** -125, -1.5], np.float32)[:, None].T.repeat(heads, 0)
    x[:, 4:8] = np.array([0.0, -0.0, -3.0, 1e-30], np.float32)[:, None].T.repeat(heads, 0)
    p = np.zeros(n, np.float32)
    P = np.zeros(n, np.float32)
    for h in range(heads):
        p = _fma32(w[h], np.maximum(x[h], np.float32(0)), p)
        P = _fma32((np.float32(0.5) * w[h]).astype(np.float32), (x[h] + np.abs(x[h])).astype(np.float32), P)
        assert np.array_equal(p.view(np.uint32), P.view(np.uint32))
