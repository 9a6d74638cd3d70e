"""The scan's epilogue evaluates some of its head-sum chains on doubled values: ReLU as
x + |x| (= 2 max(x, 0)) and the chain's pair sum halved at the end. These checks pin
the two facts the kernel relies on, in FP32 arithmetic on the host: x + |x| equals
2 max(x, 0) exactly for every finite x (negatives and -0 give +0), and a chain of fused
multiply-adds on doubled operands ends exactly twice the plain chain's value, so halving
it returns the plain chain's bits."""
import numpy as np


def _fma32(a, b, c):
    """fma rounded once to FP32: the product of two FP32 values is exact in FP64, and so is
    its sum with an FP32 value of similar scale here (magnitudes within 2^24 of each other)."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def test_x_plus_abs_x_is_twice_relu():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * np.float32(50),
                        np.array([0.0, -0.0, 1e-30, -1e-30, 3e37, -3e37], np.float32)])
    doubled = (x + np.abs(x)).astype(np.float32)
    plain = np.maximum(x, np.float32(0))
    assert np.array_equal((np.float32(2) * plain).view(np.uint32), doubled.view(np.uint32))
    assert not np.any(np.signbit(doubled))  # never -0


def test_doubled_chain_halves_to_the_plain_chain_bits():
    rng = np.random.default_rng(1)
    n, heads = 20000, 8
    w = (rng.standard_normal((heads, n)) / 8).astype(np.float32)
    x = (rng.standard_normal((heads, n)) * 11).astype(np.float32)
    p = np.zeros(n, np.float32)
    P = np.zeros(n, np.float32)
    for h in range(heads):
        p = _fma32(w[h], np.maximum(x[h], np.float32(0)), p)
        P = _fma32(w[h], (x[h] + np.abs(x[h])).astype(np.float32), P)
    assert np.array_equal((np.float32(2) * p).view(np.uint32), P.view(np.uint32))
    q = np.zeros(n, np.float32)  # a pair: (a + b) of plain chains against 0.5 (A + B) of doubled ones
    Q = (np.float32(0.5) * (P + P).astype(np.float32)).astype(np.float32)
    q = (p + p).astype(np.float32)
    assert np.array_equal(q.view(np.uint32), Q.view(np.uint32))
