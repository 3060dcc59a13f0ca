"""Parity of the rotate+quantize step (CUDA) with the oracle.

Q_X must match exactly except +-1 where the oracle's pre-round value lies
within 1e-4 of a .5 tie (the kernel rotates in fp32, the oracle exactly), and
s_X to 1e-6 relative.  Sizes cover the TMA tile kernel (K/64 a power of two up
to 16384), the two-pass row kernel (other K), ragged M and the degenerate rows.
"""
import numpy as np
import pytest

import oracle
import workloads

from . import gpu_util as gu

pytestmark = pytest.mark.gpu

# Small problems take the 32-values-per-lane variant of the tile kernel in
# 4-warp tiles; rows of up to 1024 values beyond that the same in one-warp
# tiles; the other large ones the 64-values-per-lane one; K that is not 256
# times a power of two, or above 16384, the two-pass row kernel.
SHAPES = [(64, 256), (37, 256), (1, 256), (130, 512), (37, 1024), (1024, 2048),
          (33, 4096), (9, 8192), (5, 16384), (7, 768), (3, 20480), (2, 65536),
          (1300, 2048), (10000, 256), (1024, 256), (609, 256), (701, 256),
          (1024, 1024), (700, 512), (3000, 1024)]


@pytest.mark.parametrize("M,K", SHAPES)
def test_rotate_quantize_matches_oracle(M, K):
    gu.require_gpu()
    X = workloads.make_x(M, K, seed=7 * M + K)
    q, s = gu.rotate_quantize(X)
    ref = oracle.rotate_quantize(X)
    flips = gu.compare_q(q, ref["Q_X"], ref["pre"])
    np.testing.assert_allclose(s, ref["s_X64"], rtol=1e-6, atol=0)
    print(f"M={M} K={K}: {flips} near-tie flips of {q.size}")


@pytest.mark.parametrize("K", [256, 2048, 768])
def test_degenerate_rows(K):
    gu.require_gpu()
    X = workloads.make_x(6, K, seed=K)
    X[0] = 0                                    # zero row -> s = 0, Q = 0
    X[1] = 0
    X[1, 3] = np.float16(2.0)                   # delta: |X_rot| equal everywhere
    X[2] = np.float16(65504.0)                  # fp16 max
    X[3] = (X[3].astype(np.float32) * np.float32(1e-6)).astype(np.float16)  # subnormal range
    X[4] = -X[4]
    q, s = gu.rotate_quantize(X)
    ref = oracle.rotate_quantize(X)
    gu.compare_q(q, ref["Q_X"], ref["pre"])
    np.testing.assert_allclose(s, ref["s_X64"], rtol=1e-6, atol=0)
    assert s[0] == 0 and np.all(q[0] == 0)
    # The delta's own 256-group rotates to +-2/16 everywhere (codes +-127);
    # the other groups of that row are zero.
    assert np.all(np.abs(q[1, :256].astype(int)) == 127)
    assert np.all(q[1, 256:] == 0)


@pytest.mark.parametrize("K", [256, 1024, 768])
def test_exact_ties_round_half_even(K):
    # X = v H with v sparse half-integers and max |v| = 127: every X entry is
    # a multiple of 1/32 below 64 (exact in fp16) and the rotation back is
    # exact in fp32, so X_rot = v exactly and the codes must equal
    # round-half-even(v) with no tie allowance.
    gu.require_gpu()
    rng = np.random.default_rng(K)
    H = oracle.hadamard256()
    v = np.zeros((4, K))
    for r in range(4):
        for g in range(K // 256):
            idx = rng.choice(256, size=40, replace=False) + 256 * g
            v[r, idx] = rng.choice([-3.5, -2.5, -1.5, -0.5, 0.5, 1.5, 2.5, 3.5], size=40)
    v[:, 0] = 127.0
    X64 = np.concatenate([v[:, g * 256:(g + 1) * 256] @ H for g in range(K // 256)], axis=1)
    X = X64.astype(np.float16)
    assert np.array_equal(X.astype(np.float64), X64)
    q, s = gu.rotate_quantize(X)
    ref = oracle.rotate_quantize(X)
    np.testing.assert_array_equal(q, ref["Q_X"])
    assert np.all(s == np.float32(1.0))
    assert (np.abs(v - np.trunc(v)) == 0.5).sum() > 100  # the test has ties to decide
