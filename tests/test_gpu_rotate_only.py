"""convrot_rotate: the rotated activation X H alone, in fp16 (the activation
side of the weight-only W8A16 comparator).

The oracle's X H is exact in fp64 for fp16 inputs; the kernel sums in fp32
(8 butterfly stages) and rounds to fp16 once.  Each stage's fp32 rounding
is at most 2^-24 of a partial sum, and every partial sum is bounded by the
group's sum of |x| (times 1/16 at the end), so each output is within one
fp16 step plus 8 * 2^-24 * sum_group |x| / 16 of the correctly rounded
value (the second term matters only where the group's terms nearly cancel).
Nearly all outputs must be the correctly rounded value.  Unsupported shapes
are rejected.
"""
import numpy as np
import pytest

import oracle
import workloads
import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = gu.torch


def _f16_step(v: np.ndarray) -> np.ndarray:
    """The spacing of fp16 values at |v| (subnormal spacing below 2^-14)."""
    a = np.maximum(np.abs(v), 2.0 ** -14)
    return 2.0 ** (np.floor(np.log2(a)) - 10)


@pytest.mark.parametrize("shape", [(1024, 2048), (300, 256), (7, 8192), (64, 16384), (1, 1024)],
                         ids=lambda s: "x".join(map(str, s)))
def test_rotate_matches_oracle(shape):
    gu.require_gpu()
    M, K = shape
    X = workloads.make_x(M, K, 91, workloads.n_outliers(K))
    Xd = gu.dev(X)
    R = torch.empty((M, K), dtype=torch.float16, device="cuda")
    cr.convrot_rotate(Xd, R)
    gu.check_no_device_error()
    got = gu.host(R).astype(np.float64)
    exact = oracle.rotate(X.astype(np.float64))
    ref = exact.astype(np.float16).astype(np.float64)     # correctly rounded
    err = np.abs(got - ref)
    absx = np.abs(X.astype(np.float64)).reshape(M, K // 256, 256).sum(axis=2) / 16
    acc = 8 * 2.0 ** -24 * np.repeat(absx, 256, axis=1)
    bound = _f16_step(exact) + acc
    assert np.all(err <= bound), float((err - bound).max())
    assert np.mean(got == ref) > 0.999


def test_rotate_rejects_unsupported_shapes():
    gu.require_gpu()
    X = torch.zeros((4, 768), dtype=torch.float16, device="cuda")   # K / 64 = 12
    R = torch.empty_like(X)
    with pytest.raises(RuntimeError):
        cr.convrot_rotate(X, R)
