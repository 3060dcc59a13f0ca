"""The entry point that allocates nothing (convrot_linear_noalloc).

It serves callers that can neither pass a workspace nor allocate device
memory -- plugin hosts that give a layer no scratch buffer, engines that
forbid cudaMalloc once running -- by using a fixed scratch array inside the
library.  Its output must agree with the regular convrot_linear (which takes
a caller workspace) within the tolerance the layer tests use, and with the
oracle, on two calls in a row (the second call reuses the scratch the first
one left behind).  This file is collected last so that a run which stops at
the first failure has already run every other test.
"""
import numpy as np
import pytest

import oracle
import workloads
import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu

pytestmark = pytest.mark.gpu


def _noalloc(X, Q_W, s_W):
    torch = gu.torch
    M = X.shape[0]
    N = Q_W.shape[0]
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    cr.convrot_linear_noalloc(gu.dev(X), gu.dev(Q_W), gu.dev(s_W), Y)
    gu.check_no_device_error()
    return gu.host(Y)


# (16, 70000, 256): many columns at the largest M -- the scratch holds only
# the codes and scales, so the width of the weight does not count against it.
@pytest.mark.parametrize("M,N,K", [(1, 8192, 2048), (16, 2048, 8192), (3, 80, 768),
                                   (16, 70000, 256)])
def test_noalloc_matches_linear_and_oracle_on_two_calls(M, N, K):
    gu.require_gpu()
    W = workloads.make_w(N, K, seed=M + K)
    prep = oracle.prepare_weight(W)
    for call in range(2):
        X = workloads.make_x(M, K, seed=100 * call + M, n_out=workloads.n_outliers(K))
        y_lin = gu.linear(X, prep["Q_W"], prep["s_W"])
        y = _noalloc(X, prep["Q_W"], prep["s_W"])
        np.testing.assert_allclose(y.astype(np.float64), y_lin.astype(np.float64),
                                   rtol=1e-3, atol=1e-3)
        gu.compare_y(y, oracle.linear(X, prep["Q_W"], prep["s_W"]))


def test_noalloc_rejects_rows_beyond_its_limit():
    gu.require_gpu()
    torch = gu.torch
    K, N = 256, 64
    X = torch.zeros((cr.CONVROT_NOALLOC_MAX_M + 1, K), dtype=torch.float16, device="cuda")
    Q = torch.zeros((N, K), dtype=torch.int8, device="cuda")
    s = torch.zeros((N,), dtype=torch.float32, device="cuda")
    Y = torch.empty((X.shape[0], N), dtype=torch.float16, device="cuda")
    with pytest.raises(cr.ConvRotError) as e:
        cr.convrot_linear_noalloc(X, Q, s, Y)
    assert e.value.status == cr.CONVROT_ERR_WORKSPACE
