"""Index arithmetic past 2^31 elements (the PR page "[PR #249] Add an mps
backend: weight-only INT8 and W4A8/W6A8 linears for Apple GPUs", section "How
tested", checks its kernels' index arithmetic past 2^32).

  * M = 131328, N = 16384, K = 256: Y has 2^31 + 2^22 elements, and its last
    256 rows start at or beyond element 2^31 (4.3 GB of fp16);
  * M = 2^23 + 2^15, N = 64, K = 256: X and the activation codes have more
    than 2^31 elements (4.3 GB each).
Sampled rows -- the first, the last and rows on both sides of the 2^31
boundary -- against the oracle within the layer tolerance.  The large
activation is drawn on the device from a seeded torch generator (distinct
rows everywhere), and the sampled rows are copied back for the oracle.
"""
import math

import numpy as np
import pytest

import oracle
import workloads
import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = gu.torch


def _need(nbytes):
    free, _ = torch.cuda.mem_get_info()
    if free < nbytes * 1.2:
        pytest.skip(f"needs {nbytes / 1e9:.1f} GB of free device memory")


def _x_device(M, K, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    X = torch.empty((M, K), dtype=torch.float16, device="cuda")
    step = 1 << 20
    for r0 in range(0, M, step):
        r1 = min(M, r0 + step)
        X[r0:r1] = torch.randn((r1 - r0, K), generator=g, device="cuda").half()
    return X


@pytest.mark.parametrize("M,N,K", [(131328, 16384, 256), ((1 << 23) + (1 << 15), 64, 256)])
def test_layer_past_2_31_elements(M, N, K):
    gu.require_gpu()
    ws_bytes = cr.convrot_linear_workspace_bytes(M, N, K, 0, True)
    _need(2 * M * K + 2 * M * N + ws_bytes + 4 * N * K)
    X = _x_device(M, K, seed=M)
    prep = oracle.prepare_weight(workloads.make_w(N, K, seed=N))
    Q_W, s_W = gu.dev(prep["Q_W"]), gu.dev(prep["s_W"])
    img = gu.dev(prep["Q_W"].astype(np.float16))
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = gu.workspace(ws_bytes)
    cr.convrot_linear(X, Q_W, s_W, Y, ws, W_img=img)
    gu.check_no_device_error()
    # Rows whose first output element lies just below / above 2^31, and the
    # same for the first activation element.
    edge_y = (1 << 31) // N
    edge_x = (1 << 31) // K
    rows = {0, M - 1, M - 2, M // 2}
    for e in (edge_y, edge_x):
        rows.update(r for r in (e - 2, e - 1, e, e + 1, e + 2) if 0 <= r < M)
    rows.update(np.random.default_rng(M).choice(M, 24, replace=False).tolist())
    rows = np.array(sorted(rows))
    sel = torch.from_numpy(rows).cuda()
    xs = gu.host(X.index_select(0, sel))
    ys = gu.host(Y.index_select(0, sel))
    ref = oracle.linear(xs, prep["Q_W"], prep["s_W"])
    gu.compare_y(ys, ref)
    assert math.isfinite(float(np.abs(ys.astype(np.float64)).max()))
    del X, Y, ws
