"""The bytes the hot path's rotate + quantize step really writes.

convrot_linear_prologue leaves the activation codes and scales in the caller's
workspace (page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix, and
MLX", section "What changed in the computation": X_rot = X H, s_X =
max|X_rot| / 127, Q_X = round(X_rot / s_X) clamped to [-128, 127]): an fp16
image of the int8 codes for the tensor-core engines, int8 codes for the
small-M engine.  convrot_linear_workspace_layout says where.  Each code must
equal the oracle's exactly, except +-1 where the oracle's pre-round value
lies within 1e-4 of a .5 tie (counted), and s_X must agree to 1e-6 relative;
at the sweep's shapes (K = 2048, 256, 1024, 8192 at M = 1024) and at small M,
with ragged row counts.
"""
import numpy as np
import pytest

import oracle
import workloads
import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = gu.torch

CASES = [
    (1024, 2048, 2048),
    (1024, 256, 2048),
    (1024, 6144, 256),
    (1024, 2048, 1024),
    (1024, 8192, 2048),
    (1024, 2048, 8192),
    (1000, 2048, 4096),  # rows not a multiple of any tile
    (16, 8192, 2048),    # small M: int8 codes for the small-M engine
    (3, 2048, 8192),
]


@pytest.mark.parametrize("M,N,K", CASES, ids=lambda v: str(v))
def test_prologue_codes_and_scales_match_oracle(M, N, K):
    gu.require_gpu()
    X = workloads.make_x(M, K, seed=M + 7 * K, n_out=workloads.n_outliers(K))
    ws = gu.workspace(cr.convrot_linear_workspace_bytes(M, N, K, 0, True))
    ws.fill_(0xA5)  # garbage: every code and scale must be written
    cr.convrot_linear_prologue(gu.dev(X), N, ws, with_weight_image=True)
    gu.check_no_device_error()
    q_off, fmt, s_off = cr.convrot_linear_workspace_layout(M, N, K, 0, True)
    raw = gu.host(ws)
    if fmt == cr.CONVROT_CODES_F16:
        img = raw[q_off:q_off + 2 * M * K].view(np.float16).reshape(M, K).astype(np.float32)
        assert np.all(img == np.round(img)) and img.min() >= -128 and img.max() <= 127
        q = img.astype(np.int8)
    else:
        q = raw[q_off:q_off + M * K].view(np.int8).reshape(M, K)
    s = raw[s_off:s_off + 4 * M].view(np.float32)
    # Rows are independent: the oracle on a sample at the large sizes.
    rows = np.arange(M) if M * K <= (1 << 22) else np.unique(np.concatenate(
        [[0, M - 1], np.random.default_rng(K).choice(M, 96, replace=False)]))
    ref = oracle.rotate_quantize(X[rows])
    flips = gu.compare_q(q[rows], ref["Q_X"], ref["pre"])
    np.testing.assert_allclose(s[rows], ref["s_X"], rtol=1e-6, atol=0)
    print(f"M={M} K={K}: {flips} near-tie flips of {rows.size * K} codes "
          f"({'fp16 image' if fmt == cr.CONVROT_CODES_F16 else 'int8'})")
