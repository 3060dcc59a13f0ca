"""The streaming CTA-pair split of the tensor-core GEMM (gemm_pairk.cu): one
128 x 256 (or 128 x 128) output tile per 2-CTA cluster, each CTA one half of
K as a single exact fp32 chunk (K <= 2048), the partner's fp32 partial moved
from tensor memory through distributed shared memory and added on the way
out.  Each half is an exact integer of at most 2^24, so their fp32 sum is
(float)A and Y must be bit-identical to the single-CTA engine; on ragged M and
N tiles (a CTA's whole half past N included), K = 256 .. 2048, several waves
of clusters, the extreme codes, against the oracle, and inside graphs."""
import numpy as np
import pytest

import oracle
import workloads
import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = gu.torch

SHAPES = [
    (1024, 2048, 2048),
    (1024, 2048, 1024),
    (1024, 256, 2048),
    (300, 640, 1024),    # N = 2.5 x 256: the last tile's second half lies past N
    (1000, 384, 512),
    (129, 256, 256),     # one K block per half (BN = 256) / one stage (BN = 128)
    (257, 1000, 2048),
    (1024, 8192, 2048),  # 512 CTAs: several waves of clusters
]


@pytest.fixture
def modes():
    gu.require_gpu()
    yield
    cr.convrot_set_split_mode(0)
    cr.convrot_set_tile_override(0, 0)


def _layer(M, N, K, seed):
    X = workloads.make_x(M, K, seed, workloads.n_outliers(K))
    Q_W, s_W, img = gu.prepare_weight(workloads.make_w(N, K, seed))
    return X, Q_W, s_W, img


def _y(X, Q_W, s_W, img, split_mode, bn=0):
    cr.convrot_set_split_mode(split_mode)
    cr.convrot_set_tile_override(bn, 0)
    return gu.linear(X, Q_W, s_W, img).view(np.uint16)


def test_planner_takes_the_stream_engine_when_forced(modes):
    cr.convrot_set_split_mode(3)
    for bn in (128, 256):
        cr.convrot_set_tile_override(bn, 0)
        assert cr.convrot_plan_gemm(1024, 2048, 2048) == (bn, 2, cr.CONVROT_ENGINE_PAIR_STREAM)
    # K beyond 2048 (two chunks per half): another engine.
    assert cr.convrot_plan_gemm(1024, 2048, 4096)[2] != cr.CONVROT_ENGINE_PAIR_STREAM


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_stream_split_is_bit_identical(modes, shape, bn):
    M, N, K = shape
    X, Q_W, s_W, img = _layer(M, N, K, seed=51)
    y_stream = _y(X, Q_W, s_W, img, 3, bn)
    gu.check_no_device_error()
    y_one = _y(X, Q_W, s_W, img, 1, 128)
    diff = int((y_stream != y_one).sum())
    assert diff == 0, f"{diff} of {y_stream.size} outputs differ"


def test_stream_split_matches_oracle(modes):
    M, N, K = 1024, 2048, 2048
    seed = 52
    X = workloads.make_x(M, K, seed, workloads.n_outliers(K))
    prep = oracle.prepare_weight(workloads.make_w(N, K, seed))
    cr.convrot_set_split_mode(3)
    Y = gu.linear(X, prep["Q_W"], prep["s_W"], prep["Q_W"].astype(np.float16))
    rows = np.unique(np.concatenate([[0, M - 1],
                                     np.random.default_rng(seed).choice(M, 62, replace=False)]))
    ref = oracle.linear(X, prep["Q_W"], prep["s_W"], rows=rows)
    gu.compare_y(Y[rows], ref)


@pytest.mark.parametrize("bn", [128, 256])
def test_stream_split_extreme_codes(modes, bn):
    # All codes -128 at K = 2048: each K half sums to exactly 2^24, the largest
    # value the fp32 accumulator holds exactly, and the halves meet as
    # 2^24 + 2^24.  A mixed-sign pattern too.  Y must equal the oracle's
    # epilogue of the exact product.
    M, N, K = 256, 512, 2048
    QX = np.full((M, K), -128, dtype=np.int8)
    QW = np.full((N, K), -128, dtype=np.int8)
    rng = np.random.default_rng(bn)
    QX2 = np.where(rng.random((M, K)) < 0.5, np.int8(127), np.int8(-128)).astype(np.int8)
    QW2 = np.where(rng.random((N, K)) < 0.3, np.int8(-128), np.int8(127)).astype(np.int8)
    sX = (rng.random(M) * 1e-6 + 1e-7).astype(np.float32)
    sW = (rng.random(N) * 1e-3).astype(np.float32)
    cr.convrot_set_split_mode(3)
    cr.convrot_set_tile_override(bn, 0)
    for qx, qw in ((QX, QW), (QX2, QW), (QX2, QW2)):
        Y = gu.gemm_dequant(qx, sX, qw, sW, cr.CONVROT_PATH_TCGEN05)
        ref = oracle.epilogue_f32(oracle.int_gemm(qx, qw), sX, sW).astype(np.float16)
        diff = int((Y.view(np.uint16) != ref.view(np.uint16)).sum())
        assert diff == 0, f"{diff} of {Y.size} outputs differ"


def test_stream_split_in_graph_replays(modes):
    # Back-to-back launches (and their cluster hand-offs) inside a graph.
    M, N, K = 1024, 2048, 2048
    X, Q_W, s_W, img = _layer(M, N, K, seed=53)
    cr.convrot_set_split_mode(1)
    ref = gu.linear(X, Q_W, s_W, img).view(np.uint16)
    cr.convrot_set_split_mode(3)
    Xd = gu.dev(X)
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = gu.workspace(cr.convrot_linear_workspace_bytes(M, N, K, 0, True))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        cr.convrot_linear(Xd, Q_W, s_W, Y, ws, W_img=img)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(4):
            cr.convrot_linear(Xd, Q_W, s_W, Y, ws, W_img=img)
    for _ in range(3):
        Y.zero_()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        gu.check_no_device_error()
        assert np.array_equal(gu.host(Y).view(np.uint16), ref)
