"""The CTA-pair split of the tensor-core GEMM: the two halves of K of each
output tile on the two CTAs of a thread-block cluster, partials added through
distributed shared memory.  Integer partial sums add exactly, so Y must be
bit-identical to the single-CTA engines; on shapes with ragged M and N tiles
(a partner half entirely past N included) and both tile widths."""
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
    (1024, 256, 2048),
    (300, 640, 1024),    # N = 2.5 x 256: the last tile's second half lies past N
    (1000, 384, 512),
    (129, 256, 8192),
    (257, 1000, 2048),
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


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_pair_split_is_bit_identical(modes, shape, bn):
    M, N, K = shape
    X, Q_W, s_W, img = _layer(M, N, K, seed=41)
    y_pair = _y(X, Q_W, s_W, img, 2, bn)
    y_one = _y(X, Q_W, s_W, img, 1, bn)
    diff = int((y_pair != y_one).sum())
    assert diff == 0, f"{diff} of {y_pair.size} outputs differ"


def test_pair_split_matches_oracle(modes):
    M, N, K = 1024, 2048, 2048
    seed = 42
    X = workloads.make_x(M, K, seed, workloads.n_outliers(K))
    prep = oracle.prepare_weight(workloads.make_w(N, K, seed))
    cr.convrot_set_split_mode(2)
    Y = gu.linear(X, prep["Q_W"], prep["s_W"], prep["Q_W"].astype(np.float16))
    rows = np.unique(np.concatenate([[0, M - 1],
                                     np.random.default_rng(seed).choice(M, 62, replace=False)]))
    ref = oracle.linear(X, prep["Q_W"], prep["s_W"], rows=rows)
    gu.compare_y(Y[rows], ref)


def test_pair_split_in_graph_replays(modes):
    # Back-to-back pair launches (and their cluster barriers) inside a graph.
    M, N, K = 1024, 2048, 2048
    X, Q_W, s_W, img = _layer(M, N, K, seed=43)
    cr.convrot_set_split_mode(1)
    ref = gu.linear(X, Q_W, s_W, img).view(np.uint16)
    cr.convrot_set_split_mode(2)
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


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("K", [2048, 4096])
def test_pair_split_extreme_codes(modes, bn, K):
    # All codes -128: each 1024-K chunk sums to exactly 2^24, the largest
    # value the fp32 accumulator holds exactly.  At K = 2048 each K half is
    # one chunk and the halves meet as exact fp32 values (2^24 + 2^24); at
    # K = 4096 they are added in int32.  Either way Y must equal the oracle's
    # epilogue of the exact product, and a mixed-sign pattern must too.
    M, N = 256, 512
    QX = np.full((M, K), -128, dtype=np.int8)
    QW = np.full((N, K), -128, dtype=np.int8)
    rng = np.random.default_rng(K + bn)
    flip = rng.random((M, K)) < 0.5
    QX2 = np.where(flip, np.int8(127), np.int8(-128)).astype(np.int8)
    sX = (rng.random(M) * 1e-6 + 1e-7).astype(np.float32)
    sW = (rng.random(N) * 1e-3).astype(np.float32)
    cr.convrot_set_split_mode(2)
    cr.convrot_set_tile_override(bn, 0)
    for qx in (QX, QX2):
        Y = gu.gemm_dequant(qx, sX, QW, sW, cr.CONVROT_PATH_TCGEN05)
        ref = oracle.epilogue_f32(oracle.int_gemm(qx, QW), sX, sW).astype(np.float16)
        diff = int((Y.view(np.uint16) != ref.view(np.uint16)).sum())
        assert diff == 0, f"{diff} of {Y.size} outputs differ"
