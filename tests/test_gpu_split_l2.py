"""Split K through L2: each split of an output tile adds its exact int32
partial into the workspace accumulator with TMA bulk reduce-adds, and the
tile's last split loads the sum back, writes Y and leaves the tile and its
counter zero.  In convrot_linear (and convrot_linear_prologue) the rotate +
quantize kernel zeroes the accumulator and its tile counters on the way; the
GEMM entry points on caller operands zero them with memsets.

Integer partials add exactly, so Y must be bit-identical to the unsplit
engine and to the oracle's epilogue: every tile width and split count,
ragged M, N and K splits, more units than SMs (several per CTA), a
garbage-filled workspace, the same workspace reused across calls and shapes,
and CUDA graph replays.
"""
import numpy as np
import pytest

import oracle
import workloads
import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = gu.torch

TC = cr.CONVROT_PATH_TCGEN05


@pytest.fixture
def modes():
    gu.require_gpu()
    # Splits only: neither CTA-pair engine.
    cr.convrot_set_split_mode(1)
    cr.convrot_set_pair_mma(1)
    yield
    cr.convrot_set_split_mode(0)
    cr.convrot_set_pair_mma(0)
    cr.convrot_set_tile_override(0, 0)


def _rand(M, N, K, seed):
    rng = np.random.default_rng(seed)
    QX = rng.integers(-128, 128, (M, K), dtype=np.int8)
    QW = rng.integers(-128, 128, (N, K), dtype=np.int8)
    return QX, QW


SPLITS = [(64, 4), (64, 16), (128, 2), (128, 3), (256, 2), (256, 5)]
GEMM_SHAPES = [(200, 264, 2048), (1024, 256, 2048), (129, 320, 3072), (512, 2560, 1024)]


@pytest.mark.parametrize("bn,splits", SPLITS, ids=lambda v: str(v))
@pytest.mark.parametrize("shape", GEMM_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_split_dequant_bit_exact(modes, shape, bn, splits):
    M, N, K = shape
    cr.convrot_set_tile_override(bn, splits)
    QX, QW = _rand(M, N, K, seed=M + 7 * N + K)
    rng = np.random.default_rng(M * N)
    sX = (rng.random(M) * 0.1).astype(np.float32)
    sW = (rng.random(N) * 0.01).astype(np.float32)
    Y = gu.gemm_dequant(QX, sX, QW, sW, TC)
    ref = oracle.epilogue_f32(oracle.int_gemm(QX, QW), sX, sW).astype(np.float16)
    diff = int((Y.view(np.uint16) != ref.view(np.uint16)).sum())
    assert diff == 0, f"{diff} of {Y.size} outputs differ"


def _layer(M, N, K, seed):
    X = workloads.make_x(M, K, seed, workloads.n_outliers(K))
    Q_W, s_W, img = gu.prepare_weight(workloads.make_w(N, K, seed))
    return gu.dev(X), Q_W, s_W, img


def _linear(Xd, Q_W, s_W, img, ws, bn, splits):
    cr.convrot_set_tile_override(bn, splits)
    M, N = Xd.shape[0], Q_W.shape[0]
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    cr.convrot_linear(Xd, Q_W, s_W, Y, ws, W_img=img)
    gu.check_no_device_error()
    return gu.host(Y).view(np.uint16)


LINEAR_SHAPES = [(1024, 256, 2048), (300, 640, 1024), (1024, 2048, 2048), (129, 384, 8192)]


@pytest.mark.parametrize("bn,splits", [(64, 4), (128, 2), (256, 2), (128, 8)], ids=lambda v: str(v))
@pytest.mark.parametrize("shape", LINEAR_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_split_linear_zeroed_by_prologue(modes, shape, bn, splits):
    M, N, K = shape
    Xd, Q_W, s_W, img = _layer(M, N, K, seed=61)
    ws = gu.workspace(cr.convrot_linear_workspace_bytes(M, N, K, 0, True))
    ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, device="cuda"))  # garbage
    y1 = _linear(Xd, Q_W, s_W, img, ws, bn, splits)
    y2 = _linear(Xd, Q_W, s_W, img, ws, bn, splits)  # the same workspace again
    ref = _linear(Xd, Q_W, s_W, img, gu.workspace(ws.numel()), 128, 1)
    assert np.array_equal(y1, ref)
    assert np.array_equal(y2, ref)


def test_split_linear_matches_oracle(modes):
    M, N, K = 1024, 256, 2048
    seed = 62
    X = workloads.make_x(M, K, seed, workloads.n_outliers(K))
    prep = oracle.prepare_weight(workloads.make_w(N, K, seed))
    cr.convrot_set_tile_override(64, 4)
    Y = gu.linear(X, prep["Q_W"], prep["s_W"], prep["Q_W"].astype(np.float16))
    rows = np.unique(np.concatenate([[0, M - 1],
                                     np.random.default_rng(seed).choice(M, 62, replace=False)]))
    ref = oracle.linear(X, prep["Q_W"], prep["s_W"], rows=rows)
    gu.compare_y(Y[rows], ref)


def test_split_linear_graph_replays(modes):
    # Split layers of different shapes sharing one workspace inside a graph:
    # each layer's prologue must re-zero the accumulator the previous
    # layer's GEMM left holding its sums.
    layers = [(1024, 256, 2048), (300, 640, 1024), (1024, 256, 2048)]
    ws = gu.workspace(max(cr.convrot_linear_workspace_bytes(M, N, K, 0, True)
                          for M, N, K in layers))
    bufs = []
    for i, (M, N, K) in enumerate(layers):
        Xd, Q_W, s_W, img = _layer(M, N, K, seed=70 + i)
        bufs.append((Xd, Q_W, s_W, img, torch.empty((M, N), dtype=torch.float16, device="cuda")))
    cr.convrot_set_tile_override(64, 4)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for Xd, Q_W, s_W, img, Y in bufs:
            cr.convrot_linear(Xd, Q_W, s_W, Y, ws, W_img=img)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for Xd, Q_W, s_W, img, Y in bufs:
            cr.convrot_linear(Xd, Q_W, s_W, Y, ws, W_img=img)
    refs = [_linear(Xd, Q_W, s_W, img, gu.workspace(ws.numel()), 128, 1)
            for Xd, Q_W, s_W, img, _ in bufs]
    cr.convrot_set_tile_override(64, 4)
    for rep in range(3):
        for _, _, _, _, Y in bufs:
            Y.zero_()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        gu.check_no_device_error()
        for i, (_, _, _, _, Y) in enumerate(bufs):
            assert np.array_equal(gu.host(Y).view(np.uint16), refs[i]), (rep, i)


@pytest.mark.parametrize("bn,splits", [(64, 4), (128, 2)], ids=lambda v: str(v))
def test_split_two_stage_api_repeated_gemm(modes, bn, splits):
    # convrot_linear_prologue zeroes the accumulator (whatever the workspace
    # held); each split GEMM leaves it zero, so the GEMM stage may run again.
    M, N, K = 1024, 256, 2048
    Xd, Q_W, s_W, img = _layer(M, N, K, seed=63)
    ws = gu.workspace(cr.convrot_linear_workspace_bytes(M, N, K, 0, True))
    ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, device="cuda"))
    ref = _linear(Xd, Q_W, s_W, img, gu.workspace(ws.numel()), 128, 1)
    cr.convrot_set_tile_override(bn, splits)
    cr.convrot_linear_prologue(Xd, N, ws, with_weight_image=True)
    for rep in range(3):
        Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        cr.convrot_linear_gemm(M, K, Q_W, s_W, Y, ws, W_img=img)
        gu.check_no_device_error()
        assert np.array_equal(gu.host(Y).view(np.uint16), ref), rep
