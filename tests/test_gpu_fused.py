"""The single-kernel engine of convrot_linear (rotate + quantize, grid
barrier and tensor-core product in one cooperative launch; selected with
convrot_set_fused).

* Y is bit-identical to the two-kernel engine's (same butterfly order, same
  rounding, same product) on shapes that reach every branch of the fused
  prologue: rows spanning 4 lanes up to 8 warps, fewer rows than CTAs,
  several passes per CTA, ragged tiles, direct (non-TMA) output stores, the
  weight widened per call.
* Y matches the oracle within the layer's tolerance.
* The grid barrier carries its state in the workspace from call to call:
  garbage-, zero- and 0xFF-filled workspaces, shapes alternating on one
  workspace, and CUDA graph replays with X changed between replays (a barrier
  that let a CTA through early would leave codes of the previous X).
"""
import numpy as np
import pytest

import oracle
import workloads
import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = gu.torch

# (M, N, K): K/64 = 4 .. 256 segments per row; M below, at and above the SM count.
SHAPES = [
    (1024, 2048, 2048),
    (17, 256, 256),
    (100, 512, 1024),
    (300, 77, 4096),     # N % 8 != 0: direct stores instead of TMA stores
    (2000, 640, 8192),   # a row spans 4 warps; several passes per CTA
    (64, 256, 16384),    # a row spans all 8 epilogue warps
    (1024, 6144, 256),
    (461, 384, 512),     # 3 * 152 + 5 rows: uneven shares
]


@pytest.fixture
def engines():
    gu.require_gpu()
    yield
    cr.convrot_set_fused(False)  # the default engine


def _layer(M, N, K, seed):
    X = workloads.make_x(M, K, seed, workloads.n_outliers(K))
    W = workloads.make_w(N, K, seed)
    Q_W, s_W, img = gu.prepare_weight(W)
    return gu.dev(X), Q_W, s_W, img


def _run(Xd, Q_W, s_W, img, ws, fused, Y=None):
    cr.convrot_set_fused(fused)
    M = Xd.shape[0]
    N = Q_W.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    cr.convrot_linear(Xd, Q_W, s_W, Y, ws, W_img=img)
    return Y


def _ws(M, N, K, with_img=True, fill=None):
    ws = gu.workspace(cr.convrot_linear_workspace_bytes(M, N, K, 0, with_img))
    if fill == "garbage":
        ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, device="cuda"))
    elif fill is not None:
        ws.fill_(fill)
    return ws


def _bits(Y):
    return gu.host(Y).view(np.uint16)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fused_is_bit_identical_to_two_kernels(engines, shape):
    M, N, K = shape
    Xd, Q_W, s_W, img = _layer(M, N, K, seed=11)
    ws = _ws(M, N, K, fill="garbage")
    yf = _bits(_run(Xd, Q_W, s_W, img, ws, True))
    gu.check_no_device_error()
    yu = _bits(_run(Xd, Q_W, s_W, img, ws, False))
    gu.check_no_device_error()
    diff = int((yf != yu).sum())
    assert diff == 0, f"{diff} of {yf.size} outputs differ between the engines"


def test_fused_without_weight_image(engines):
    M, N, K = 300, 512, 2048
    Xd, Q_W, s_W, img = _layer(M, N, K, seed=12)
    yu = _bits(_run(Xd, Q_W, s_W, img, _ws(M, N, K), False))
    yf = _bits(_run(Xd, Q_W, s_W, None, _ws(M, N, K, with_img=False, fill="garbage"), True))
    gu.check_no_device_error()
    assert np.array_equal(yf, yu)


@pytest.mark.parametrize("shape", [(1024, 2048, 2048), (100, 512, 1024), (64, 256, 16384)],
                         ids=lambda s: "x".join(map(str, s)))
def test_fused_matches_oracle(engines, shape):
    M, N, K = shape
    seed = 13
    X = workloads.make_x(M, K, seed, workloads.n_outliers(K))
    W = workloads.make_w(N, K, seed)
    prep = oracle.prepare_weight(W)
    cr.convrot_set_fused(True)
    Y = gu.linear(X, prep["Q_W"], prep["s_W"], prep["Q_W"].astype(np.float16))
    rows = np.arange(M) if M <= 128 else np.unique(
        np.concatenate([[0, M - 1], np.random.default_rng(seed).choice(M, 62, replace=False)]))
    ref = oracle.linear(X, prep["Q_W"], prep["s_W"], rows=rows)
    err = gu.compare_y(Y[rows], ref)
    print(f"fused {shape}: max |Y - Y_ref| = {err:.3g}")


@pytest.mark.parametrize("fill", ["garbage", 0, 255])
def test_workspace_state_across_calls_and_shapes(engines, fill):
    # One workspace, sized for the largest shape, shared by alternating shapes.
    shapes = [(1024, 2048, 2048), (17, 256, 256), (300, 77, 4096), (1024, 2048, 2048)]
    big = max(cr.convrot_linear_workspace_bytes(M, N, K, 0, True) for M, N, K in shapes)
    ws = gu.workspace(big)
    if fill == "garbage":
        ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, device="cuda"))
    else:
        ws.fill_(fill)
    for i, (M, N, K) in enumerate(shapes * 2):
        Xd, Q_W, s_W, img = _layer(M, N, K, seed=20 + i)
        yf = _bits(_run(Xd, Q_W, s_W, img, ws, True))
        gu.check_no_device_error()
        ref_ws = gu.workspace(cr.convrot_linear_workspace_bytes(M, N, K, 0, True))
        yu = _bits(_run(Xd, Q_W, s_W, img, ref_ws, False))
        assert np.array_equal(yf, yu), f"call {i} shape {(M, N, K)}"


def test_graph_replays_with_new_inputs(engines):
    layers = [(1024, 2048, 2048), (256, 640, 1024), (1024, 6144, 256)]
    ws = gu.workspace(max(cr.convrot_linear_workspace_bytes(M, N, K, 0, True)
                          for M, N, K in layers))
    bufs = []
    for i, (M, N, K) in enumerate(layers):
        Xd, Q_W, s_W, img = _layer(M, N, K, seed=30 + i)
        Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        bufs.append((Xd, Q_W, s_W, img, Y))
    cr.convrot_set_fused(True)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for Xd, Q_W, s_W, img, Y in bufs:  # eager first: settles the launch mode
            cr.convrot_linear(Xd, Q_W, s_W, Y, ws, W_img=img)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for Xd, Q_W, s_W, img, Y in bufs:
            cr.convrot_linear(Xd, Q_W, s_W, Y, ws, W_img=img)
    ref_ws = gu.workspace(ws.numel())
    for rep in range(4):
        for i, (Xd, *_rest) in enumerate(bufs):
            M, _, K = layers[i]
            Xd.copy_(gu.dev(workloads.make_x(M, K, 100 * rep + i, workloads.n_outliers(K))))
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        gu.check_no_device_error()
        for i, (Xd, Q_W, s_W, img, Y) in enumerate(bufs):
            yu = _bits(_run(Xd, Q_W, s_W, img, ref_ws, False))
            assert np.array_equal(_bits(Y), yu), f"replay {rep} layer {i}"
