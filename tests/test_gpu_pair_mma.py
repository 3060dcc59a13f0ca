"""GEMM tiles on CTA-pair MMAs (tcgen05 .cta_group::2): a 256 x BN output
tile computed by the two CTAs of a thread-block cluster, each SM holding 128
rows of A and of the output and half of the tile's weight rows.  The product
is the same exact integer sum, so Y must be bit-identical to the one-SM
engine's; on shapes with ragged M (the odd CTA's rows partly or wholly past
M), ragged N (the odd CTA's weight rows past N), one or many fp32 chunks of K,
fewer K blocks than ring stages, and several units per cluster.  Also against
the oracle, and in CUDA graph replays."""
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
    (1024, 8192, 2048),  # more units than clusters: several per cluster
    (300, 640, 1024),    # M = 256 + 44, N = 2.5 x 256
    (100, 256, 512),     # M < 128: the odd CTA's rows all past M
    (2048, 1024, 8192),  # 8 fp32 chunks: int32 partials, then the fp32 switch
    (129, 384, 256),     # 4 K blocks: fewer than the ring's stages
    (4096, 2048, 1024),
]


@pytest.fixture
def modes():
    gu.require_gpu()
    yield
    cr.convrot_set_pair_mma(0)
    cr.convrot_set_tile_override(0, 0)


def _layer(M, N, K, seed):
    X = workloads.make_x(M, K, seed, workloads.n_outliers(K))
    Q_W, s_W, img = gu.prepare_weight(workloads.make_w(N, K, seed))
    return X, Q_W, s_W, img


def _y(X, Q_W, s_W, img, mode, bn=0):
    cr.convrot_set_pair_mma(mode)
    cr.convrot_set_tile_override(bn, 0)
    y = gu.linear(X, Q_W, s_W, img).view(np.uint16)
    gu.check_no_device_error()
    return y


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_pair_mma_is_bit_identical(modes, shape, bn):
    M, N, K = shape
    X, Q_W, s_W, img = _layer(M, N, K, seed=51)
    y_pair = _y(X, Q_W, s_W, img, 2, bn)
    y_one = _y(X, Q_W, s_W, img, 1, bn)
    diff = int((y_pair != y_one).sum())
    assert diff == 0, f"{diff} of {y_pair.size} outputs differ"


@pytest.mark.parametrize("bn", [128, 256])
def test_pair_mma_matches_oracle(modes, bn):
    M, N, K = 1024, 2048, 2048
    seed = 52
    X = workloads.make_x(M, K, seed, workloads.n_outliers(K))
    prep = oracle.prepare_weight(workloads.make_w(N, K, seed))
    cr.convrot_set_pair_mma(2)
    cr.convrot_set_tile_override(bn, 0)
    Y = gu.linear(X, prep["Q_W"], prep["s_W"], prep["Q_W"].astype(np.float16))
    gu.check_no_device_error()
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, M - 1],
                                     np.random.default_rng(seed).choice(M, 58, replace=False)]))
    ref = oracle.linear(X, prep["Q_W"], prep["s_W"], rows=rows)
    gu.compare_y(Y[rows], ref)


def test_pair_mma_in_graph_replays(modes):
    # Back-to-back pair-MMA launches (cluster barriers, tensor memory of both
    # CTAs) inside a graph, with programmatic dependent launch between them.
    M, N, K = 1024, 2048, 2048
    X, Q_W, s_W, img = _layer(M, N, K, seed=53)
    cr.convrot_set_pair_mma(1)
    ref = gu.linear(X, Q_W, s_W, img).view(np.uint16)
    cr.convrot_set_pair_mma(2)
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


def test_pair_mma_gemm_dequant_entry(modes):
    # The GEMM-only entry point takes the same engine.
    M, N, K = 512, 1024, 2048
    rng = np.random.default_rng(54)
    QX = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
    QW = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    sX = rng.uniform(0.5, 2.0, size=M).astype(np.float32) / 127
    sW = rng.uniform(0.5, 2.0, size=N).astype(np.float32) / 127
    cr.convrot_set_pair_mma(2)
    y_pair = gu.gemm_dequant(QX, sX, QW, sW).view(np.uint16)
    gu.check_no_device_error()
    cr.convrot_set_pair_mma(1)
    y_one = gu.gemm_dequant(QX, sX, QW, sW).view(np.uint16)
    assert np.array_equal(y_pair, y_one)


LORA_SHAPES = [
    (4096, 2048, 8192, 32),  # the LoRA layer of the benchmark
    (300, 640, 1024, 12),    # ragged M and N, a rank count not a multiple of 8
    (100, 256, 512, 64),     # the odd CTA's rows all past M
]


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("shape", LORA_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_pair_mma_lora_is_bit_identical(modes, shape, bn):
    # A LoRA layer on pair-MMA tiles: the epilogue adds lora_scale * S in the
    # same fp32 expression as the one-SM tiles, so Y is the same bits; and
    # within tolerance of the oracle's layer on sampled rows.
    M, N, K, R = shape
    X, Q_W, s_W, img = _layer(M, N, K, seed=55)
    down, up = workloads.make_lora(N, K, R, seed=55)
    outs = []
    for mode in (2, 1):
        cr.convrot_set_pair_mma(mode)
        cr.convrot_set_tile_override(bn, 0)
        outs.append(gu.linear(X, Q_W, s_W, img, down, up, 0.8).view(np.uint16))
        gu.check_no_device_error()
    diff = int((outs[0] != outs[1]).sum())
    assert diff == 0, f"{diff} of {outs[0].size} outputs differ"
    rows = np.unique(np.concatenate([[0, min(M, 255) - 1, M - 1],
                                     np.random.default_rng(55).choice(M, min(M, 29), replace=False)]))
    ref = oracle.linear(X, gu.host(Q_W), gu.host(s_W), down, up, 0.8, rows=rows)
    gu.compare_y(outs[0].view(np.float16)[rows], ref)


def test_pair_mma_bf16_lora(modes):
    # bf16 X, Y and LoRA weights with a bias (the extended epilogue) on
    # pair-MMA tiles: the same bits as the one-SM tiles.
    M, N, K, R = 512, 1024, 2048, 32
    X, Q_W, s_W, img = _layer(M, N, K, seed=56)
    down, up = workloads.make_lora(N, K, R, seed=56)
    Xb = gu.dev(X).to(torch.bfloat16)
    db, ub = gu.dev(down).to(torch.bfloat16), gu.dev(up).to(torch.bfloat16)
    bias = gu.dev(np.random.default_rng(56).standard_normal(N).astype(np.float32))
    outs = []
    for mode in (2, 1):
        cr.convrot_set_pair_mma(mode)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ws = gu.workspace(cr.convrot_linear_workspace_bytes(M, N, K, R, True))
        cr.convrot_linear_ex(Xb, Q_W, s_W, Y, ws, W_img=img, bias=bias, lora_down=db,
                             lora_up=ub, lora_scale=0.8)
        gu.check_no_device_error()
        outs.append(gu.host(Y.view(torch.int16)))
    assert np.array_equal(outs[0], outs[1])
