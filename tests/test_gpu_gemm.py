"""The int8 product A = Q_X Q_W^T must be bit-exact on both engines (the
tcgen05 tensor-core tiles and the small-M mma.sync kernel), for every tile
width, K split, ragged edge and the extreme operands that stress the fp32
chunk bound of the tensor-core path.  The scale restore from given operands
and scales must match the oracle's fp32 epilogue rounded to fp16 bit for bit.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads
import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu

pytestmark = pytest.mark.gpu

TC = cr.CONVROT_PATH_TCGEN05
SK = cr.CONVROT_PATH_SKINNY


@pytest.fixture(autouse=True)
def _reset_override():
    yield
    if gu.torch.cuda.is_available():
        cr.convrot_set_tile_override(0, 0)


def _rand(M, N, K, seed):
    return workloads.make_int8((M, K), seed), workloads.make_int8((N, K), seed + 1)


@pytest.mark.parametrize("path", [TC, SK])
def test_page_example_2x4x3(path, golden_dir):
    # Page "INT8ConvRot GEMM vs fp16 ...", section "Calling MPSGraph and
    # MPSMatrix directly": 70, 80, 90, 26, 28, 30.  K is padded with zeros to
    # the 256-wide group the library requires.
    gu.require_gpu()
    g = json.load(open(os.path.join(golden_dir, "mpsmatrix_2x4x3.json")))
    QX = np.zeros((2, 256), np.int8)
    QW = np.zeros((3, 256), np.int8)
    QX[:, :4] = np.array(g["left_MxK"], np.int8)
    QW[:, :4] = np.array(g["right_KxN"], np.int8).T
    A = gu.gemm_i32(QX, QW, path)
    assert A.ravel().tolist() == g["printed_output_row_major"]


@pytest.mark.parametrize("path", [TC, SK])
def test_exactness_protocol_37x80x256(path, golden_dir):
    # The pages' own check: 2,960 int32 outputs, 0 mismatches.
    gu.require_gpu()
    g = json.load(open(os.path.join(golden_dir, "exactness_protocol.json")))
    QX, QW = _rand(g["M"], g["N"], g["K"], seed=37)
    A = gu.gemm_i32(QX, QW, path)
    ref = oracle.int_gemm(QX, QW)
    assert A.size == g["elements"]
    assert int((A != ref).sum()) == g["mismatches"]


@pytest.mark.parametrize("K", [1024, 8192])
@pytest.mark.parametrize("path", [TC, SK])
def test_extreme_operands(K, path):
    gu.require_gpu()
    M, N = 40, 72
    cases = {
        "all_min": (np.full((M, K), -128, np.int8), np.full((N, K), -128, np.int8)),
        "max_min": (np.full((M, K), 127, np.int8), np.full((N, K), -128, np.int8)),
        "alternating": (np.where(np.arange(K) % 2 == 0, 127, -128).astype(np.int8)[None].repeat(M, 0),
                        np.where(np.arange(K) % 2 == 0, -128, 127).astype(np.int8)[None].repeat(N, 0)),
        "blocks": (np.where((np.arange(K) // 1024) % 2 == 0, -128, 127).astype(np.int8)[None].repeat(M, 0),
                   np.full((N, K), -128, np.int8)),
    }
    for name, (QX, QW) in cases.items():
        A = gu.gemm_i32(QX, QW, path)
        ref = oracle.int_gemm(QX, QW)
        assert np.array_equal(A, ref), name
    assert gu.gemm_i32(*cases["all_min"], path)[0, 0] == 2 ** 24 * (K // 1024)


def test_largest_k_exact():
    gu.require_gpu()
    K = 65536
    QX = np.full((3, K), -128, np.int8)
    QW = np.full((5, K), -128, np.int8)
    assert np.all(gu.gemm_i32(QX, QW, TC) == 2 ** 30)
    QX, QW = _rand(3, 5, K, seed=9)
    assert np.array_equal(gu.gemm_i32(QX, QW, TC), oracle.int_gemm(QX, QW))


@pytest.mark.parametrize("bn,splits", [(64, 1), (128, 1), (256, 1), (64, 4), (128, 3), (256, 2),
                                       (256, 16), (0, 0)])
def test_tc_tiles_and_splits(bn, splits):
    gu.require_gpu()
    cr.convrot_set_tile_override(bn, splits)
    # The last shape has more work units than SMs for every tile width, so
    # persistent CTAs walk several units (and accumulators alternate across
    # tiles).
    for (M, N, K) in [(200, 300, 2048), (128, 256, 1024), (1, 8, 256), (257, 129, 3072),
                      (512, 2560, 1024)]:
        QX, QW = _rand(M, N, K, seed=M + N + K)
        A = gu.gemm_i32(QX, QW, TC)
        assert np.array_equal(A, oracle.int_gemm(QX, QW)), (M, N, K)


@pytest.mark.parametrize("M", [1, 3, 16, 17, 33, 64])
@pytest.mark.parametrize("N,K", [(80, 256), (200, 2048), (33, 768)])
def test_skinny_exact(M, N, K):
    gu.require_gpu()
    QX, QW = _rand(M, N, K, seed=3 * M + N + K)
    A = gu.gemm_i32(QX, QW, SK)
    assert np.array_equal(A, oracle.int_gemm(QX, QW))


@pytest.mark.parametrize("path,bn,splits", [(TC, 0, 0), (TC, 64, 1), (TC, 128, 1), (TC, 256, 1),
                                            (TC, 128, 2), (SK, 0, 0)])
@pytest.mark.parametrize("M,N,K", [(37, 80, 256), (64, 264, 2048), (200, 77, 1024),
                                   (129, 320, 512)])
def test_dequant_epilogue_bit_exact(path, bn, splits, M, N, K):
    # fp16 outputs through the TMA-store epilogue (N a multiple of 8) and the
    # direct-store one (N = 77), every tile width, with and without split-K.
    gu.require_gpu()
    if path == SK and M > 64:
        pytest.skip("the small-M engine takes M <= 64")
    cr.convrot_set_tile_override(bn, splits)
    QX, QW = _rand(M, N, K, seed=M * N)
    rng = np.random.default_rng(M + N)
    sX = (rng.random(M) * 0.1).astype(np.float32)
    sW = (rng.random(N) * 0.01).astype(np.float32)
    sX[0] = 0.0
    Y = gu.gemm_dequant(QX, sX, QW, sW, path)
    ref = oracle.epilogue_f32(oracle.int_gemm(QX, QW), sX, sW).astype(np.float16)
    assert np.array_equal(Y.view(np.uint16), ref.view(np.uint16))


@pytest.mark.parametrize("K", [1024, 2048, 3072, 8192])
def test_dequant_partial_sum_boundaries(K):
    # The tile epilogue keeps (float)A in fp32 once every partial sum of the
    # earlier 1024-K chunks is within 2^24, and stays in int32 otherwise:
    # partial sums of exactly 2^24 (all -128 over a chunk), beyond it
    # (3 chunks), totals 2^24 + 1 and + 3 (not representable in fp32: the
    # epilogue's (float)A must round them to even), and random operands.
    gu.require_gpu()
    M, N = 64, 64
    QX = np.zeros((M, K), np.int8)
    QW = np.zeros((N, K), np.int8)
    QX[:, :] = -128
    QW[:, :] = -128
    QX[1, :], QW[1, :] = 0, 0
    QX[1, :1024], QW[1, :1024] = -128, -128
    if K > 1024:
        QX[1, 1024] = 1
        QW[:, 1024] = np.where(np.arange(N) % 2 == 0, 1, 3).astype(np.int8)
    rng = np.random.default_rng(K)
    QX[2:32] = rng.integers(-128, 128, (30, K), dtype=np.int8)
    QW[32:] = rng.integers(-128, 128, (32, K), dtype=np.int8)
    A = oracle.int_gemm(QX, QW)
    sX = np.full(M, 2.0 ** -16, np.float32)
    sW = np.full(N, 2.0 ** -10, np.float32)
    ref = oracle.epilogue_f32(A, sX, sW).astype(np.float16)
    for bn in (0, 128, 256):
        cr.convrot_set_tile_override(bn, 1)
        Y = gu.gemm_dequant(QX, sX, QW, sW, TC)
        assert np.array_equal(Y.view(np.uint16), ref.view(np.uint16)), bn
    cr.convrot_set_tile_override(0, 0)


def test_dequant_overflow_to_inf():
    gu.require_gpu()
    QX = np.full((2, 256), 127, np.int8)
    QW = np.full((8, 256), 127, np.int8)
    Y = gu.gemm_dequant(QX, np.array([1.0, -1.0], np.float32), QW, np.ones(8, np.float32), TC)
    assert np.all(np.isposinf(Y[0])) and np.all(np.isneginf(Y[1]))
