"""The tensor-core GEMM's planner on the host (convrot_plan_gemm; no GPU).

For a GB300 (152 SMs, 76 resident 2-CTA clusters) it must pick the engines
that measured fastest on the benchmark's layers (same-box comparisons of every
engine per shape), and honour its constraints: plain stores keep to one-SM
tiles, LoRA to engines without a CTA-pair K split, the test hooks apply, bad
arguments are rejected."""
import pytest

import w8a8_hadamard_rotated_gb300 as cr

ONE, PAIR, PMMA, L2, STREAM = (cr.CONVROT_ENGINE_ONE_SM, cr.CONVROT_ENGINE_PAIR_SPLIT,
                              cr.CONVROT_ENGINE_PAIR_MMA, cr.CONVROT_ENGINE_L2_SPLIT,
                              cr.CONVROT_ENGINE_PAIR_STREAM)


@pytest.fixture(scope="module", autouse=True)
def lib():
    cr.build()
    cr.load()
    yield
    cr.convrot_set_split_mode(0)
    cr.convrot_set_pair_mma(0)
    cr.convrot_set_tile_override(0, 0)


# (M, N, K) -> (tile width, K splits, engine): the measured-best choices.
EXPECTED = {
    (1024, 2048, 2048): (128, 1, ONE),
    (1024, 256, 2048): (128, 2, STREAM),
    (1024, 6144, 256): (128, 1, ONE),
    (1024, 2048, 1024): (128, 1, ONE),
    (1024, 8192, 2048): (256, 1, PMMA),
    (1024, 2048, 8192): (256, 2, PAIR),
    (128, 2048, 8192): (64, 4, L2),
    (128, 8192, 2048): (128, 2, STREAM),
    (4096, 8192, 2048): (256, 1, PMMA),
    (16384, 2048, 8192): (256, 1, PMMA),
}


@pytest.mark.parametrize("shape", list(EXPECTED), ids=lambda s: "x".join(map(str, s)))
def test_planner_picks_the_measured_engines(shape):
    assert cr.convrot_plan_gemm(*shape) == EXPECTED[shape]


@pytest.mark.parametrize("shape", list(EXPECTED), ids=lambda s: "x".join(map(str, s)))
def test_lora_and_plain_stores_keep_to_their_engines(shape):
    # The CTA-pair K splits carry no LoRA term; plain stores (rows that are
    # not 16-byte multiples) leave only from one-SM tiles.
    _, _, engine = cr.convrot_plan_gemm(*shape, R=16)
    assert engine in (ONE, L2, PMMA)
    _, _, engine = cr.convrot_plan_gemm(*shape, tma_store=False)
    assert engine in (ONE, L2)


def test_lora_layer_takes_pair_mma_tiles():
    # The LoRA layer of the benchmark (M = 4096, N = 2048, K = 8192) runs on
    # 256-wide pair-MMA tiles, as the same layer without LoRA does.
    assert cr.convrot_plan_gemm(4096, 2048, 8192, R=32) == (256, 1, PMMA)


def test_without_pair_clusters_no_pair_mma():
    for shape in EXPECTED:
        _, _, engine = cr.convrot_plan_gemm(*shape, pair_clusters_128=0, pair_clusters_256=0)
        assert engine != PMMA


def test_hooks_apply():
    try:
        cr.convrot_set_split_mode(1)
        cr.convrot_set_pair_mma(1)
        for shape in EXPECTED:
            assert cr.convrot_plan_gemm(*shape)[2] in (ONE, L2)
        cr.convrot_set_split_mode(0)
        cr.convrot_set_pair_mma(0)
        cr.convrot_set_tile_override(64, 1)
        assert cr.convrot_plan_gemm(1024, 2048, 2048)[:2] == (64, 1)
    finally:
        cr.convrot_set_split_mode(0)
        cr.convrot_set_pair_mma(0)
        cr.convrot_set_tile_override(0, 0)


def test_bad_arguments():
    for args in ((0, 64, 256), (16, 0, 256), (16, 64, 300), (16, 64, 256, 0)):
        with pytest.raises(RuntimeError):
            cr.convrot_plan_gemm(*args)


# The small-M engine (convrot_plan_small_m, 152 SMs): (M, N, K) -> (engine,
# K slices, column blocks), the measured-best choices of the fp16 layer.
NONE, DP4A, MMA1, SHARED, TWO_F16, TWO_S8 = (
    cr.CONVROT_SMALL_M_NONE, cr.CONVROT_SMALL_M_ONE_DP4A, cr.CONVROT_SMALL_M_ONE_MMA,
    cr.CONVROT_SMALL_M_ONE_SHARED, cr.CONVROT_SMALL_M_TWO_F16, cr.CONVROT_SMALL_M_TWO_S8)

SMALL_M_EXPECTED = {
    (1, 8192, 2048): (DP4A, 1, 0),     # one kernel, no cluster: 5.0 us
    (1, 4096, 4096): (DP4A, 1, 0),     # one slice of 4096 (no cluster): 5.6 us, 6.4 in pairs
    (1, 2048, 8192): (DP4A, 4, 0),     # 64 column blocks: slices of 2048 in clusters of 4
    (2, 8192, 2048): (DP4A, 1, 0),     # 6.2 us against 7.5 for two kernels
    (3, 8192, 2048): (TWO_F16, 1, 0),  # 7.6 us against 8.0 for one kernel
    (16, 8192, 2048): (TWO_F16, 1, 0),  # no cluster: 8.4 us, 9.9 in pairs
    (16, 2048, 8192): (TWO_F16, 4, 0),
    (16, 4096, 4096): (TWO_F16, 2, 0),
    (17, 2048, 2048): (NONE, 0, 0),
    (1024, 2048, 2048): (NONE, 0, 0),
}


@pytest.mark.parametrize("shape", list(SMALL_M_EXPECTED), ids=lambda s: "x".join(map(str, s)))
def test_small_m_planner_picks_the_measured_engines(shape):
    assert cr.convrot_plan_small_m(*shape) == SMALL_M_EXPECTED[shape]


def test_small_m_engine_hooks_apply():
    try:
        cr.convrot_set_small_m_engine(1)  # two kernels at every M (the s8 GEMM below M = 3)
        assert cr.convrot_plan_small_m(16, 8192, 2048) == (TWO_F16, 1, 0)
        assert cr.convrot_plan_small_m(1, 8192, 2048)[0] == TWO_S8
        cr.convrot_set_small_m_engine(2)  # the dp4a form at every M
        assert cr.convrot_plan_small_m(16, 8192, 2048)[0] == DP4A
        cr.convrot_set_small_m_engine(3)  # the 128-column fp16-MMA form
        assert cr.convrot_plan_small_m(16, 8192, 2048)[0] == MMA1
        cr.convrot_set_small_m_engine(4)  # the shared-rotation form where it applies
        assert cr.convrot_plan_small_m(16, 8192, 2048) == (SHARED, 2, 4)
        assert cr.convrot_plan_small_m(16, 2048, 8192)[0] == TWO_F16  # 64 items a CTA: not taken
        cr.convrot_set_small_m_engine(0)
        cr.convrot_set_skinny_engine(1)  # the s8 small-M GEMM
        assert cr.convrot_plan_small_m(16, 8192, 2048)[0] == TWO_S8
    finally:
        cr.convrot_set_small_m_engine(0)
        cr.convrot_set_skinny_engine(0)


def test_small_m_plan_bad_arguments():
    for args in ((0, 64, 256), (1, 0, 256), (1, 64, 300), (1, 64, 256, 0)):
        with pytest.raises(RuntimeError):
            cr.convrot_plan_small_m(*args)
