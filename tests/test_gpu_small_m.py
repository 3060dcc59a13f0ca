"""The one-launch small-M layer (decode.cu): at M <= 16 with fp16 X and Y, no
bias and no LoRA, one kernel rotates and quantizes each CTA's K slice of the
rows, combines the row maxima over the slices of a thread-block cluster,
multiplies by the CTA's weight slice (exact int8 dot products) and restores
the scales (page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix,
and MLX", section "What changed in the computation").

The codes and scales are those of the two-kernel path (the same butterflies,
row max, rounding and epilogue), so Y must be the same bits in every engine
mode (auto, one kernel at every M, one kernel with the weight copied before
the dependency wait, two kernels); and Y must match the oracle's layer.
Shapes cover one 256-group, ragged N (a CTA's columns past N), one to eight
K slices per cluster including long slices, K past what the kernel takes
(the two-kernel path), every M from 1 to 16, zero and extreme rows, a base
other than Sylvester's, graph replay, and a workspace left untouched.
"""
import numpy as np
import pytest

import oracle
import workloads
import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu
from .test_gpu_hadamard_base import BASES, library_r4, to_library_order

pytestmark = pytest.mark.gpu

torch = gu.torch

SHAPES = [
    (1, 2048, 8192),
    (16, 8192, 2048),
    (3, 1000, 768),      # three groups, ragged N
    (16, 33, 256),       # one group, one ragged column block
    (5, 4096, 4096),
    (2, 8192, 20480),    # slices raised to 2560 (the GEMM would take 1 or 2)
    (1, 96, 65536),      # the maximum K: slices of 8192 are too long, two kernels
    (7, 70000, 256),     # many column blocks, one group
    (4, 512, 10496),     # 41 groups: no split fits, the two-kernel path
    (16, 4096, 14336),   # 56 groups: slices of 3584
    (1, 256, 32768),     # eight slices of 4096, the longest the kernel takes
    (1, 3900, 4096),     # M = 1, one slice of 4096 (no cluster), ragged N
]


@pytest.fixture
def modes():
    gu.require_gpu()
    yield
    cr.convrot_set_small_m_engine(0)
    cr.convrot_set_small_m_weights_early(True)
    cr.convrot_set_skinny_engine(0)
    cr.convrot_set_hadamard_base(None)


ONE_KERNEL = [(f, e) for e in (False, True) for f in (2, 3, 4)]  # (form, weight before the wait)


def _layer(M, N, K, seed):
    X = workloads.make_x(M, K, seed, workloads.n_outliers(K))
    Q_W, s_W, _ = gu.prepare_weight(workloads.make_w(N, K, seed), with_img=False)
    return X, Q_W, s_W


def _y(X, Q_W, s_W, mode):
    cr.convrot_set_small_m_engine(mode)
    return gu.linear(X, Q_W, s_W).view(np.uint16)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_same_bits_as_two_kernels(modes, shape):
    # The one-kernel forms (mode 2: dp4a, 32 columns per CTA; mode 3: fp16
    # MMA, 128; mode 4: the rotation shared by a cluster's column blocks,
    # where it applies), with the weight copied after or before the
    # dependency wait, and the default choice, against the two-kernel path
    # (mode 1).
    M, N, K = shape
    X, Q_W, s_W = _layer(M, N, K, seed=61)
    y2 = _y(X, Q_W, s_W, 1)
    for mode, early in [(0, False)] + ONE_KERNEL:
        cr.convrot_set_small_m_weights_early(early)
        y1 = _y(X, Q_W, s_W, mode)
        diff = int((y1 != y2).sum())
        assert diff == 0, f"mode {mode} early {early}: {diff} of {y1.size} outputs differ"


# Sizes where the shared-rotation form (mode 4) applies, with its cluster:
# (K slices, column blocks, 256-groups each CTA rotates per row).
SHARED_SHAPES = [
    ((16, 8192, 2048), (2, 4, 1)),
    ((4, 8192, 2048), (2, 2, 2)),
    ((1, 2048, 8192), (4, 2, 4)),
    ((5, 4096, 4096), (4, 2, 2)),
    ((16, 2048, 2048), (4, 2, 1)),
    ((8, 300, 1024), (2, 2, 1)),    # ragged last column block
    ((6, 480, 2048), (4, 2, 1)),    # 15 column blocks: the last cluster's second block empty
    ((3, 1000, 8192), (4, 2, 4)),   # ragged N inside a block
]


@pytest.mark.parametrize("case", SHARED_SHAPES, ids=lambda c: "x".join(map(str, c[0])))
def test_shared_form(modes, case):
    # Mode 4 takes one kernel at these sizes (the two-kernel path takes two
    # from M = 3), gives the two-kernel path's bits with the weight copied
    # before or after the dependency wait, and matches the oracle.
    (M, N, K), _ = case
    cr.convrot_set_small_m_engine(4)
    assert cr.convrot_linear_kernel_count(M, N, K, 0, False) == 1
    X = workloads.make_x(M, K, 70, workloads.n_outliers(K))
    prep = oracle.prepare_weight(workloads.make_w(N, K, 70))
    ref = _y(X, prep["Q_W"], prep["s_W"], 1)
    for early in (True, False):
        cr.convrot_set_small_m_weights_early(early)
        y = _y(X, prep["Q_W"], prep["s_W"], 4)
        diff = int((y != ref).sum())
        assert diff == 0, f"early {early}: {diff} of {y.size} outputs differ"
    gu.compare_y(ref.view(np.float16), oracle.linear(X, prep["Q_W"], prep["s_W"]))


@pytest.mark.parametrize("form", [2, 3, 4])
@pytest.mark.parametrize("M", list(range(1, 17)))
def test_every_m_matches_oracle(modes, M, form):
    N, K = 320, 1024
    X = workloads.make_x(M, K, 62 + M, workloads.n_outliers(K))
    prep = oracle.prepare_weight(workloads.make_w(N, K, 62))
    cr.convrot_set_small_m_engine(form)
    Y = gu.linear(X, prep["Q_W"], prep["s_W"])
    gu.compare_y(Y, oracle.linear(X, prep["Q_W"], prep["s_W"]))


@pytest.mark.parametrize("form", [2, 3, 4])
@pytest.mark.parametrize("shape", [(1, 2048, 8192), (16, 8192, 2048), (4, 1000, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_matches_oracle(modes, shape, form):
    M, N, K = shape
    X = workloads.make_x(M, K, 63, workloads.n_outliers(K))
    prep = oracle.prepare_weight(workloads.make_w(N, K, 63))
    cr.convrot_set_small_m_engine(form)
    Y = gu.linear(X, prep["Q_W"], prep["s_W"])
    gu.compare_y(Y, oracle.linear(X, prep["Q_W"], prep["s_W"]))


@pytest.mark.parametrize("form", [2, 3, 4])
def test_zero_and_extreme_rows(modes, form):
    # A zero row (s_X = 0: codes 0, Y = 0), a row holding fp16's largest value
    # once, a constant row (one nonzero rotated entry per 256-group), and a
    # row of the smallest subnormal.
    M, N, K = 4, 256, 2048
    X = np.zeros((M, K), dtype=np.float16)
    X[1, 1234] = np.float16(65504.0)
    X[2, :] = np.float16(-1000.0)
    X[3, :] = np.float16(2.0 ** -24)
    prep = oracle.prepare_weight(workloads.make_w(N, K, 64))
    cr.convrot_set_small_m_engine(form)
    Y = gu.linear(X, prep["Q_W"], prep["s_W"])
    assert np.all(Y[0] == 0)
    gu.compare_y(Y, oracle.linear(X, prep["Q_W"], prep["s_W"]))
    assert np.array_equal(Y.view(np.uint16), _y(X, prep["Q_W"], prep["s_W"], 1))


@pytest.mark.parametrize("form", [2, 3, 4])
@pytest.mark.parametrize("name", list(BASES))
def test_other_base(modes, name, form):
    # The input signs of a non-Sylvester base: Y within tolerance of the
    # oracle's layer of base B (weight codes carried into the library's
    # column order as the base tests derive it), and the same bits as the
    # two-kernel path.
    B = BASES[name]
    R4 = library_r4(B)
    H = oracle.hadamard256(B.astype(np.float64))
    M, N, K = 6, 512, 2048
    X = workloads.make_x(M, K, 65, workloads.n_outliers(K))
    prep = oracle.prepare_weight(workloads.make_w(N, K, 65), H=H)
    Q_int = to_library_order(prep["Q_W"], R4).astype(np.int8)
    cr.convrot_set_hadamard_base(B)
    y1 = _y(X, Q_int, prep["s_W"], form)
    y2 = _y(X, Q_int, prep["s_W"], 1)
    assert np.array_equal(y1, y2)
    gu.compare_y(y1.view(np.float16), oracle.linear(X, prep["Q_W"], prep["s_W"], H=H))


@pytest.mark.parametrize("form", [2, 3, 4])
def test_graph_replay_and_workspace_untouched(modes, form):
    M, N, K = 8, 2048, 4096
    X, Q_W, s_W = _layer(M, N, K, seed=66)
    ref = _y(X, Q_W, s_W, 1)
    cr.convrot_set_small_m_engine(form)
    Xd = gu.dev(X)
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    nbytes = cr.convrot_linear_workspace_bytes(M, N, K, 0, False)
    ws = gu.workspace(nbytes)
    ws.fill_(0xA5)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        cr.convrot_linear(Xd, Q_W, s_W, Y, ws)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(3):
            cr.convrot_linear(Xd, Q_W, s_W, Y, ws)
    for _ in range(3):
        Y.zero_()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        gu.check_no_device_error()
        assert np.array_equal(gu.host(Y).view(np.uint16), ref)
    assert bool((ws == 0xA5).all())


def test_weight_written_by_the_call_ahead(modes):
    # The weight of a small-M layer is the int8 output of the call right
    # before it on the same stream (convrot_rotate_quantize): the layer copies
    # its weight before its dependency wait, so that kernel must not let it
    # start early.  Back to back in one graph, several times.
    gu.require_gpu()
    M, N, K = 1, 512, 2048
    A = workloads.make_x(N, K, 67, workloads.n_outliers(K))
    X = workloads.make_x(M, K, 68, workloads.n_outliers(K))
    Ad, Xd = gu.dev(A), gu.dev(X)
    Q = torch.empty((N, K), dtype=torch.int8, device="cuda")
    sA = torch.empty((N,), dtype=torch.float32, device="cuda")
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = gu.workspace(cr.convrot_linear_workspace_bytes(M, N, K, 0, False))
    stream = torch.cuda.Stream()

    def pair():
        Q.fill_(0)  # the layer would see zeros if it read Q too early
        cr.convrot_rotate_quantize(Ad, Q, sA)
        cr.convrot_linear(Xd, Q, sA, Y, ws)

    with torch.cuda.stream(stream):
        pair()
    stream.synchronize()
    QA = gu.host(Q)
    exp = oracle.linear(X, QA, gu.host(sA))
    gu.compare_y(gu.host(Y), exp)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(4):
            pair()
    for _ in range(3):
        Y.zero_()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        gu.check_no_device_error()
        gu.compare_y(gu.host(Y), exp)


SKINNY_SHAPES = [
    (3, 8192, 2048),
    (5, 2048, 8192),
    (8, 1000, 768),     # ragged N, three groups
    (9, 4096, 4096),    # two n8 tiles of rows
    (16, 8192, 2048),
    (16, 200, 256),     # one 256-group, one ragged column block
    (2, 512, 2048),     # below the default's M: engine 2 only
    (12, 2048, 20480),  # slices of 2560 (the fp16 kernel takes up to 4096)
    (4, 96, 65536),     # K past what the fp16 kernel takes: the s8 kernel
]


@pytest.mark.parametrize("shape", SKINNY_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_skinny_engines_same_bits(modes, shape):
    # The two-kernel path's small-M GEMM: the fp16-MMA bulk-copy kernel
    # (skinny engine 2 and the default, with the weight copied before or
    # after the dependency wait) against the mma.sync s8 kernel (engine 1),
    # and the oracle.
    M, N, K = shape
    X = workloads.make_x(M, K, 69, workloads.n_outliers(K))
    prep = oracle.prepare_weight(workloads.make_w(N, K, 69))
    cr.convrot_set_small_m_engine(1)
    cr.convrot_set_skinny_engine(1)
    ref = gu.linear(X, prep["Q_W"], prep["s_W"]).view(np.uint16)
    for early in (True, False):
        cr.convrot_set_small_m_weights_early(early)
        for eng in (2, 0):
            cr.convrot_set_skinny_engine(eng)
            y = gu.linear(X, prep["Q_W"], prep["s_W"]).view(np.uint16)
            diff = int((y != ref).sum())
            assert diff == 0, f"engine {eng} early {early}: {diff} of {y.size} outputs differ"
    gu.compare_y(ref.view(np.float16), oracle.linear(X, prep["Q_W"], prep["s_W"]))
