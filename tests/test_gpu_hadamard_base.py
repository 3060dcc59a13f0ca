"""A 4x4 Hadamard base other than Sylvester's (page "INT8ConvRot GEMM vs fp16
on M1 Max with Metal, MPSMatrix, and MLX", section "What changed in the
computation": H = B (x) B (x) B (x) B / 16 over groups of 256, symmetric).

The library runs the Sylvester transform on sign-flipped inputs and leaves
out a signed permutation of the rotated columns, common to X and W.  This
test derives that factorization on its own (a brute-force search, written
here, independent of the library's) and checks:

* activation and weight codes equal the oracle's codes of base B with their
  columns carried through the test's permutation, except +-1 flips at the
  oracle's near-ties; the scales equal the oracle's;
* the layer Y matches the oracle's layer of base B (tile and row kernels,
  the small-M engine, the no-allocation entry), and is bit-exact against the
  oracle's epilogue of the GPU's own codes;
* convrot_rotate refuses a base other than Sylvester's; the default comes
  back unchanged.
"""
import numpy as np
import pytest

import oracle
import workloads
import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = gu.torch

from .test_hadamard_base import H4, factors, kron4

# J - 2I: symmetric, Hadamard, and not a signed permutation of Sylvester's
# rows alone (its factorization needs input signs and a column permutation).
JM2I = np.ones((4, 4), dtype=np.int64) - 2 * np.eye(4, dtype=np.int64)
# Sylvester's with rows 1 and 2 negated and columns 1 and 2 negated: symmetric.
SIGNED = np.diag([1, -1, -1, 1]) @ H4 @ np.diag([1, -1, -1, 1])
BASES = {"jm2i": JM2I, "signed": SIGNED}


def to_library_order(Q, R4):
    """Codes of base B (columns in B's order) -> the library's order:
    per 256-group, Q R4^T (a signed permutation; exact in int64)."""
    M, K = Q.shape
    g = Q.reshape(M, K // 256, 256).astype(np.int64)
    return np.einsum("mgj,kj->mgk", g, R4).reshape(M, K)


def pre_in_library_order(pre, R4):
    M, K = pre.shape
    g = np.abs(pre.reshape(M, K // 256, 256))
    P = np.abs(R4)  # which B-order column lands on each library column
    return np.einsum("mgj,kj->mgk", g, P).reshape(M, K)


def matching_r4(q_gpu, q_b, pre_b, B):
    """R (x) R (x) R (x) R of the factorization of B that carries the oracle's
    codes of base B onto the GPU's (up to +-1 at near-ties).  (d1, R) and
    (-d1, -R) give the same column map, so the eight factorizations give four
    distinct maps; exactly one must fit."""
    maps = {}
    for _, R in factors(B):
        R4 = kron4(R)
        maps[R4.tobytes()] = R4
    hits = []
    for R4 in maps.values():
        try:
            gu.compare_q(q_gpu, to_library_order(q_b, R4), pre_in_library_order(pre_b, R4))
            hits.append(R4)
        except AssertionError:
            pass
    assert len(maps) == 4 and len(hits) == 1, f"{len(hits)} of {len(maps)} column maps match"
    return hits[0]


def library_r4(B):
    """The factorization the library uses for B, found from its weight codes
    on a small probe (the same for activations: see the code tests)."""
    W = workloads.make_w(64, 512, 99)
    cr.convrot_set_hadamard_base(B)
    Q, _, _ = gu.prepare_weight(W, with_img=False)
    ref = oracle.prepare_weight(W, H=oracle.hadamard256(B.astype(np.float64)))
    return matching_r4(gu.host(Q), ref["Q_W"], ref["pre"], B)


@pytest.fixture
def base_mode():
    gu.require_gpu()
    yield
    cr.convrot_set_hadamard_base(None)


@pytest.mark.parametrize("name", list(BASES))
@pytest.mark.parametrize("K", [2048, 768, 256])   # tile kernel, row kernel, one group
def test_activation_codes(base_mode, name, K):
    B = BASES[name]
    R4 = library_r4(B)
    M = 300
    X = workloads.make_x(M, K, 17, workloads.n_outliers(K))
    cr.convrot_set_hadamard_base(B)
    q, s = gu.rotate_quantize(X)
    ref = oracle.rotate_quantize(X, H=oracle.hadamard256(B.astype(np.float64)))
    # Exactly one factorization fits, and it is the weights' one.
    assert np.array_equal(matching_r4(q, ref["Q_X"], ref["pre"], B), R4)
    np.testing.assert_allclose(s, ref["s_X64"], rtol=1e-6, atol=0)


@pytest.mark.parametrize("name", list(BASES))
def test_weight_codes(base_mode, name):
    B = BASES[name]
    N, K = 320, 1024
    W = workloads.make_w(N, K, 18)
    cr.convrot_set_hadamard_base(B)
    Q, s, img = gu.prepare_weight(W)
    ref = oracle.prepare_weight(W, H=oracle.hadamard256(B.astype(np.float64)))
    matching_r4(gu.host(Q), ref["Q_W"], ref["pre"], B)
    np.testing.assert_allclose(gu.host(s), ref["s_W64"], rtol=1e-6, atol=0)
    assert np.array_equal(gu.host(img).astype(np.float64), gu.host(Q).astype(np.float64))


@pytest.mark.parametrize("name", list(BASES))
@pytest.mark.parametrize("shape", [(1024, 2048, 2048), (257, 640, 768), (8, 512, 2048),
                                   (64, 512, 2048)],
                         ids=lambda s: "x".join(map(str, s)))
def test_layer_matches_oracle(base_mode, name, shape):
    M, N, K = shape
    B = BASES[name]
    R4 = library_r4(B)
    H = oracle.hadamard256(B.astype(np.float64))
    X = workloads.make_x(M, K, 19, workloads.n_outliers(K))
    prep = oracle.prepare_weight(workloads.make_w(N, K, 19), H=H)
    Q_int = to_library_order(prep["Q_W"], R4).astype(np.int8)
    cr.convrot_set_hadamard_base(B)
    Y = gu.linear(X, Q_int, prep["s_W"], Q_int.astype(np.float16))
    rows = np.unique(np.concatenate([[0, M - 1],
                                     np.random.default_rng(19).choice(M, min(M, 40), replace=False)]))
    ref = oracle.linear(X, prep["Q_W"], prep["s_W"], rows=rows, H=H)
    gu.compare_y(Y[rows], ref)


@pytest.mark.parametrize("name", list(BASES))
def test_layer_bit_exact_on_own_codes(base_mode, name):
    M, N, K = 512, 1024, 2048
    cr.convrot_set_hadamard_base(BASES[name])
    X = workloads.make_x(M, K, 20, workloads.n_outliers(K))
    Q_W, s_W, img = gu.prepare_weight(workloads.make_w(N, K, 20))
    Y = gu.linear(X, Q_W, s_W, img).view(np.uint16)
    QX, sX = gu.rotate_quantize(X)
    exp = oracle.epilogue_f32(oracle.int_gemm(QX, gu.host(Q_W)), sX, gu.host(s_W))
    assert np.array_equal(Y, exp.astype(np.float16).view(np.uint16))


def test_noalloc_entry_follows_the_base(base_mode):
    M, N, K = 4, 768, 1024
    B = JM2I
    R4 = library_r4(B)
    H = oracle.hadamard256(B.astype(np.float64))
    X = workloads.make_x(M, K, 21, workloads.n_outliers(K))
    prep = oracle.prepare_weight(workloads.make_w(N, K, 21), H=H)
    Q_int = to_library_order(prep["Q_W"], R4).astype(np.int8)
    cr.convrot_set_hadamard_base(B)
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    cr.convrot_linear_noalloc(gu.dev(X), gu.dev(Q_int), gu.dev(prep["s_W"]), Y)
    gu.check_no_device_error()
    gu.compare_y(gu.host(Y), oracle.linear(X, prep["Q_W"], prep["s_W"], H=H))


def test_rotate_refuses_other_bases_and_default_returns(base_mode):
    M, K = 64, 1024
    X = workloads.make_x(M, K, 22, workloads.n_outliers(K))
    q0, s0 = gu.rotate_quantize(X)
    cr.convrot_set_hadamard_base(JM2I)
    R = torch.empty((M, K), dtype=torch.float16, device="cuda")
    with pytest.raises(RuntimeError):
        cr.convrot_rotate(gu.dev(X), R)
    cr.convrot_set_hadamard_base(None)
    cr.convrot_rotate(gu.dev(X), R)
    gu.check_no_device_error()
    q1, s1 = gu.rotate_quantize(X)
    assert np.array_equal(q0, q1) and np.array_equal(s0, s1)
    cr.convrot_set_hadamard_base(H4)  # Sylvester's given explicitly: the default
    q2, s2 = gu.rotate_quantize(X)
    assert np.array_equal(q0, q2) and np.array_equal(s0, s2)


@pytest.mark.parametrize("M", [1024, 64])   # 64 values per lane, and 32 (small M)
def test_bf16_input_with_signed_base(base_mode, M):
    # On values that fp16 and bf16 both hold exactly, the bf16 input path
    # (its own signed kernel variant) must give the fp16 path's Y bit for bit.
    N, K = 512, 2048
    rng = np.random.default_rng(23)
    X = (rng.integers(-200, 201, (M, K)) * 2.0 ** rng.integers(-6, 2, (M, K))).astype(np.float16)
    cr.convrot_set_hadamard_base(JM2I)
    Q_W, s_W, img = gu.prepare_weight(workloads.make_w(N, K, 23))
    Xd = gu.dev(X)
    ws = gu.workspace(cr.convrot_linear_workspace_bytes(M, N, K, 0, True))
    ys = []
    for xt in (Xd, Xd.to(torch.bfloat16)):
        Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        cr.convrot_linear_ex(xt, Q_W, s_W, Y, ws, W_img=img)
        gu.check_no_device_error()
        ys.append(gu.host(Y).view(np.uint16))
    assert np.array_equal(ys[0], ys[1])

