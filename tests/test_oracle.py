"""Pins for the CPU oracle, checked against what the pages and mathematics fix.

Nothing here re-types an oracle formula: each check comes from a closed form,
an invariant the page states, a printed example, a library routine of an
independent definition (numpy's Kronecker product and matmul), exact rational
arithmetic, or brute force on tiny inputs.  Pages cited:

  [GEMM page]  "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix, and MLX"
  [PR page]    "[PR #249] Add an mps backend: weight-only INT8 and W4A8/W6A8
               linears for Apple GPUs"
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads


# Rows of a Hadamard matrix in another order: orthogonal, not symmetric.
NONSYM_BASE = np.array([[1, -1, 1, -1], [1, 1, 1, 1], [1, 1, -1, -1], [1, -1, -1, 1]], float)


def _popcount(v):
    return bin(v).count("1")


# --------------------------------------------------------------------------
# H -- [GEMM page] "What changed in the computation": Kronecker products of
# 4x4 Hadamards up to 256x256, divided by 16; symmetric; HH = I.
# --------------------------------------------------------------------------

def test_h_symmetric_and_involutory():
    H = oracle.hadamard256()
    assert H.shape == (256, 256)
    assert np.array_equal(H, H.T)
    assert np.abs(H @ H - np.eye(256)).max() <= 1e-12


def test_h_closed_form_entries():
    # Sylvester's construction: H[i][j] = (-1)^popcount(i & j) / 16.
    H = oracle.hadamard256()
    ref = np.array([[(-1) ** _popcount(i & j) / 16.0 for j in range(256)]
                    for i in range(256)])
    assert np.array_equal(H, ref)


def test_h_matches_numpy_kron_for_nonsymmetric_base():
    # A row-permuted Hadamard base is orthogonal but not symmetric, so any
    # index or ordering slip in the Kronecker expansion shows up here.
    B = NONSYM_BASE
    H = oracle.hadamard256(B)
    ref = np.kron(np.kron(np.kron(B, B), B), B) / 16.0
    assert np.array_equal(H, ref)
    assert np.abs(H @ H.T - np.eye(256)).max() <= 1e-12
    assert not np.array_equal(H, H.T)


def test_identity_base_gives_identity():
    H = oracle.hadamard256(2.0 * np.eye(4))
    assert np.array_equal(H, np.eye(256))


# --------------------------------------------------------------------------
# Rotation: X_rot = X H and W_rot = W H^T, group-wise over the last dimension.
# --------------------------------------------------------------------------

def test_rotation_against_numpy_matmul_nonsymmetric():
    rng = np.random.default_rng(11)
    B = NONSYM_BASE
    H = oracle.hadamard256(B)
    x = rng.standard_normal((5, 768))
    xr = oracle.rotate(x, H, transpose_h=False)
    wr = oracle.rotate(x, H, transpose_h=True)
    for g in range(3):
        sl = slice(256 * g, 256 * (g + 1))
        np.testing.assert_allclose(xr[:, sl], x[:, sl] @ H, rtol=0, atol=1e-12)
        np.testing.assert_allclose(wr[:, sl], x[:, sl] @ H.T, rtol=0, atol=1e-12)


def test_rotation_invariance_xw():
    # [GEMM page]: X_rot W_rot^T = (XH)(WH^T)^T = X H H W^T = X W^T.
    X = workloads.make_x(16, 1024, seed=5).astype(np.float64)
    W = workloads.make_w(24, 1024, seed=5).astype(np.float64)
    lhs = oracle.matmul_nt(oracle.rotate(X), oracle.rotate(W, transpose_h=True))
    rhs = oracle.matmul_nt(X, W)
    rel = np.abs(lhs - rhs).max() / np.abs(rhs).max()
    assert rel <= 1e-9


def test_rotation_preserves_group_norms():
    X = workloads.make_x(8, 512, seed=6).astype(np.float64)
    Xr = oracle.rotate(X)
    for g in range(2):
        sl = slice(256 * g, 256 * (g + 1))
        np.testing.assert_allclose(np.linalg.norm(Xr[:, sl], axis=1),
                                   np.linalg.norm(X[:, sl], axis=1), rtol=1e-13)


def _fwht_reference(v):
    # Independent fast Walsh-Hadamard butterflies (unnormalized), then / 16.
    a = [Fraction(float(t)) for t in v]
    h = 1
    while h < len(a):
        for i in range(0, len(a), 2 * h):
            for j in range(i, i + h):
                a[j], a[j + h] = a[j] + a[j + h], a[j] - a[j + h]
        h *= 2
    return [t / 16 for t in a]


def test_rotation_exact_for_fp16_inputs():
    # fp16 inputs: each X_rot entry is a sum of 256 dyadic rationals /16 that
    # fits in fp64's 53 bits, so the oracle's fp64 rotation must be exact.
    X = workloads.make_x(3, 256, seed=7, n_out=4)
    X[0, 0] = np.float16(6.0e-8)       # fp16 subnormal
    X[0, 1] = np.float16(65504.0)      # fp16 max
    X[1, :] = np.float16(-0.0)
    Xr = oracle.rotate(X.astype(np.float64))
    for r in range(3):
        exact = _fwht_reference(X[r].astype(np.float64))
        assert [Fraction(float(t)) for t in Xr[r]] == exact


# --------------------------------------------------------------------------
# Quantization: s = max|v|/127, Q = round(v/s), clamp to [-128, 127].
# --------------------------------------------------------------------------

def _round_half_even_bruteforce(p):
    # Pick the integer in [-128, 127] nearest to p; on an exact tie take the
    # even one.  Enumerates every candidate.
    best = None
    for q in range(-128, 128):
        d = abs(Fraction(p) - q)
        if best is None or d < best[0] or (d == best[0] and q % 2 == 0):
            best = (d, q)
    return best[1]


def test_quantize_bruteforce_tiny():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((4, 256)) * np.array([[1.0], [0.01], [300.0], [1e-6]])
    q, s, pre = oracle.quantize_rows(v)
    for r in range(4):
        amax = max(abs(float(t)) for t in v[r])
        assert s[r] == amax / 127.0
        for k in range(256):
            assert q[r, k] == _round_half_even_bruteforce(v[r, k] / s[r])


def test_quantize_exact_ties_round_to_even():
    v = np.array([[127.0, 2.5, -2.5, 3.5, 0.5, -0.5, 1.5, -1.5] + [0.0] * 248])
    q, s, _ = oracle.quantize_rows(v)
    assert s[0] == 1.0
    assert list(q[0, :8]) == [127, 2, -2, 4, 0, 0, 2, -2]


def test_quantize_invariants_on_workload():
    X = workloads.make_x(64, 2048, seed=1)
    act = oracle.rotate_quantize(X)
    q, pre = act["Q_X"].astype(int), act["pre"]
    assert q.min() >= -128 and q.max() <= 127
    assert np.all(np.abs(pre - q) <= 0.5)
    # Each row's max-abs element maps to +-127.
    arg = np.argmax(np.abs(act["X_rot"]), axis=1)
    assert np.all(np.abs(q[np.arange(64), arg]) == 127)
    np.testing.assert_allclose(act["s_X64"], np.abs(act["X_rot"]).max(axis=1) / 127,
                               rtol=0, atol=0)


def test_quantize_zero_row():
    q, s, pre = oracle.quantize_rows(np.zeros((2, 256)))
    assert np.all(q == 0) and np.all(s == 0) and np.all(pre == 0)


def test_prepare_weight_rows():
    W = workloads.make_w(16, 512, seed=8)
    prep = oracle.prepare_weight(W)
    Wrot = oracle.rotate(W.astype(np.float64), transpose_h=True)
    assert prep["s_W"].dtype == np.float32
    np.testing.assert_array_equal(prep["s_W64"], np.abs(Wrot).max(axis=1) / 127)
    assert np.all(np.abs(prep["Q_W"][np.arange(16), np.argmax(np.abs(Wrot), 1)]) == 127)


# --------------------------------------------------------------------------
# Integer GEMM: A = Q_X Q_W^T in int32.
# --------------------------------------------------------------------------

def test_int_gemm_page_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "mpsmatrix_2x4x3.json")))
    left = np.array(g["left_MxK"], dtype=np.int8)
    right = np.array(g["right_KxN"], dtype=np.int8)
    A = oracle.int_gemm(left, right.T.copy())
    assert A.ravel().tolist() == g["printed_output_row_major"]


def test_int_gemm_exactness_protocol(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "exactness_protocol.json")))
    M, N, K = g["M"], g["N"], g["K"]
    QX = workloads.make_int8((M, K), seed=37)
    QW = workloads.make_int8((N, K), seed=80)
    A = oracle.int_gemm(QX, QW)
    ref = QX.astype(np.int64) @ QW.astype(np.int64).T
    assert A.size == g["elements"]
    assert int((A != ref).sum()) == g["mismatches"]
    assert int(np.abs(A - ref).max()) == g["max_abs_diff"]


def test_int_gemm_bruteforce_python_ints():
    QX = workloads.make_int8((3, 256), seed=1)
    QW = workloads.make_int8((4, 256), seed=2)
    A = oracle.int_gemm(QX, QW)
    for m in range(3):
        for n in range(4):
            assert A[m, n] == sum(int(a) * int(b) for a, b in zip(QX[m], QW[n]))


def test_int_gemm_extremes():
    K = 1024
    neg = np.full((2, K), -128, np.int8)
    A = oracle.int_gemm(neg, neg)
    assert np.all(A == 2 ** 24)
    pos = np.full((1, K), 127, np.int8)
    assert oracle.int_gemm(pos, neg)[0, 0] == -127 * 128 * K
    # 16384 * 131328 > 2^31 - 1: the oracle must refuse, not wrap silently.
    big = np.full((1, 131328), -128, np.int8)
    with pytest.raises(OverflowError):
        oracle.int_gemm(big, big)


# --------------------------------------------------------------------------
# Scale restore: Y = A (.) s_X s_W^T.
# --------------------------------------------------------------------------

def test_epilogue_special_cases():
    A = np.array([[1, -2, 3], [2 ** 24 + 1, -7, 0]], np.int32)
    ones = oracle.epilogue_f32(A, np.ones(2, np.float32), np.ones(3, np.float32))
    # s = 1: Y is A rounded once to fp32 (2^24 + 1 -> 2^24).
    assert ones.tolist() == [[1.0, -2.0, 3.0], [16777216.0, -7.0, 0.0]]
    pow2 = oracle.epilogue_f32(A[:1], np.array([0.5], np.float32),
                               np.array([0.25, 2.0, 0.125], np.float32))
    assert pow2.tolist() == [[0.125, -2.0, 0.1875]]


def test_epilogue_outer_product_structure():
    rng = np.random.default_rng(0)
    A = rng.integers(-10 ** 6, 10 ** 6, size=(6, 5)).astype(np.int32)
    sX = rng.random(6).astype(np.float32)
    sW = rng.random(5).astype(np.float32)
    Y = oracle.epilogue_f32(A, sX, sW).astype(np.float64)
    exact = A.astype(np.float64) * sX.astype(np.float64)[:, None] * sW.astype(np.float64)[None, :]
    # Two fp32 roundings (plus the int->fp32 one): within 3 half-ulps.
    assert np.all(np.abs(Y - exact) <= 3 * 2.0 ** -24 * np.abs(exact) + 1e-30)


# --------------------------------------------------------------------------
# LoRA -- [PR page] "What": lora_down [R,K], lora_up [N,R], lora_scale.
# --------------------------------------------------------------------------

def test_lora_special_cases():
    X = workloads.make_x(4, 256, seed=9).astype(np.float64)
    down, up = workloads.make_lora(6, 256, 3, seed=9)
    assert np.all(oracle.lora(X, down, up, 0.0) == 0)
    assert np.all(oracle.lora(X, down, np.zeros_like(up), 0.8) == 0)
    # rank 1, down = e_k, up = ones: the term is scale * X[:, k] on every column.
    e = np.zeros((1, 256)); e[0, 17] = 1.0
    L = oracle.lora(X, e, np.ones((6, 1)), 0.5)
    np.testing.assert_array_equal(L, np.repeat(0.5 * X[:, 17:18], 6, axis=1))


def test_lora_against_numpy():
    X = workloads.make_x(5, 512, seed=10).astype(np.float64)
    down, up = workloads.make_lora(7, 512, 3, seed=10)
    L = oracle.lora(X, down, up, 0.8)
    ref = 0.8 * (X @ down.astype(np.float64).T) @ up.astype(np.float64).T
    np.testing.assert_allclose(L, ref, rtol=1e-12, atol=1e-15)


# --------------------------------------------------------------------------
# The whole layer.
# --------------------------------------------------------------------------

def test_linear_rows_subset_matches_full():
    cfg = workloads.TINY
    X, W, _, _ = workloads.make_inputs(cfg)
    prep = oracle.prepare_weight(W)
    full = oracle.linear(X, prep["Q_W"], prep["s_W"])
    rows = np.array([0, 5, 63])
    part = oracle.linear(X, prep["Q_W"], prep["s_W"], rows=rows)
    np.testing.assert_array_equal(part["A"], full["A"][rows])
    np.testing.assert_array_equal(part["Y32"], full["Y32"][rows])


def test_linear_quant_error_and_rotation_benefit():
    # [GEMM page]: the rotation spreads outliers so INT8 rounding error drops
    # (the QuaRot argument).  With an identity "rotation" the same layer must
    # be clearly worse on outlier-heavy activations.
    X, W, _, _ = workloads.make_inputs(workloads.Config("t", 64, 128, 1024, seed=3))
    exact = oracle.matmul_nt(X.astype(np.float64), W.astype(np.float64))

    def err(H):
        prep = oracle.prepare_weight(W, H)
        y = oracle.linear(X, prep["Q_W"], prep["s_W"], H=H)["Y_ref"]
        return np.linalg.norm(y - exact) / np.linalg.norm(exact)

    e_rot = err(None)
    e_id = err(np.eye(256))
    assert e_rot < 0.02
    assert e_rot < 0.5 * e_id


def test_linear_with_lora_adds_term():
    cfg = workloads.Config("t", 8, 64, 512, seed=12, R=5, lora_scale=0.8)
    X, W, down, up = workloads.make_inputs(cfg)
    prep = oracle.prepare_weight(W)
    base = oracle.linear(X, prep["Q_W"], prep["s_W"])
    withl = oracle.linear(X, prep["Q_W"], prep["s_W"], down, up, 0.8)
    np.testing.assert_array_equal(withl["Y32"], base["Y32"])
    ref = 0.8 * (X.astype(np.float64) @ down.astype(np.float64).T) @ up.astype(np.float64).T
    np.testing.assert_allclose(withl["Y_ref"] - base["Y_ref"], ref, rtol=1e-9, atol=1e-12)


def test_near_tie_bound_counts_flips():
    pre = np.array([[0.5, 1.50005, 2.3, -3.49995]])
    assert oracle.near_tie_mask(pre).tolist() == [[True, True, False, True]]


# --------------------------------------------------------------------------
# The workload table transcribed from the [GEMM page] per-shape table.
# --------------------------------------------------------------------------

def test_sweep_table_matches_page(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "sweep_shapes.json")))
    shapes = tuple((s["N"], s["K"], s["layers"]) for s in g["shapes"])
    assert shapes == workloads.SWEEP_SHAPES
    assert sum(c for _, _, c in shapes) == g["total_layers"]
    for col, key in (("fp16_ms", "fp16"), ("dequant_ms", "dequant"),
                     ("weight_only_ms", "weight_only")):
        total = sum(s[col] * s["layers"] for s in g["shapes"])
        assert abs(total - g["weighted_ms_printed"][key]) < 1.0


# ----------------------------------------------------------------------------
# Bias and bf16 output ([PR page], section "Design": bias added in eager's
# order; bf16 written bit-exactly with torch's cast).
# ----------------------------------------------------------------------------

def _bf16_special_values():
    f = np.float32
    vals = [0.0, -0.0, 1.0, -1.0, np.inf, -np.inf,
            1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8,        # ties: down to even, up to even
            1.0 + 2.0 ** -8 + 2.0 ** -20,                # just above a tie
            3.3895e38, 3.39e38, 3.4e38, -3.4e38,         # around the top of the range
            1e-40, -1e-40, 2.0 ** -133, 2.0 ** -126,     # fp32 subnormals, smallest normal
            65504.0, 65520.0, 1e-8]
    return np.array(vals, dtype=f)


def test_round_bf16_matches_torch_cast():
    # torch's CPU float -> bfloat16 conversion is an independent
    # implementation of the same IEEE round-to-nearest-even.
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = np.concatenate([
        _bf16_special_values(),
        (rng.standard_normal(20000) * 10.0 ** rng.uniform(-30, 30, 20000)).astype(np.float32),
        # every tie pattern in the low half-word, with random upper halves
        ((rng.integers(0, 1 << 16, 4096, dtype=np.uint32) << 16) | np.uint32(0x8000)).view(np.float32),
    ]).astype(np.float32)
    finite = np.isfinite(x)
    ours = oracle.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours[finite | np.isinf(x)], ref[finite | np.isinf(x)])


def test_round_bf16_nan_and_decode():
    nan = np.array([np.nan, -np.nan], dtype=np.float32)
    b = oracle.round_bf16(nan)
    assert np.all(np.isnan(oracle.bf16_to_f32(b)))
    # decode is exact and inverts the rounding on representable values
    bits = np.arange(0, 1 << 16, 7, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_f32(bits)
    ok = np.isfinite(vals)
    assert np.array_equal(oracle.round_bf16(vals[ok]), bits[ok])
    torch = pytest.importorskip("torch")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(vals[ok], ref[ok])


def test_bias_special_cases():
    rng = np.random.default_rng(6)
    M, N = 5, 33
    A = rng.integers(-2 ** 20, 2 ** 20, (M, N), dtype=np.int64).astype(np.int32)
    A[2] = 0                                            # a zero row
    sX = rng.uniform(0.1, 2.0, M).astype(np.float32)
    sW = rng.uniform(0.001, 0.01, N).astype(np.float32)
    bias = rng.standard_normal(N).astype(np.float32) * 100
    Y0 = oracle.epilogue_f32(A, sX, sW)
    Yb = oracle.epilogue_f32(A, sX, sW, bias)
    # zero bias changes nothing; a zero row of A gives the bias itself
    assert np.array_equal(oracle.epilogue_f32(A, sX, sW, np.zeros(N, np.float32)), Y0)
    assert np.array_equal(Yb[2], bias)
    # the bias is per output column: rows differ from Y0 by the same vector
    # (up to the one rounding of the add), and a bias equal to -Y0[r]
    # cancels row r exactly
    assert np.array_equal(oracle.epilogue_f32(A, sX, sW, -Y0[1])[1], np.zeros(N, np.float32))
    # huge biases absorb the product entirely (|Y0| < ulp(2^40) / 2)
    big = np.full(N, 2.0 ** 40, np.float32)
    assert np.all(np.abs(Y0) < 2.0 ** 16)
    assert np.array_equal(oracle.epilogue_f32(A, sX, sW, big), np.broadcast_to(big, (M, N)))


def test_bias_is_a_separate_rounding():
    # Eager rounds the scale restore, then adds the bias: two roundings.  A
    # fused multiply-add would give the product's rounding error instead of
    # an exact zero when the bias cancels the rounded product.
    A = np.array([[3]], np.int32)
    sX = np.array([1.0], np.float32)
    sW = np.array([np.float32(0.1)], np.float32)           # 3 * 0.1 is not exact in fp32
    y = oracle.epilogue_f32(A, sX, sW)
    assert float(Fraction(float(y[0, 0]))) != float(3 * Fraction(float(sW[0])))
    out = oracle.epilogue_f32(A, sX, sW, -y[0])
    assert out[0, 0] == 0.0
