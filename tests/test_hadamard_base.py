"""The 4x4 Hadamard base (page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal,
MPSMatrix, and MLX", section "What changed in the computation": H is the
Kronecker power of a 4x4 Hadamard base over groups of 256, divided by 16, and
symmetric).  On the CPU:

* every symmetric 4x4 Hadamard base B (found here by enumerating all 2^16
  sign matrices) factors as diag(d1) H4 R with R a signed permutation, and
  that factorization reproduces the oracle's dense 256 x 256 H of base B
  (D H_S R (x) R (x) R (x) R) -- the identity the GPU path relies on;
* convrot_set_hadamard_base accepts exactly those bases (and NULL), and
  rejects the rest with CONVROT_ERR_INVALID_ARG, with no GPU needed.

The helpers here (factor, kron4) are the test's own; the GPU tests use them
to carry the oracle's codes into the library's column order.
"""
import ctypes
import itertools

import numpy as np
import pytest

import oracle
import w8a8_hadamard_rotated_gb300 as cr

H4 = np.array(cr.SYLVESTER_BASE, dtype=np.int64)


def factor(B):
    """B = diag(d1) H4 R with R a signed permutation, by search."""
    B = np.asarray(B, dtype=np.int64)
    for d1 in itertools.product((1, -1), repeat=4):
        for perm in itertools.permutations(range(4)):
            R = np.zeros((4, 4), dtype=np.int64)
            for j in range(4):
                R[perm[j], j] = B[0, j] * d1[0] * H4[0, perm[j]]
            if np.array_equal(np.diag(d1) @ H4 @ R, B):
                return np.array(d1), R
    raise AssertionError("no factorization")


def factors(B):
    """Every (d1, R) with B = diag(d1) H4 R, R a signed permutation."""
    B = np.asarray(B, dtype=np.int64)
    out = []
    for d1 in itertools.product((1, -1), repeat=4):
        for perm in itertools.permutations(range(4)):
            R = np.zeros((4, 4), dtype=np.int64)
            for j in range(4):
                R[perm[j], j] = B[0, j] * d1[0] * H4[0, perm[j]]
            if np.array_equal(np.diag(d1) @ H4 @ R, B):
                out.append((np.array(d1), R))
    return out


def kron4(a):
    return np.kron(np.kron(np.kron(a, a), a), a)


def all_4x4(symmetric_only=True):
    out = []
    for bits in range(1 << 16):
        B = np.array([1 - 2 * ((bits >> i) & 1) for i in range(16)], dtype=np.int64).reshape(4, 4)
        if np.array_equal(B @ B.T, 4 * np.eye(4, dtype=np.int64)):
            if not symmetric_only or np.array_equal(B, B.T):
                out.append(B)
    return out


SYMMETRIC = all_4x4(True)


def test_enumeration_counts():
    # There are 768 Hadamard matrices of order 4; the symmetric ones are a
    # proper subset that includes Sylvester's and J - 2I.
    assert len(all_4x4(False)) == 768
    names = {tuple(B.ravel()) for B in SYMMETRIC}
    assert tuple(H4.ravel()) in names
    assert tuple((np.ones((4, 4), dtype=np.int64) - 2 * np.eye(4, dtype=np.int64)).ravel()) in names
    assert len(SYMMETRIC) == 64


@pytest.mark.parametrize("i", range(len(SYMMETRIC)))
def test_factorization_reproduces_the_oracle_h(i):
    B = SYMMETRIC[i]
    d1, R = factor(B)
    HB = oracle.hadamard256(B.astype(np.float64))
    HS = oracle.hadamard256()
    D = kron4(np.diag(d1)).astype(np.float64)
    assert np.array_equal(D @ HS @ kron4(R).astype(np.float64), HB)


@pytest.mark.parametrize("i", range(0, len(SYMMETRIC), 7))
def test_every_factorization_reproduces_the_oracle_h(i):
    # The factorization is not unique (eight per base); each one reproduces
    # H, which is why the library may pick any of them.
    B = SYMMETRIC[i]
    HB = oracle.hadamard256(B.astype(np.float64))
    HS = oracle.hadamard256()
    fs = factors(B)
    assert len(fs) == 8
    for d1, R in fs:
        D = kron4(np.diag(d1)).astype(np.float64)
        assert np.array_equal(D @ HS @ kron4(R).astype(np.float64), HB)


@pytest.fixture
def lib():
    cr.build()
    lb = cr.load()
    yield lb
    lb.convrot_set_hadamard_base(None)


def _set(lib, flat):
    buf = (ctypes.c_int8 * 16)(*flat)
    return lib.convrot_set_hadamard_base(ctypes.cast(buf, ctypes.c_void_p))


def test_setter_accepts_exactly_the_symmetric_hadamard_bases(lib):
    sym = {tuple(B.ravel()) for B in SYMMETRIC}
    for B in all_4x4(False):
        st = _set(lib, [int(v) for v in B.ravel()])
        assert st == (cr.CONVROT_OK if tuple(B.ravel()) in sym else cr.CONVROT_ERR_INVALID_ARG)
    assert lib.convrot_set_hadamard_base(None) == cr.CONVROT_OK


def test_setter_rejects_non_hadamard_and_bad_entries(lib):
    assert _set(lib, [1] * 16) == cr.CONVROT_ERR_INVALID_ARG
    bad = list(H4.ravel())
    bad[5] = 0
    assert _set(lib, bad) == cr.CONVROT_ERR_INVALID_ARG
    bad[5] = 2
    assert _set(lib, bad) == cr.CONVROT_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        cr.convrot_set_hadamard_base([[1, 1], [1, -1]])
    cr.convrot_set_hadamard_base(None)
