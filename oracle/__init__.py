"""CPU oracle for the INT8ConvRot (W8A8 Hadamard-rotated) linear layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library never imports, links or calls it, and this
package imports nothing from the product library.

The arithmetic lives in ``convrot_oracle.c`` (plain C, fp64, naive loops,
compiled here with gcc and loaded through ctypes).  This module only marshals
numpy arrays and composes the steps in the order the pages give them:

* the page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix, and MLX",
  section "What changed in the computation" -- H, the group-wise rotation,
  row-wise max-abs/127 quantization with a clamp to [-128, 127], the int32
  product A = Q_X Q_W^T and the scale restore Y = A (.) s_X s_W^T;
* the page "[PR #249] Add an mps backend: weight-only INT8 and W4A8/W6A8
  linears for Apple GPUs", section "What" -- the unmerged LoRA arguments
  lora_down [R, K], lora_up [N, R], lora_scale.

Readings where the pages are silent:
the 4x4 base is Sylvester's [[1,1],[1,-1]] (x) [[1,1],[1,-1]]; "round" is
round-half-to-even; an all-zero row quantizes to s = 0, Q = 0; the scale
restore is ((float)A * s_X) * s_W in fp32; the LoRA term is evaluated in fp64
and added to that fp32 result.

Parity pins: every function here is pinned by ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "convrot_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libconvrot_oracle.so")

_lock = threading.Lock()
_lib = None

GROUP = 256

#: Sylvester 4x4 Hadamard [[1,1],[1,-1]] (x) [[1,1],[1,-1]] (a reading: the
#: pages say "4x4 Hadamard matrices" and that H is symmetric).
SYLVESTER4 = np.array(
    [[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]], dtype=np.float64
)

NEAR_TIE = 1e-4  # a pre-round value within this of a .5 tie may round either way


def build(force: bool = False) -> str:
    """Compile convrot_oracle.c into a shared library (OpenMP if available)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        D = ctypes.c_double
        lib.oracle_hadamard256.argtypes = [P, P]
        lib.oracle_hadamard256.restype = None
        lib.oracle_rotate_groups.argtypes = [P, I64, I64, P, I, P, I]
        lib.oracle_rotate_groups.restype = None
        lib.oracle_quantize_rows.argtypes = [P, I64, I64, P, P, P, I]
        lib.oracle_quantize_rows.restype = None
        lib.oracle_int_gemm.argtypes = [P, P, I64, I64, I64, P, I]
        lib.oracle_int_gemm.restype = I64
        lib.oracle_epilogue_f32.argtypes = [P, P, P, I64, I64, P]
        lib.oracle_epilogue_f32.restype = None
        lib.oracle_add_bias_f32.argtypes = [P, P, I64, I64]
        lib.oracle_add_bias_f32.restype = None
        lib.oracle_round_bf16.argtypes = [P, P, I64]
        lib.oracle_round_bf16.restype = None
        lib.oracle_lora.argtypes = [P, I64, I64, P, I64, P, I64, D, P, I]
        lib.oracle_lora.restype = None
        lib.oracle_matmul_nt.argtypes = [P, P, I64, I64, I64, P, I]
        lib.oracle_matmul_nt.restype = None
        lib.oracle_max_threads.argtypes = [I]
        lib.oracle_max_threads.restype = I
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def threads_used(nthreads: int = 0) -> int:
    """Threads the oracle's parallel loops use for a given request (0 = all)."""
    return int(_load().oracle_max_threads(int(nthreads)))


# ----------------------------------------------------------------------------
# The steps, one function each.
# ----------------------------------------------------------------------------

def hadamard256(base4: np.ndarray | None = None) -> np.ndarray:
    """Dense 256x256 H = (B (x) B (x) B (x) B) / 16 in fp64."""
    b = _c(SYLVESTER4 if base4 is None else base4, np.float64)
    assert b.shape == (4, 4)
    H = np.empty((GROUP, GROUP), dtype=np.float64)
    _load().oracle_hadamard256(_ptr(b), _ptr(H))
    return H


def rotate(x: np.ndarray, H: np.ndarray | None = None, transpose_h: bool = False,
           nthreads: int = 0) -> np.ndarray:
    """Group-wise rotation of the last dimension: x H (or x H^T), fp64."""
    x = _c(x, np.float64)
    rows, K = x.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 256")
    H = hadamard256() if H is None else _c(H, np.float64)
    out = np.empty_like(x)
    _load().oracle_rotate_groups(_ptr(x), rows, K, _ptr(H), int(bool(transpose_h)),
                                 _ptr(out), int(nthreads))
    return out


def quantize_rows(v: np.ndarray, nthreads: int = 0):
    """Row-wise int8 quantization. Returns (q int8, s fp64, pre fp64)."""
    v = _c(v, np.float64)
    rows, K = v.shape
    q = np.empty((rows, K), dtype=np.int8)
    s = np.empty((rows,), dtype=np.float64)
    pre = np.empty((rows, K), dtype=np.float64)
    _load().oracle_quantize_rows(_ptr(v), rows, K, _ptr(q), _ptr(s), _ptr(pre),
                                 int(nthreads))
    return q, s, pre


def int_gemm(QX: np.ndarray, QW: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """A = Q_X Q_W^T, exact int32 (raises if an entry does not fit int32)."""
    QX = _c(QX, np.int8)
    QW = _c(QW, np.int8)
    M, K = QX.shape
    N, K2 = QW.shape
    assert K == K2
    A = np.empty((M, N), dtype=np.int32)
    ovf = _load().oracle_int_gemm(_ptr(QX), _ptr(QW), M, N, K, _ptr(A), int(nthreads))
    if ovf:
        raise OverflowError(f"{ovf} entries of A do not fit int32")
    return A


def epilogue_f32(A: np.ndarray, sX: np.ndarray, sW: np.ndarray,
                 bias: np.ndarray | None = None) -> np.ndarray:
    """Y = ((float)A * s_X[m]) * s_W[n] in fp32, then + bias[n] (one fp32 add)."""
    A = _c(A, np.int32)
    sX = _c(sX, np.float32)
    sW = _c(sW, np.float32)
    M, N = A.shape
    Y = np.empty((M, N), dtype=np.float32)
    _load().oracle_epilogue_f32(_ptr(A), _ptr(sX), _ptr(sW), M, N, _ptr(Y))
    if bias is not None:
        b = _c(bias, np.float32)
        assert b.shape == (N,)
        _load().oracle_add_bias_f32(_ptr(Y), _ptr(b), M, N)
    return Y


def round_bf16(Y: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    Y = _c(Y, np.float32)
    out = np.empty(Y.shape, dtype=np.uint16)
    _load().oracle_round_bf16(_ptr(Y), _ptr(out), Y.size)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 values (exact: bf16 is the top half
    of an fp32 pattern)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def lora(X: np.ndarray, down: np.ndarray, up: np.ndarray, scale: float,
         nthreads: int = 0) -> np.ndarray:
    """scale * (X down^T) up^T in fp64 on the unrotated X."""
    X = _c(X, np.float64)
    down = _c(down, np.float64)
    up = _c(up, np.float64)
    M, K = X.shape
    R, K2 = down.shape
    N, R2 = up.shape
    assert K == K2 and R == R2
    L = np.empty((M, N), dtype=np.float64)
    _load().oracle_lora(_ptr(X), M, K, _ptr(down), R, _ptr(up), N, float(scale),
                        _ptr(L), int(nthreads))
    return L


def matmul_nt(X: np.ndarray, W: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """Unquantized fp64 X W^T."""
    X = _c(X, np.float64)
    W = _c(W, np.float64)
    M, K = X.shape
    N, K2 = W.shape
    assert K == K2
    Y = np.empty((M, N), dtype=np.float64)
    _load().oracle_matmul_nt(_ptr(X), _ptr(W), M, N, K, _ptr(Y), int(nthreads))
    return Y


# ----------------------------------------------------------------------------
# The two operations of the layer, composed from the steps above.
# ----------------------------------------------------------------------------

def prepare_weight(W: np.ndarray, H: np.ndarray | None = None, nthreads: int = 0):
    """Offline weight prep: W_rot = W H^T, s_W = max|W_rot|/127, Q_W = round.

    Returns a dict with Q_W (int8 [N,K]), s_W (fp32 [N], the stored scale),
    s_W64 (fp64) and pre (fp64 W_rot / s_W, for near-tie analysis).
    """
    W64 = _c(W, np.float32).astype(np.float64)
    Wrot = rotate(W64, H, transpose_h=True, nthreads=nthreads)
    q, s, pre = quantize_rows(Wrot, nthreads=nthreads)
    return {"Q_W": q, "s_W": s.astype(np.float32), "s_W64": s, "pre": pre,
            "W_rot": Wrot}


def rotate_quantize(X: np.ndarray, H: np.ndarray | None = None, nthreads: int = 0,
                    bf16: bool = False):
    """Per-call activation step: X_rot = X H, s_X = max|X_rot|/127, Q_X = round.

    X is fp16 [M, K] (or, with bf16=True, bf16 bit patterns as uint16); each
    value converts to fp64 exactly.  For fp16 inputs every X_rot entry is
    exact in fp64 (K-groups of 256 entries of +-1/16 over fp16's exponent
    range); for bf16 inputs, whose exponents span far wider, the fp64 sums
    are correctly rounded at each step rather than exact.
    Returns a dict with Q_X (int8), s_X (fp32), s_X64 (fp64), pre (fp64).
    """
    if bf16:
        X64 = bf16_to_f32(X).astype(np.float64)
    else:
        X64 = np.asarray(X, dtype=np.float16).astype(np.float64)
    Xrot = rotate(X64, H, transpose_h=False, nthreads=nthreads)
    q, s, pre = quantize_rows(Xrot, nthreads=nthreads)
    return {"Q_X": q, "s_X": s.astype(np.float32), "s_X64": s, "pre": pre,
            "X_rot": Xrot}


def linear(X: np.ndarray, Q_W: np.ndarray, s_W: np.ndarray,
           lora_down: np.ndarray | None = None, lora_up: np.ndarray | None = None,
           lora_scale: float = 0.0, rows: np.ndarray | None = None,
           H: np.ndarray | None = None, nthreads: int = 0, tie_bound: bool = True,
           bias: np.ndarray | None = None, bf16: bool = False):
    """The per-call layer Y = (Q_X Q_W^T) (.) s_X s_W^T [+ bias] [+ lora], on given rows.

    bf16=True: X (and lora_down, lora_up) are bf16 bit patterns (uint16);
    otherwise fp16 arrays.  The bias (fp32 [N]) is added to the fp32 scale
    restore before the LoRA term, in eager's order.

    ``rows`` selects a subset of X's rows (each output row depends on its own
    input row only).  Returns a dict:
      A      int32 [m, N]    exact Q_X Q_W^T
      Y32    fp32  [m, N]    ((float)A * s_X) * s_W  (+ bias)
      L      fp64  [m, N]    LoRA term (zeros without LoRA)
      Y_ref  fp64  [m, N]    Y32 + L (the value an fp16 output is compared to)
      Q_X, s_X, pre          the activation quantization
      near_tie_bound fp64 [m, N]: sum over near-tie k of |Q_W[n,k]| * s_X * s_W,
             the largest change a +-1 flip of near-tie Q_X entries can make
             (test bookkeeping, not part of the layer; skipped when
             tie_bound is False).
    """
    X = np.asarray(X, dtype=np.uint16 if bf16 else np.float16)
    if rows is not None:
        X = X[np.asarray(rows)]
    act = rotate_quantize(X, H, nthreads=nthreads, bf16=bf16)
    A = int_gemm(act["Q_X"], Q_W, nthreads=nthreads)
    Y32 = epilogue_f32(A, act["s_X"], s_W, bias)
    M, N = Y32.shape
    if lora_down is not None and lora_up is not None and np.asarray(lora_down).shape[0] > 0:
        def f64(a):
            return bf16_to_f32(a).astype(np.float64) if bf16 else \
                np.asarray(a, dtype=np.float16).astype(np.float64)
        L = lora(f64(X), f64(lora_down), f64(lora_up), lora_scale, nthreads=nthreads)
    else:
        L = np.zeros((M, N), dtype=np.float64)
    near = near_tie_mask(act["pre"]) if tie_bound else np.zeros((1, 1), dtype=bool)
    if near.any():
        # flips[m, n] = sum_k near[m,k] * |Q_W[n,k]|: small integers, exact in fp64
        absQW = np.abs(np.asarray(Q_W, dtype=np.int8).astype(np.float64))
        flips = near.astype(np.float64) @ absQW.T
    else:
        flips = np.zeros((M, N))
    bound = flips * act["s_X"].astype(np.float64)[:, None] * \
        np.asarray(s_W, dtype=np.float64)[None, :]
    return {"A": A, "Y32": Y32, "L": L, "Y_ref": Y32.astype(np.float64) + L,
            "Q_X": act["Q_X"], "s_X": act["s_X"], "s_X64": act["s_X64"],
            "pre": act["pre"], "near_tie_bound": bound}


def near_tie_mask(pre: np.ndarray, eps: float = NEAR_TIE) -> np.ndarray:
    """True where a pre-round value lies within eps of a .5 tie."""
    frac = np.abs(pre - np.floor(pre) - 0.5)
    return frac < eps
