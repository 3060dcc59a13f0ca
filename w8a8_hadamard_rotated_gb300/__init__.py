"""Python binding of the INT8ConvRot (W8A8 Hadamard-rotated) linear library.

The compute lives in the CUDA library ``libconvrot.so`` (built from
``csrc/`` by :func:`build`); its C ABI is declared in ``include/convrot.h``.
This module only marshals arguments: every function named ``convrot_*`` here
calls the C function of the same name with device pointers taken from torch
tensors and the current torch CUDA stream.  There is no CPU or PyTorch
fallback: if the library is missing or the device is not sm_103, the calls
raise :class:`ConvRotError`.

The layer (page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix,
and MLX", section "What changed in the computation"):
  prep   W_rot = W H^T, s_W = max|W_rot|/127 per row, Q_W = round(W_rot / s_W)
  call   X_rot = X H, s_X = max|X_rot|/127 per row, Q_X = round(X_rot / s_X),
         A = Q_X Q_W^T (int32), Y = A (.) s_X s_W^T  [+ lora_scale (X down^T) up^T]
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build_mod

__all__ = [
    "ConvRotError", "build", "library_path", "load",
    "CONVROT_OK", "CONVROT_ERR_INVALID_ARG", "CONVROT_ERR_UNSUPPORTED_DEVICE",
    "CONVROT_ERR_CUDA", "CONVROT_ERR_TIMEOUT", "CONVROT_ERR_WORKSPACE",
    "CONVROT_PATH_AUTO", "CONVROT_PATH_TCGEN05", "CONVROT_PATH_SKINNY",
    "convrot_status_string", "convrot_version", "convrot_weight_image_bytes",
    "convrot_linear_workspace_bytes", "convrot_linear_host_workspace_bytes",
    "convrot_gemm_workspace_bytes", "convrot_prepare_weight", "convrot_linear",
    "convrot_linear_host", "convrot_linear_prologue", "convrot_linear_gemm",
    "convrot_check_device_error", "convrot_rotate_quantize",
    "convrot_gemm_i32", "convrot_gemm_dequant", "convrot_set_tile_override",
    "convrot_set_fused", "convrot_set_small_m_engine", "convrot_set_small_m_weights_early",
    "convrot_set_skinny_engine",
    "convrot_set_split_mode", "convrot_set_pair_mma", "convrot_linear_ex", "convrot_rotate",
    "CONVROT_DTYPE_F16", "CONVROT_DTYPE_BF16",
    "convrot_selftest_wait_timeout",
    "convrot_linear_noalloc", "CONVROT_DETAIL_SELFTEST", "CONVROT_NOALLOC_SCRATCH_BYTES", "CONVROT_NOALLOC_MAX_M", "CONVROT_MAX_DIM",
    "convrot_measure_engine_peak", "CONVROT_PEAK_MMA_S8", "CONVROT_PEAK_TCGEN05_F16",
    "CONVROT_PEAK_MMA_F16", "CONVROT_PEAK_DP4A",
    "convrot_linear_workspace_layout", "CONVROT_CODES_I8", "CONVROT_CODES_F16",
    "convrot_linear_kernel_count", "convrot_plan_gemm", "convrot_plan_small_m",
    "CONVROT_SMALL_M_NONE", "CONVROT_SMALL_M_ONE_DP4A", "CONVROT_SMALL_M_ONE_MMA",
    "CONVROT_SMALL_M_ONE_SHARED", "CONVROT_SMALL_M_TWO_F16", "CONVROT_SMALL_M_TWO_S8",
]

CONVROT_OK = 0
CONVROT_ERR_INVALID_ARG = 1
CONVROT_ERR_UNSUPPORTED_DEVICE = 2
CONVROT_ERR_CUDA = 3
CONVROT_ERR_TIMEOUT = 4
CONVROT_ERR_WORKSPACE = 5

CONVROT_PATH_AUTO = 0
CONVROT_PATH_TCGEN05 = 1
CONVROT_PATH_SKINNY = 2

CONVROT_MAX_K = 65536
CONVROT_MAX_DIM = 2**31 - 1
CONVROT_PEAK_MMA_S8 = 0
CONVROT_PEAK_TCGEN05_F16 = 1
CONVROT_PEAK_MMA_F16 = 2
CONVROT_PEAK_DP4A = 3
CONVROT_CODES_I8 = 0
CONVROT_CODES_F16 = 1
CONVROT_NOALLOC_SCRATCH_BYTES = 4 << 20
CONVROT_NOALLOC_MAX_M = 16

_lock = threading.Lock()
_lib = None


class ConvRotError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = int(status)
        super().__init__(f"{fn} failed: {convrot_status_string(status)} (status {status})")


def build(force: bool = False) -> str:
    """Compile libconvrot.so for sm_103a (in-tree) and return its path."""
    return _build_mod.build(force=force)


def library_path() -> str:
    return _build_mod.LIB


_SIGS = {
    "convrot_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "convrot_version": (ctypes.c_int, []),
    "convrot_weight_image_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "convrot_linear_workspace_bytes": (
        ctypes.c_size_t, [ctypes.c_int64] * 4 + [ctypes.c_int]),
    "convrot_linear_host_workspace_bytes": (
        ctypes.c_size_t, [ctypes.c_int64] * 4 + [ctypes.c_int]),
    "convrot_gemm_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64] * 3 + [ctypes.c_int]),
    "convrot_prepare_weight": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p]),
    "convrot_linear": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "convrot_rotate": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]),
    "convrot_linear_ex": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "convrot_linear_host": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "convrot_linear_prologue": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "convrot_linear_gemm": (ctypes.c_int, [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "convrot_check_device_error": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]),
    "convrot_rotate_quantize": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p]),
    "convrot_gemm_i32": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "convrot_gemm_dequant": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
        ctypes.c_size_t, ctypes.c_void_p]),
    "convrot_set_tile_override": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "convrot_set_fused": (ctypes.c_int, [ctypes.c_int]),
    "convrot_set_small_m_engine": (ctypes.c_int, [ctypes.c_int]),
    "convrot_set_small_m_weights_early": (ctypes.c_int, [ctypes.c_int]),
    "convrot_set_skinny_engine": (ctypes.c_int, [ctypes.c_int]),
    "convrot_set_split_mode": (ctypes.c_int, [ctypes.c_int]),
    "convrot_set_pair_mma": (ctypes.c_int, [ctypes.c_int]),
    "convrot_set_hadamard_base": (ctypes.c_int, [ctypes.c_void_p]),
    "convrot_plan_gemm": (ctypes.c_int, [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int64, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
        ctypes.POINTER(ctypes.c_int)]),
    "convrot_plan_small_m": (ctypes.c_int, [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
        ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "convrot_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_int64, ctypes.c_void_p]),
    "convrot_linear_kernel_count": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                    ctypes.c_int64, ctypes.c_int]),
    "convrot_linear_workspace_layout": (ctypes.c_int, [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
        ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int),
        ctypes.POINTER(ctypes.c_int64)]),
    "convrot_measure_engine_peak": (ctypes.c_int, [
        ctypes.c_int, ctypes.c_int64, ctypes.POINTER(ctypes.c_double),
        ctypes.POINTER(ctypes.c_float), ctypes.c_void_p]),
    "convrot_linear_noalloc": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]),
}


def load():
    """Load libconvrot.so (raises ConvRotError-like RuntimeError if missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library not built: {path} is missing (run "
                "w8a8_hadamard_rotated_gb300.build() or __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


# ----------------------------------------------------------------------------
# Marshalling helpers (torch is imported lazily: the size queries and status
# strings work without it).
# ----------------------------------------------------------------------------

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, status: int):
    if status != CONVROT_OK:
        raise ConvRotError(fn, status)


def convrot_status_string(status: int) -> str:
    return load().convrot_status_string(int(status)).decode()


def convrot_version() -> int:
    return int(load().convrot_version())


def convrot_weight_image_bytes(N: int, K: int) -> int:
    return int(load().convrot_weight_image_bytes(N, K))


def convrot_linear_workspace_bytes(M: int, N: int, K: int, R: int = 0,
                                   with_weight_image: bool = True) -> int:
    return int(load().convrot_linear_workspace_bytes(M, N, K, R, int(bool(with_weight_image))))


def convrot_linear_host_workspace_bytes(M: int, N: int, K: int, R: int = 0,
                                        with_weight_image: bool = True) -> int:
    return int(load().convrot_linear_host_workspace_bytes(M, N, K, R,
                                                          int(bool(with_weight_image))))


def convrot_gemm_workspace_bytes(M: int, N: int, K: int, path: int = CONVROT_PATH_AUTO) -> int:
    return int(load().convrot_gemm_workspace_bytes(M, N, K, path))


def convrot_prepare_weight(W, Q_W, s_W, W_img=None, stream=None) -> None:
    """W fp32 [N,K] -> Q_W int8 [N,K], s_W fp32 [N] (+ W_img fp16 [N,K])."""
    N, K = W.shape
    _check("convrot_prepare_weight", load().convrot_prepare_weight(
        _ptr(W), N, K, _ptr(Q_W), _ptr(s_W), _ptr(W_img), _stream(stream)))


CONVROT_DTYPE_F16 = 0
CONVROT_DTYPE_BF16 = 1


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return CONVROT_DTYPE_F16
    if t.dtype == torch.bfloat16:
        return CONVROT_DTYPE_BF16
    raise TypeError(f"fp16 or bf16 expected, got {t.dtype}")


def convrot_linear(X, Q_W, s_W, Y, workspace, W_img=None, lora_down=None, lora_up=None,
                   lora_scale: float = 0.0, stream=None, bias=None) -> None:
    """Y [M,N] = the INT8ConvRot layer of X [M,K] (device tensors).

    X and Y are fp16 or bf16 (the LoRA weights take X's type); bias is an
    optional fp32 [N].  fp16 in and out without a bias calls convrot_linear,
    anything else convrot_linear_ex.
    """
    M, K = X.shape
    N = Q_W.shape[0]
    R = 0 if lora_down is None else lora_down.shape[0]
    xd, yd = _dtype_code(X), _dtype_code(Y)
    if xd == CONVROT_DTYPE_F16 and yd == CONVROT_DTYPE_F16 and bias is None:
        _check("convrot_linear", load().convrot_linear(
            _ptr(X), M, K, _ptr(Q_W), _ptr(s_W), _ptr(W_img), N, _ptr(lora_down), _ptr(lora_up),
            R, float(lora_scale), _ptr(Y), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream)))
        return
    convrot_linear_ex(X, Q_W, s_W, Y, workspace, W_img=W_img, bias=bias, lora_down=lora_down,
                      lora_up=lora_up, lora_scale=lora_scale, stream=stream)


def convrot_rotate(X, X_rot, stream=None) -> None:
    """X_rot fp16 [M, K] = X H (the rotation alone, for a weight-only layer)."""
    M, K = X.shape
    _check("convrot_rotate", load().convrot_rotate(_ptr(X), M, K, _ptr(X_rot), _stream(stream)))


def convrot_linear_ex(X, Q_W, s_W, Y, workspace, W_img=None, bias=None, lora_down=None,
                      lora_up=None, lora_scale: float = 0.0, stream=None) -> None:
    """convrot_linear_ex: X, Y fp16 or bf16 (types from the tensors), optional
    fp32 bias [N]; LoRA weights of X's type."""
    M, K = X.shape
    N = Q_W.shape[0]
    R = 0 if lora_down is None else lora_down.shape[0]
    _check("convrot_linear_ex", load().convrot_linear_ex(
        _ptr(X), _dtype_code(X), M, K, _ptr(Q_W), _ptr(s_W), _ptr(W_img), N, _ptr(bias),
        _ptr(lora_down), _ptr(lora_up), R, float(lora_scale), _ptr(Y), _dtype_code(Y),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def convrot_linear_host(X_host, Q_W, s_W, Y_host, workspace, W_img=None, lora_down=None,
                        lora_up=None, lora_scale: float = 0.0, stream=None) -> None:
    """convrot_linear with X_host / Y_host in (pinned) host memory."""
    M, K = X_host.shape
    N = Q_W.shape[0]
    R = 0 if lora_down is None else lora_down.shape[0]
    _check("convrot_linear_host", load().convrot_linear_host(
        _ptr(X_host), M, K, _ptr(Q_W), _ptr(s_W), _ptr(W_img), N, _ptr(lora_down),
        _ptr(lora_up), R, float(lora_scale), _ptr(Y_host), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def convrot_linear_prologue(X, N: int, workspace, lora_down=None, with_weight_image=True,
                            stream=None) -> None:
    """First stage of convrot_linear: rotate + quantize X into the workspace."""
    M, K = X.shape
    R = 0 if lora_down is None else lora_down.shape[0]
    _check("convrot_linear_prologue", load().convrot_linear_prologue(
        _ptr(X), M, K, N, _ptr(lora_down), R, int(bool(with_weight_image)), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def convrot_linear_gemm(M: int, K: int, Q_W, s_W, Y, workspace, W_img=None, lora_up=None,
                        lora_scale: float = 0.0, stream=None) -> None:
    """Second stage of convrot_linear: product + epilogue from the workspace."""
    N = Q_W.shape[0]
    R = 0 if lora_up is None else lora_up.shape[1]
    _check("convrot_linear_gemm", load().convrot_linear_gemm(
        M, K, _ptr(Q_W), _ptr(s_W), _ptr(W_img), N, _ptr(lora_up), R, float(lora_scale),
        _ptr(Y), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def convrot_check_device_error(stream=None) -> int:
    """Synchronize; return the device error detail code (0 = none)."""
    detail = ctypes.c_int(0)
    status = load().convrot_check_device_error(_stream(stream), ctypes.byref(detail))
    if status not in (CONVROT_OK, CONVROT_ERR_TIMEOUT):
        raise ConvRotError("convrot_check_device_error", status)
    return int(detail.value)


def convrot_rotate_quantize(X, Q_X, s_X, stream=None) -> None:
    M, K = X.shape
    _check("convrot_rotate_quantize", load().convrot_rotate_quantize(
        _ptr(X), M, K, _ptr(Q_X), _ptr(s_X), _stream(stream)))


def convrot_gemm_i32(Q_X, Q_W, A, workspace, path: int = CONVROT_PATH_AUTO, stream=None) -> None:
    M, K = Q_X.shape
    N = Q_W.shape[0]
    _check("convrot_gemm_i32", load().convrot_gemm_i32(
        _ptr(Q_X), _ptr(Q_W), M, N, K, _ptr(A), int(path), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def convrot_gemm_dequant(Q_X, s_X, Q_W, s_W, Y, workspace, path: int = CONVROT_PATH_AUTO,
                         stream=None) -> None:
    M, K = Q_X.shape
    N = Q_W.shape[0]
    _check("convrot_gemm_dequant", load().convrot_gemm_dequant(
        _ptr(Q_X), _ptr(s_X), _ptr(Q_W), _ptr(s_W), M, N, K, _ptr(Y), int(path),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def convrot_set_tile_override(bn: int = 0, splits: int = 0) -> None:
    _check("convrot_set_tile_override", load().convrot_set_tile_override(int(bn), int(splits)))


CONVROT_DETAIL_SELFTEST = 9


def convrot_selftest_wait_timeout(budget_cycles: int, stream=None) -> None:
    """Launch the failure-detection self-test (a wait that runs out)."""
    _check("convrot_selftest_wait_timeout",
           load().convrot_selftest_wait_timeout(int(budget_cycles), _stream(stream)))


def convrot_linear_kernel_count(M: int, N: int, K: int, R: int = 0,
                                with_weight_image: bool = True) -> int:
    """Kernels one convrot_linear call (fp16 X and Y) with these sizes launches
    on the current device under the current engine settings."""
    n = int(load().convrot_linear_kernel_count(int(M), int(N), int(K), int(R),
                                                1 if with_weight_image else 0))
    if n < 0:
        raise ValueError(f"convrot_linear_kernel_count: sizes rejected ({M}, {N}, {K}, {R})")
    return n


def convrot_linear_workspace_layout(M: int, N: int, K: int, R: int = 0,
                                    with_weight_image: bool = True):
    """Where the prologue leaves Q_X and s_X in the workspace (parity only):
    (codes byte offset, CONVROT_CODES_I8 or CONVROT_CODES_F16, s_X byte offset)."""
    qo, fmt, so = ctypes.c_int64(), ctypes.c_int(), ctypes.c_int64()
    _check("convrot_linear_workspace_layout", load().convrot_linear_workspace_layout(
        int(M), int(N), int(K), int(R), int(bool(with_weight_image)), ctypes.byref(qo),
        ctypes.byref(fmt), ctypes.byref(so)))
    return qo.value, fmt.value, so.value


def convrot_measure_engine_peak(engine: int, reps: int, stream=None):
    """Back-to-back MMAs of one exact int8 product engine on every SM
    (measurement only).  Returns (operations, milliseconds); synchronizes."""
    ops = ctypes.c_double(0.0)
    ms = ctypes.c_float(0.0)
    _check("convrot_measure_engine_peak",
           load().convrot_measure_engine_peak(int(engine), int(reps), ctypes.byref(ops),
                                              ctypes.byref(ms), _stream(stream)))
    return ops.value, float(ms.value)


def convrot_set_split_mode(mode: int = 0) -> None:
    """Testing hook: 0 automatic, 1 never split K across a CTA pair, 2 always
    where it applies, 3 the streaming CTA-pair split wherever it applies."""
    _check("convrot_set_split_mode", load().convrot_set_split_mode(int(mode)))


def convrot_set_pair_mma(mode: int = 0) -> None:
    """Testing hook: 0 automatic, 1 never run GEMM tiles on CTA-pair MMAs, 2
    always where they apply."""
    _check("convrot_set_pair_mma", load().convrot_set_pair_mma(int(mode)))


CONVROT_ENGINE_ONE_SM = 0
CONVROT_ENGINE_PAIR_SPLIT = 1
CONVROT_ENGINE_PAIR_MMA = 2
CONVROT_ENGINE_L2_SPLIT = 3
CONVROT_ENGINE_PAIR_STREAM = 4


def convrot_plan_gemm(M: int, N: int, K: int, sms: int = 152, pair_clusters_128: int = 76,
                      pair_clusters_256: int = 76, tma_store: bool = True, R: int = 0):
    """The tensor-core GEMM's plan on the host: (tile width, K splits, engine)."""
    bn, sp, eng = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check("convrot_plan_gemm", load().convrot_plan_gemm(
        M, N, K, sms, pair_clusters_128, pair_clusters_256, int(bool(tma_store)), R,
        ctypes.byref(bn), ctypes.byref(sp), ctypes.byref(eng)))
    return bn.value, sp.value, eng.value


CONVROT_SMALL_M_NONE = 0
CONVROT_SMALL_M_ONE_DP4A = 1
CONVROT_SMALL_M_ONE_MMA = 2
CONVROT_SMALL_M_ONE_SHARED = 3
CONVROT_SMALL_M_TWO_F16 = 4
CONVROT_SMALL_M_TWO_S8 = 5


def convrot_plan_small_m(M: int, N: int, K: int, sms: int = 152):
    """The small-M engine of an fp16 layer on the host: (engine, K splits,
    column blocks per cluster)."""
    eng, sp, bl = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check("convrot_plan_small_m", load().convrot_plan_small_m(
        M, N, K, sms, ctypes.byref(eng), ctypes.byref(sp), ctypes.byref(bl)))
    return eng.value, sp.value, bl.value


SYLVESTER_BASE = ((1, 1, 1, 1), (1, -1, 1, -1), (1, 1, -1, -1), (1, -1, -1, 1))


def convrot_set_hadamard_base(base=None) -> None:
    """The 4x4 Hadamard base of H for every later call (None: Sylvester's).

    base: a 4x4 array-like of +1/-1 entries, symmetric, with B B^T = 4 I."""
    if base is None:
        _check("convrot_set_hadamard_base", load().convrot_set_hadamard_base(None))
        return
    flat = [int(v) for row in base for v in row]
    if len(flat) != 16 or any(v not in (-1, 1) for v in flat):
        raise ValueError("a 4x4 base of +1/-1 entries expected")
    buf = (ctypes.c_int8 * 16)(*flat)
    _check("convrot_set_hadamard_base",
           load().convrot_set_hadamard_base(ctypes.cast(buf, ctypes.c_void_p)))


def convrot_set_fused(enable: bool = True) -> None:
    """Select convrot_linear's single-kernel engine (True) or the default
    two-kernel engine (False) for later calls."""
    _check("convrot_set_fused", load().convrot_set_fused(1 if enable else 0))


def convrot_set_small_m_engine(mode: int) -> None:
    """Engine for layers with M <= 16 (fp16 in and out, no bias, no LoRA):
    0 (default) the one-kernel layer's dp4a form at M <= 2, two kernels
    otherwise; 1 two kernels; 2 the dp4a form at every M; 3 the fp16-MMA form at
    every M; 4 the form whose clusters share the rotation among column blocks
    where it applies (0 elsewhere).  Same bits from all."""
    _check("convrot_set_small_m_engine", load().convrot_set_small_m_engine(int(mode)))


def convrot_set_small_m_weights_early(enable: bool = True) -> None:
    """True (default): the one-kernel small-M layer copies its weight before
    it waits for the kernel ahead of it on the stream (the weight must not be
    written by that kernel if it lets dependents start early; no kernel of
    this library that writes int8 data does).  False: after.  Same bits."""
    _check("convrot_set_small_m_weights_early",
           load().convrot_set_small_m_weights_early(1 if enable else 0))


def convrot_set_skinny_engine(mode: int) -> None:
    """Testing hook for the two-kernel path's small-M GEMM: 0 (default) the
    fp16-MMA bulk-copy kernel at M >= 3 where it applies, else the s8 kernel;
    1 always the s8 kernel; 2 the fp16-MMA kernel wherever it applies."""
    _check("convrot_set_skinny_engine", load().convrot_set_skinny_engine(int(mode)))


def convrot_linear_noalloc(X, Q_W, s_W, Y, stream=None) -> None:
    """Small-M layer (M <= 16, no LoRA) with the library's own fixed scratch.

    For callers that cannot give the library a workspace and cannot allocate
    device memory (plugin hosts without a scratch buffer, engines that forbid
    allocation once running).  Calls on one device share the scratch: do not
    let them overlap on the GPU.
    """
    M, K = X.shape
    N = Q_W.shape[0]
    _check("convrot_linear_noalloc", load().convrot_linear_noalloc(
        _ptr(X), M, K, _ptr(Q_W), _ptr(s_W), N, _ptr(Y), _stream(stream)))
