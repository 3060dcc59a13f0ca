"""Helpers shared by the GPU parity tests: device buffers and calls through
the C ABI binding.  Inputs come from ``workloads``; expected values from
``oracle``; nothing here computes any part of the layer."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import w8a8_hadamard_rotated_gb300 as cr  # noqa: E402


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    major, minor = torch.cuda.get_device_capability()
    if (major, minor) != (10, 3):
        pytest.skip("needs sm_103")
    cr.build()
    cr.load()


def dev(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


def workspace(nbytes: int):
    # 256-byte aligned (the caching allocator hands out 512-byte aligned blocks)
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device="cuda")


def check_no_device_error():
    assert cr.convrot_check_device_error() == 0


def rotate_quantize(X: np.ndarray):
    M, K = X.shape
    Xd = dev(X)
    Q = torch.empty((M, K), dtype=torch.int8, device="cuda")
    s = torch.empty((M,), dtype=torch.float32, device="cuda")
    cr.convrot_rotate_quantize(Xd, Q, s)
    check_no_device_error()
    return host(Q), host(s)


def prepare_weight(W: np.ndarray, with_img: bool = True):
    N, K = W.shape
    Wd = dev(W.astype(np.float32))
    Q = torch.empty((N, K), dtype=torch.int8, device="cuda")
    s = torch.empty((N,), dtype=torch.float32, device="cuda")
    img = torch.empty((N, K), dtype=torch.float16, device="cuda") if with_img else None
    cr.convrot_prepare_weight(Wd, Q, s, img)
    check_no_device_error()
    return Q, s, img


def gemm_i32(QX: np.ndarray, QW: np.ndarray, path=cr.CONVROT_PATH_AUTO):
    M, K = QX.shape
    N = QW.shape[0]
    A = torch.empty((M, N), dtype=torch.int32, device="cuda")
    ws = workspace(cr.convrot_gemm_workspace_bytes(M, N, K, path))
    cr.convrot_gemm_i32(dev(QX), dev(QW), A, ws, path)
    check_no_device_error()
    return host(A)


def gemm_dequant(QX, sX, QW, sW, path=cr.CONVROT_PATH_AUTO):
    M, K = QX.shape
    N = QW.shape[0]
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = workspace(cr.convrot_gemm_workspace_bytes(M, N, K, path))
    cr.convrot_gemm_dequant(dev(QX), dev(sX.astype(np.float32)), dev(QW),
                            dev(sW.astype(np.float32)), Y, ws, path)
    check_no_device_error()
    return host(Y)


def linear(X: np.ndarray, Q_W, s_W, W_img=None, lora_down=None, lora_up=None,
           lora_scale=0.0):
    """Runs convrot_linear; Q_W / s_W / W_img may be numpy arrays or device tensors."""
    M, K = X.shape
    if isinstance(Q_W, np.ndarray):
        Q_W = dev(Q_W)
    if isinstance(s_W, np.ndarray):
        s_W = dev(s_W.astype(np.float32))
    if isinstance(W_img, np.ndarray):
        W_img = dev(W_img.astype(np.float16))
    N = Q_W.shape[0]
    R = 0 if lora_down is None else lora_down.shape[0]
    down = None if lora_down is None else dev(lora_down)
    up = None if lora_up is None else dev(lora_up)
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = workspace(cr.convrot_linear_workspace_bytes(M, N, K, R, W_img is not None))
    cr.convrot_linear(dev(X), Q_W, s_W, Y, ws, W_img=W_img, lora_down=down, lora_up=up,
                      lora_scale=lora_scale)
    check_no_device_error()
    return host(Y)


def compare_q(q_gpu: np.ndarray, q_ref: np.ndarray, pre: np.ndarray, near_tie: float = 1e-4):
    """Q exact except +-1 where the oracle's pre-round value is within
    `near_tie` of a .5 tie.  Returns the number of such tie flips."""
    d = q_gpu.astype(np.int32) - q_ref.astype(np.int32)
    bad = d != 0
    if not bad.any():
        return 0
    frac = np.abs(pre - np.floor(pre) - 0.5)
    allowed = (np.abs(d) == 1) & (frac < near_tie)
    assert np.all(allowed[bad]), (
        f"{int((bad & ~allowed).sum())} quantized values differ away from ties; "
        f"first at {np.argwhere(bad & ~allowed)[:5].tolist()}")
    return int(bad.sum())


def compare_y(y_gpu: np.ndarray, ref: dict, rtol=1e-3, atol=1e-3):
    """fp16 Y against the oracle's Y_ref within rtol*|Y_ref| + atol, widened by
    the effect of +-1 flips at near-tie activation codes (near_tie_bound)."""
    y = y_gpu.astype(np.float64)
    yr = ref["Y_ref"]
    tol = atol + rtol * np.abs(yr) + ref["near_tie_bound"]
    err = np.abs(y - yr)
    ok = err <= tol
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        raise AssertionError(
            f"{int((~ok).sum())} of {ok.size} outputs off; worst excess "
            f"{float((err - tol).max()):.3g}; first {idx.tolist()} "
            f"gpu={[float(y[tuple(i)]) for i in idx]} ref={[float(yr[tuple(i)]) for i in idx]}")
    return float(err.max())
