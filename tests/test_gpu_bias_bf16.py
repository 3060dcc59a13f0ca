"""convrot_linear_ex: bf16 activations and outputs and an fp32 bias (page
"[PR #249] Add an mps backend: weight-only INT8 and W4A8/W6A8 linears for
Apple GPUs", section "Design": bias in eager's order, bf16 with torch's cast).

* Bit-exact: with fp16 X, Y must equal the oracle's epilogue (scale restore,
  then its own fp32 bias add, then one rounding to fp16 or bf16) applied to
  the exact product of the GPU's own activation codes -- on every engine
  (one-SM tiles of each width, the CTA-pair K split, CTA-pair MMA tiles,
  split K through L2, the small-M engine) and with N not a multiple of 8
  (plain stores instead of TMA stores).
* bf16 input is widened exactly: on values that fp16 and bf16 both hold, the
  bf16 path gives the fp16 path's Y bit for bit.
* Against the oracle within tolerance: bf16 in and out, bias, bf16 LoRA.
"""
import numpy as np
import pytest

import oracle
import workloads
import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = gu.torch


@pytest.fixture
def modes():
    gu.require_gpu()
    yield
    cr.convrot_set_split_mode(0)
    cr.convrot_set_pair_mma(0)
    cr.convrot_set_tile_override(0, 0)


def _bias(N, seed):
    return (np.random.default_rng(seed).standard_normal(N) * 0.5).astype(np.float32)


def _run(X, Q_W, s_W, img, bias, y_dtype, x_dtype=torch.float16, lora=None):
    """X: a torch tensor on the device; returns Y as a host uint16 array."""
    M, K = X.shape
    N = Q_W.shape[0]
    R = 0 if lora is None else lora[0].shape[0]
    ws = gu.workspace(cr.convrot_linear_workspace_bytes(M, N, K, R, img is not None))
    Y = torch.empty((M, N), dtype=y_dtype, device="cuda")
    b = None if bias is None else gu.dev(bias)
    down, up, scale = (None, None, 0.0) if lora is None else lora
    cr.convrot_linear_ex(X.to(x_dtype), Q_W, s_W, Y, ws, W_img=img, bias=b, lora_down=down,
                         lora_up=up, lora_scale=scale)
    gu.check_no_device_error()
    return Y.view(torch.int16).cpu().numpy().view(np.uint16)


def _expected(X16, Q_W, s_W, bias, bf16_out):
    """The oracle epilogue on the GPU's own codes (fp16 X)."""
    QX, sX = gu.rotate_quantize(X16)
    A = oracle.int_gemm(QX, gu.host(Q_W) if not isinstance(Q_W, np.ndarray) else Q_W)
    Y32 = oracle.epilogue_f32(A, sX, gu.host(s_W) if not isinstance(s_W, np.ndarray) else s_W,
                              bias)
    return oracle.round_bf16(Y32) if bf16_out else Y32.astype(np.float16).view(np.uint16)


ENGINES = {
    "auto": lambda: None,
    "bn64": lambda: cr.convrot_set_tile_override(64, 1),
    "bn128": lambda: cr.convrot_set_tile_override(128, 1),
    "bn256": lambda: cr.convrot_set_tile_override(256, 1),
    "pair_split": lambda: cr.convrot_set_split_mode(2),
    "pair_mma": lambda: (cr.convrot_set_split_mode(1), cr.convrot_set_pair_mma(2)),
    "l2_split": lambda: (cr.convrot_set_split_mode(1), cr.convrot_set_pair_mma(1),
                         cr.convrot_set_tile_override(64, 4)),
}


@pytest.mark.parametrize("bf16_out", [False, True], ids=["f16out", "bf16out"])
@pytest.mark.parametrize("engine", list(ENGINES), ids=list(ENGINES))
@pytest.mark.parametrize("shape", [(300, 640, 1024), (1024, 256, 2048), (16, 264, 512),
                                   (129, 77, 768)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bias_bit_exact_on_every_engine(modes, shape, engine, bf16_out):
    M, N, K = shape
    X = workloads.make_x(M, K, 81, workloads.n_outliers(K))
    Q_W, s_W, img = gu.prepare_weight(workloads.make_w(N, K, 81))
    bias = _bias(N, 82)
    exp = _expected(X, Q_W, s_W, bias, bf16_out)
    ENGINES[engine]()
    got = _run(gu.dev(X), Q_W, s_W, img, bias, torch.bfloat16 if bf16_out else torch.float16)
    diff = int((got != exp).sum())
    assert diff == 0, f"{diff} of {got.size} outputs differ"


def test_no_bias_bf16_out_is_the_rounding_of_the_f16_path_value(modes):
    # Without a bias the fp32 value is the plain scale restore: the bf16
    # output is its bf16 rounding (checked against the oracle's epilogue).
    M, N, K = 1024, 2048, 2048
    X = workloads.make_x(M, K, 83, workloads.n_outliers(K))
    Q_W, s_W, img = gu.prepare_weight(workloads.make_w(N, K, 83))
    got = _run(gu.dev(X), Q_W, s_W, img, None, torch.bfloat16)
    assert np.array_equal(got, _expected(X, Q_W, s_W, None, True))


@pytest.mark.parametrize("shape", [(1024, 2048, 2048), (300, 640, 1024), (8, 256, 768),
                                   (64, 512, 16384)], ids=lambda s: "x".join(map(str, s)))
def test_bf16_input_widened_exactly(modes, shape):
    # Values held exactly by fp16 and bf16 alike (integers below 256 times
    # powers of two): both input paths must give the same Y bit for bit.
    M, N, K = shape
    rng = np.random.default_rng(84)
    X = (rng.integers(-200, 201, (M, K)) * 2.0 ** rng.integers(-6, 2, (M, K))).astype(np.float16)
    Q_W, s_W, img = gu.prepare_weight(workloads.make_w(N, K, 84))
    bias = _bias(N, 85)
    Xd = gu.dev(X)
    y16 = _run(Xd, Q_W, s_W, img, bias, torch.float16, x_dtype=torch.float16)
    yb = _run(Xd, Q_W, s_W, img, bias, torch.float16, x_dtype=torch.bfloat16)
    assert np.array_equal(yb, y16)


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("R", [0, 32])
def test_bf16_in_out_with_bias_matches_oracle(modes, R):
    M, N, K = 512, 1024, 2048
    seed = 86
    Xf = workloads.make_x(M, K, seed, workloads.n_outliers(K)).astype(np.float32)
    Xb = _bf16_bits(Xf)
    prep = oracle.prepare_weight(workloads.make_w(N, K, seed))
    bias = _bias(N, 87)
    lora = None
    down_b = up_b = None
    if R:
        down, up = workloads.make_lora(N, K, R, seed)
        down_b, up_b = _bf16_bits(down.astype(np.float32)), _bf16_bits(up.astype(np.float32))
        def dev_b(bits):
            return gu.dev(bits.view(np.int16)).view(torch.bfloat16)
        lora = (dev_b(down_b), dev_b(up_b), 0.8)
    Xd = gu.dev(Xb.view(np.int16)).view(torch.bfloat16)
    img = gu.dev(prep["Q_W"].astype(np.float16))
    got = _run(Xd, gu.dev(prep["Q_W"]), gu.dev(prep["s_W"]), img, bias, torch.bfloat16,
               x_dtype=torch.bfloat16, lora=lora)
    rows = np.unique(np.concatenate([[0, M - 1],
                                     np.random.default_rng(seed).choice(M, 60, replace=False)]))
    ref = oracle.linear(Xb, prep["Q_W"], prep["s_W"], lora_down=down_b, lora_up=up_b,
                        lora_scale=0.8 if R else 0.0, rows=rows, bias=bias, bf16=True)
    y = oracle.bf16_to_f32(got[rows])
    # bf16 keeps 8 significant bits: half an ulp is 2^-8 relative.
    gu.compare_y(y, ref, rtol=2.0 ** -8 + 1e-4, atol=1e-3)
