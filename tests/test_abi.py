"""The C ABI library builds, loads and exports every entry point include/convrot.h
declares, and rejects bad arguments before any CUDA call (so these run on a
machine without a GPU)."""
import ctypes
import os
import re

import pytest

import w8a8_hadamard_rotated_gb300 as cr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "convrot.h")


@pytest.fixture(scope="module")
def lib():
    cr.build()
    return cr.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(convrot_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_two_layer_calls():
    names = declared_functions()
    assert "convrot_prepare_weight" in names and "convrot_linear" in names
    assert len(names) >= 10


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert cr.__dict__.get(name) is not None, f"binding lacks {name}"


def test_status_strings_and_version(lib):
    assert cr.convrot_status_string(cr.CONVROT_OK) == "ok"
    assert "workspace" in cr.convrot_status_string(cr.CONVROT_ERR_WORKSPACE)
    assert cr.convrot_status_string(99) == "unknown status"
    assert cr.convrot_version() >= 100


def test_size_queries(lib):
    assert cr.convrot_weight_image_bytes(8192, 2048) == 2 * 8192 * 2048
    ws = cr.convrot_linear_workspace_bytes(1024, 2048, 2048, 0, True)
    assert ws >= 2 * 1024 * 2048 + 4 * 1024          # fp16 Q_X image + s_X
    ws2 = cr.convrot_linear_workspace_bytes(1024, 2048, 2048, 0, False)
    assert ws2 >= ws + 2 * 2048 * 2048                 # plus the widened weight
    assert cr.convrot_linear_workspace_bytes(1024, 2048, 2048, 32, True) >= ws + 4 * 1024 * 32
    assert cr.convrot_linear_workspace_bytes(1024, 2048, 300, 0, True) == 0  # bad K
    assert cr.convrot_linear_host_workspace_bytes(16, 64, 256, 0, True) >= \
        cr.convrot_linear_workspace_bytes(16, 64, 256, 0, True) + 2 * 16 * 256 + 2 * 16 * 64
    assert cr.convrot_gemm_workspace_bytes(37, 80, 256, cr.CONVROT_PATH_TCGEN05) >= \
        2 * 37 * 256 + 2 * 80 * 256


def test_workspace_layout_query(lib):
    # Tensor-core engines keep an fp16 image of the codes, the small-M engine int8.
    qo, fmt, so = cr.convrot_linear_workspace_layout(1024, 2048, 2048)
    ws = cr.convrot_linear_workspace_bytes(1024, 2048, 2048, 0, True)
    assert fmt == cr.CONVROT_CODES_F16 and qo % 256 == 0 and so % 256 == 0
    assert qo + 2 * 1024 * 2048 <= so and so + 4 * 1024 <= ws
    qo, fmt, so = cr.convrot_linear_workspace_layout(16, 2048, 2048)
    assert fmt == cr.CONVROT_CODES_I8 and qo + 16 * 2048 <= so
    with pytest.raises(RuntimeError):
        cr.convrot_linear_workspace_layout(16, 2048, 300)


def _p(v):
    return ctypes.c_void_p(v)


FAKE = 0x10000  # a 16-byte aligned non-null address that is never dereferenced


def test_invalid_arguments_rejected_without_gpu(lib):
    P = FAKE
    ws = 1 << 30
    # K not a multiple of 256, K = 0, K too large
    for K in (0, 100, 257, 65536 + 256):
        assert lib.convrot_linear(_p(P), 4, K, _p(P), _p(P), None, 8, None, None, 0, 0.0,
                                  _p(P), _p(P), ws, None) == cr.CONVROT_ERR_INVALID_ARG
    # null required pointers
    assert lib.convrot_linear(None, 4, 256, _p(P), _p(P), None, 8, None, None, 0, 0.0,
                              _p(P), _p(P), ws, None) == cr.CONVROT_ERR_INVALID_ARG
    # misaligned X
    assert lib.convrot_linear(_p(P + 2), 4, 256, _p(P), _p(P), None, 8, None, None, 0, 0.0,
                              _p(P), _p(P), ws, None) == cr.CONVROT_ERR_INVALID_ARG
    # LoRA rank without pointers, negative rank, rank above the limit
    for R in (4, -1, 4096):
        assert lib.convrot_linear(_p(P), 4, 256, _p(P), _p(P), None, 8, None, None, R, 0.5,
                                  _p(P), _p(P), ws, None) == cr.CONVROT_ERR_INVALID_ARG
    # negative sizes
    assert lib.convrot_linear(_p(P), -1, 256, _p(P), _p(P), None, 8, None, None, 0, 0.0,
                              _p(P), _p(P), ws, None) == cr.CONVROT_ERR_INVALID_ARG
    # M or N beyond CONVROT_MAX_DIM (the kernels take them as int; element
    # counts such as M*N may still pass 2^31)
    big = cr.CONVROT_MAX_DIM + 1
    assert lib.convrot_linear(_p(P), big, 256, _p(P), _p(P), None, 8, None, None, 0, 0.0,
                              _p(P), _p(P), ws, None) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_linear(_p(P), 4, 256, _p(P), _p(P), None, big, None, None, 0, 0.0,
                              _p(P), _p(P), ws, None) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_prepare_weight(_p(P), big, 256, _p(P), _p(P), None, None) == \
        cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_rotate_quantize(_p(P), big, 256, _p(P), _p(P), None) == \
        cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_gemm_i32(_p(P), _p(P), 8, big, 256, _p(P), 0, _p(P), ws, None) == \
        cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_linear_noalloc(_p(P), 1, 256, _p(P), _p(P), big, _p(P), None) == \
        cr.CONVROT_ERR_INVALID_ARG
    assert cr.convrot_linear_workspace_bytes(big, 64, 256, 0, True) == 0
    assert cr.convrot_gemm_workspace_bytes(64, big, 256, 0) == 0
    # workspace missing, too small, misaligned
    assert lib.convrot_linear(_p(P), 4, 256, _p(P), _p(P), None, 8, None, None, 0, 0.0,
                              _p(P), None, ws, None) == cr.CONVROT_ERR_WORKSPACE
    assert lib.convrot_linear(_p(P), 4, 256, _p(P), _p(P), None, 8, None, None, 0, 0.0,
                              _p(P), _p(P), 16, None) == cr.CONVROT_ERR_WORKSPACE
    assert lib.convrot_linear(_p(P), 4, 256, _p(P), _p(P), None, 8, None, None, 0, 0.0,
                              _p(P), _p(P + 16), ws, None) == cr.CONVROT_ERR_WORKSPACE
    # prepare_weight / rotate_quantize / gemm entry checks
    assert lib.convrot_prepare_weight(_p(P), 8, 200, _p(P), _p(P), None, None) == \
        cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_prepare_weight(None, 8, 256, _p(P), _p(P), None, None) == \
        cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_rotate_quantize(_p(P), 8, 255, _p(P), _p(P), None) == \
        cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_gemm_i32(_p(P), _p(P), 8, 8, 256, None, 0, _p(P), ws, None) == \
        cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_gemm_i32(_p(P), _p(P), 8, 8, 256, _p(P), 7, _p(P), ws, None) == \
        cr.CONVROT_ERR_INVALID_ARG
    # skinny engine only for M <= 64
    assert lib.convrot_gemm_i32(_p(P), _p(P), 65, 8, 256, _p(P), cr.CONVROT_PATH_SKINNY,
                                _p(P), ws, None) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_set_tile_override(32, 0) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_set_fused(2) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_set_split_mode(4) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_set_split_mode(-1) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_set_split_mode(0) == cr.CONVROT_OK
    assert lib.convrot_set_pair_mma(3) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_set_pair_mma(-1) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_set_pair_mma(0) == cr.CONVROT_OK
    assert lib.convrot_set_small_m_engine(5) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_set_small_m_engine(-1) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_set_small_m_engine(0) == cr.CONVROT_OK
    assert lib.convrot_set_small_m_weights_early(2) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_set_small_m_weights_early(0) == cr.CONVROT_OK
    assert lib.convrot_set_skinny_engine(3) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_set_skinny_engine(0) == cr.CONVROT_OK
    for budget in (0, -5, 2_000_000_001):
        assert lib.convrot_selftest_wait_timeout(budget, None) == cr.CONVROT_ERR_INVALID_ARG
    assert lib.convrot_set_fused(0) == cr.CONVROT_OK
    assert lib.convrot_set_tile_override(128, 17) == cr.CONVROT_ERR_INVALID_ARG
    # convrot_linear_ex: dtypes other than fp16 / bf16, a misaligned bias
    def ex(x_dtype=0, y_dtype=0, bias=None):
        return lib.convrot_linear_ex(_p(P), x_dtype, 8, 256, _p(P), _p(P), None, 8, bias, None,
                                     None, 0, 0.0, _p(P), y_dtype, ws, 1 << 20, None)
    assert ex(x_dtype=2) == cr.CONVROT_ERR_INVALID_ARG
    assert ex(y_dtype=-1) == cr.CONVROT_ERR_INVALID_ARG
    assert ex(bias=_p(P + 2)) == cr.CONVROT_ERR_INVALID_ARG


def test_empty_shapes_are_noops_without_gpu(lib):
    P = FAKE
    # M = 0 or N = 0: OK with nothing launched (no CUDA call is made).
    assert lib.convrot_linear(_p(P), 0, 256, _p(P), _p(P), None, 8, None, None, 0, 0.0,
                              _p(P), None, 0, None) == cr.CONVROT_OK
    assert lib.convrot_linear(_p(P), 4, 256, _p(P), _p(P), None, 0, None, None, 0, 0.0,
                              _p(P), None, 0, None) == cr.CONVROT_OK
    assert lib.convrot_prepare_weight(_p(P), 0, 256, _p(P), _p(P), None, None) == cr.CONVROT_OK
    assert lib.convrot_rotate_quantize(_p(P), 0, 256, _p(P), _p(P), None) == cr.CONVROT_OK


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "w8a8_hadamard_rotated_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "convrot_oracle" not in src, f
