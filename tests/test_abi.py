"""The C-ABI library loads without a GPU, exports every function that
include/moe.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import expert_ffn_layer_affinity_b300 as moe
from expert_ffn_layer_affinity_b300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert "moe_router_topk" in names and len(names) >= 8
    L = ctypes.CDLL(_lib.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_version_and_workspace():
    assert moe.moe_abi_version() == 1
    T, d, E, K, I = 8192, 7168, 256, 8, 2048
    ws = moe.moe_workspace_bytes(T, d, E, K, I)
    assert ws >= T * E * 4 + ((T * K + 1023) // 1024) * E * 4
    assert ws % 256 == 0
    assert moe.moe_workspace_bytes(-1, d, E, K, I) == 0


FAKE = 1 << 20  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("T,E,K,G,M,code", [
    (16, 16, 17, 1, 1, moe.MOE_ERR_UNSUPPORTED_SHAPE),   # K > E
    (16, 24, 2, 5, 1, moe.MOE_ERR_UNSUPPORTED_SHAPE),    # E % G
    (16, 64, 2, 4, 5, moe.MOE_ERR_UNSUPPORTED_SHAPE),    # M > G
    (16, 1024, 8, 1, 1, moe.MOE_ERR_UNSUPPORTED_SHAPE),  # E too large
    (16, 64, 33, 1, 1, moe.MOE_ERR_UNSUPPORTED_SHAPE),   # K > 32
    (16, 256, 8, 64, 4, moe.MOE_ERR_UNSUPPORTED_SHAPE),  # group narrower than a lane's slice
    (16, 16, 8, 8, 1, moe.MOE_ERR_UNSUPPORTED_SHAPE),    # K > M * group size
    (-1, 16, 2, 1, 1, moe.MOE_ERR_INVALID_ARG),
])
def test_router_rejects_bad_shapes(T, E, K, G, M, code):
    r = moe.moe_router_topk(None, None, FAKE, None, FAKE, T, 64, E, K, G, M, 1.0, FAKE, FAKE,
                            FAKE, None, None, None, 0, stream=0, check=False)
    assert r == code


def test_router_rejects_null_bias():
    r = moe.moe_router_topk(None, None, FAKE, None, None, 4, 64, 16, 2, 1, 1, 1.0, FAKE, FAKE,
                            FAKE, None, None, None, 0, stream=0, check=False)
    assert r == moe.MOE_ERR_INVALID_ARG


def test_other_calls_reject_bad_arguments():
    assert moe.moe_grouped_swiglu(FAKE, FAKE, 4, 128, 100, 128, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  None, stream=0, check=False) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert moe.moe_grouped_swiglu(FAKE, FAKE, 4, 128, 128, 96, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  None, stream=0, check=False) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert moe.moe_grouped_swiglu(FAKE + 8, FAKE, 4, 128, 128, 128, FAKE, FAKE, FAKE, FAKE,
                                  FAKE, None, stream=0, check=False) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert moe.moe_grouped_swiglu(None, FAKE, 4, 128, 128, 128, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  None, stream=0, check=False) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_combine(FAKE, FAKE, FAKE, None, 4, 2, 12, FAKE, stream=0,
                           check=False) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert moe.moe_combine(None, FAKE, FAKE, None, 4, 2, 16, FAKE, stream=0,
                           check=False) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_bias_update(None, FAKE, 4, 2, 16, 1e-3, None, stream=0,
                               check=False) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_permute(FAKE, 4, 2, 16, FAKE, 12, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 20,
                           stream=0, check=False) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert moe.moe_permute(FAKE, 4, 2, 16, None, 0, FAKE, FAKE, FAKE, None, None, FAKE, 0,
                           stream=0, check=False) == moe.MOE_ERR_WORKSPACE
    assert moe.moe_router_prepare(None, 16, 64, FAKE, stream=0, check=False) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_router_prepare(FAKE, 16, 65, FAKE, stream=0, check=False) == moe.MOE_ERR_UNSUPPORTED_SHAPE


def test_tiled_weight_calls_reject_bad_arguments():
    # d must be a multiple of 128 and I of 64 (whole boxes); pointers 16-byte aligned
    assert moe.moe_tile_expert_weights(FAKE, FAKE, FAKE, 4, 128, 192, FAKE, FAKE, stream=0,
                                       check=False) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert moe.moe_tile_expert_weights(FAKE, FAKE, FAKE, 4, 96, 256, FAKE, FAKE, stream=0,
                                       check=False) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert moe.moe_tile_expert_weights(FAKE, None, FAKE, 4, 128, 256, FAKE, FAKE, stream=0,
                                       check=False) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_tile_expert_weights(None, None, None, 4, 128, 256, None, None, stream=0,
                                       check=False) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_tile_expert_weights(FAKE + 8, FAKE, None, 4, 128, 256, FAKE, None, stream=0,
                                       check=False) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert moe.moe_grouped_swiglu_tiled(FAKE, FAKE, 4, 128, 192, 128, FAKE, FAKE, FAKE, FAKE,
                                        None, stream=0, check=False) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert moe.moe_grouped_swiglu_tiled(None, FAKE, 4, 128, 256, 128, FAKE, FAKE, FAKE, FAKE,
                                        None, stream=0, check=False) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_grouped_swiglu_tiled(FAKE, FAKE, 4, 128, 256, 128, FAKE + 8, FAKE, FAKE, FAKE,
                                        None, stream=0, check=False) == moe.MOE_ERR_UNSUPPORTED_SHAPE


def test_binding_raises_on_error():
    with pytest.raises(moe.MoEError):
        moe.moe_combine(None, FAKE, FAKE, None, 4, 2, 16, FAKE, stream=0)


def test_fp8_calls_reject_bad_arguments():
    E_SHAPE, E_ARG = moe.MOE_ERR_UNSUPPORTED_SHAPE, moe.MOE_ERR_INVALID_ARG
    # quantize: cols not a multiple of 128, ld_s < rows, null input
    assert moe.moe_quantize_fp8(FAKE, 4, 192, FAKE, FAKE, 4, stream=0, check=False) == E_SHAPE
    assert moe.moe_quantize_fp8(FAKE, 4, 256, FAKE, FAKE, 3, stream=0, check=False) == E_ARG
    assert moe.moe_quantize_fp8(None, 4, 256, FAKE, FAKE, 4, stream=0, check=False) == E_ARG
    assert moe.moe_quantize_fp8(FAKE + 8, 4, 256, FAKE, FAKE, 4, stream=0, check=False) == E_SHAPE
    # weights: rows / cols multiples of 128
    assert moe.moe_quantize_weights_fp8(FAKE, None, 2, 192, 256, FAKE, FAKE, stream=0,
                                        check=False) == E_SHAPE
    assert moe.moe_quantize_weights_fp8(FAKE, FAKE + 8, 2, 128, 256, FAKE, FAKE, stream=0,
                                        check=False) == E_SHAPE
    # permute: d multiple of 128, ld_out >= T*K
    assert moe.moe_permute_fp8(FAKE, FAKE, 4, 4, 2, 192, FAKE, FAKE, FAKE, 8, stream=0,
                               check=False) == E_SHAPE
    assert moe.moe_permute_fp8(FAKE, FAKE, 4, 4, 2, 256, FAKE, FAKE, FAKE, 7, stream=0,
                               check=False) == E_ARG
    # grouped experts: d, I multiples of 128; ld_as >= R; groups <= 512
    args = dict(stream=0, check=False)
    assert moe.moe_grouped_swiglu_fp8(FAKE, FAKE, 64, FAKE, 4, 64, 192, 128, FAKE, FAKE, FAKE,
                                      FAKE, FAKE, FAKE, FAKE, FAKE, None, **args) == E_SHAPE
    assert moe.moe_grouped_swiglu_fp8(FAKE, FAKE, 64, FAKE, 4, 64, 256, 64, FAKE, FAKE, FAKE,
                                      FAKE, FAKE, FAKE, FAKE, FAKE, None, **args) == E_SHAPE
    assert moe.moe_grouped_swiglu_fp8(FAKE, FAKE, 63, FAKE, 4, 64, 256, 128, FAKE, FAKE, FAKE,
                                      FAKE, FAKE, FAKE, FAKE, FAKE, None, **args) == E_ARG
    assert moe.moe_grouped_swiglu_fp8(FAKE, FAKE, 64, FAKE, 513, 64, 256, 128, FAKE, FAKE, FAKE,
                                      FAKE, FAKE, FAKE, FAKE, FAKE, None, **args) == E_SHAPE
    assert moe.moe_grouped_swiglu_fp8(FAKE, FAKE, 64, None, 4, 64, 256, 128, FAKE, FAKE, FAKE,
                                      FAKE, FAKE, FAKE, FAKE, FAKE, None, **args) == E_ARG
    # rows of activation scales must be whole 16-byte units (ld_as % 4 == 0)
    assert moe.moe_grouped_swiglu_fp8(FAKE, FAKE, 66, FAKE, 4, 64, 256, 128, FAKE, FAKE, FAKE,
                                      FAKE, FAKE, FAKE, FAKE, FAKE, None, **args) == E_SHAPE


def test_backward_calls_reject_bad_arguments():
    E_SHAPE, E_ARG = moe.MOE_ERR_UNSUPPORTED_SHAPE, moe.MOE_ERR_INVALID_ARG
    args = dict(stream=0, check=False)
    # d % 8, null input
    assert moe.moe_combine_backward(FAKE, FAKE, FAKE, FAKE, 4, 2, 12, FAKE, FAKE, **args) == E_SHAPE
    assert moe.moe_combine_backward(None, FAKE, FAKE, FAKE, 4, 2, 16, FAKE, FAKE, **args) == E_ARG
    # odd I; null output (h may be null)
    assert moe.moe_swiglu_backward(FAKE, FAKE, FAKE, 4, 7, FAKE, None, **args) == E_SHAPE
    assert moe.moe_swiglu_backward(FAKE, FAKE, FAKE, 4, 8, None, None, **args) == E_ARG
    # NT GEMM: K % 64, N % 8, too many groups
    assert moe.moe_grouped_gemm(FAKE, FAKE, 2, 8, 96, 64, FAKE, FAKE, None, **args) == E_SHAPE
    assert moe.moe_grouped_gemm(FAKE, FAKE, 2, 8, 128, 60, FAKE, FAKE, None, **args) == E_SHAPE
    assert moe.moe_grouped_gemm(FAKE, FAKE, 513, 8, 128, 64, FAKE, FAKE, None, **args) == E_SHAPE
    # wgrad: M % 8, N % 8, null operand
    assert moe.moe_grouped_gemm_wgrad(FAKE, FAKE, FAKE, 2, 64, 60, 64, FAKE, None,
                                      **args) == E_SHAPE
    assert moe.moe_grouped_gemm_wgrad(FAKE, FAKE, FAKE, 2, 64, 64, 12, FAKE, None,
                                      **args) == E_SHAPE
    assert moe.moe_grouped_gemm_wgrad(None, FAKE, FAKE, 2, 64, 64, 64, FAKE, None, **args) == E_ARG
    # K-N GEMM: K % 64 per part, N % 8
    assert moe.moe_grouped_gemm_kn(FAKE, FAKE, 2, 8, 96, 64, FAKE, None, FAKE, None, **args) == E_SHAPE
    assert moe.moe_grouped_gemm_kn(FAKE, FAKE, 2, 8, 192, 64, FAKE, FAKE, FAKE, None,
                                   **args) == E_SHAPE
    assert moe.moe_grouped_gemm_kn(FAKE, FAKE, 2, 8, 128, 60, FAKE, None, FAKE, None,
                                   **args) == E_SHAPE
    assert moe.moe_grouped_gemm_kn(None, FAKE, 2, 8, 128, 64, FAKE, None, FAKE, None,
                                   **args) == E_ARG
    # router backward: K > E, ldk < K
    assert moe.moe_router_backward(FAKE, FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 16, 2, 4,
                                   1.0, FAKE, FAKE, None, FAKE, **args) == E_ARG
    assert moe.moe_router_backward(FAKE, FAKE, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 16, 8, 2,
                                   1.0, FAKE, FAKE, None, FAKE, **args) == E_ARG
    # combine_dx: d % 8
    assert moe.moe_combine_dx(FAKE, FAKE, 2, None, None, 4, 12, FAKE, **args) == E_SHAPE


def test_wait_selftest_rejects_bad_limits():
    assert moe.moe_wait_selftest(0, FAKE, stream=0, check=False) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_wait_selftest(2_000_000_000, FAKE, stream=0, check=False) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_wait_selftest(1_000_000, None, stream=0, check=False) == moe.MOE_ERR_INVALID_ARG
