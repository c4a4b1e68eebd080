"""ctypes binding of libmoe_b300.so: the C ABI of include/moe.h with the same
names.  Argument marshalling only -- every step runs in the library's CUDA
kernels.  Loading fails loudly when the library is missing; there is no
other implementation to fall back to."""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_b300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED_SHAPE = -2
MOE_ERR_CUDA = -3
MOE_ERR_WORKSPACE = -4
MOE_ERR_SCRATCH_LIMIT = -5
MOE_DEV_TIMEOUT = 1
MOE_DEV_NONFINITE = 2
MOE_DEV_BAD_INDEX = 4

_STATUS_NAMES = {
    MOE_ERR_INVALID_ARG: "MOE_ERR_INVALID_ARG",
    MOE_ERR_UNSUPPORTED_SHAPE: "MOE_ERR_UNSUPPORTED_SHAPE",
    MOE_ERR_CUDA: "MOE_ERR_CUDA",
    MOE_ERR_WORKSPACE: "MOE_ERR_WORKSPACE",
    MOE_ERR_SCRATCH_LIMIT: "MOE_ERR_SCRATCH_LIMIT",
}

# name -> (restype, argtypes); every pointer is passed as c_void_p
P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
LL = ctypes.c_longlong
SIGNATURES = {
    "moe_abi_version": (I, []),
    "moe_workspace_bytes": (Z, [I, I, I, I, I]),
    "moe_router_prepare": (I, [P, I, I, P, P]),
    "moe_router_topk": (I, [P, P, P, P, P, I, I, I, I, I, I, F, I, P, P, P, P, P, P, Z, P]),
    "moe_permute": (I, [P, I, I, I, P, I, P, P, P, P, P, P, Z, P]),
    "moe_permute_static": (I, [P, I, I, I, P, I, P, P, P, P, P, P]),
    "moe_grouped_swiglu": (I, [P, P, I, I, I, I, P, P, P, P, P, P, P]),
    "moe_tile_expert_weights": (I, [P, P, P, I, I, I, P, P, P]),
    "moe_grouped_swiglu_tiled": (I, [P, P, I, I, I, I, P, P, P, P, P, P]),
    "moe_combine": (I, [P, P, P, P, I, I, I, P, P]),
    "moe_replica_plan": (I, [P, I, I, P, P, P]),
    "moe_replica_remap": (I, [P, I, I, I, I, P, P, P, P]),
    "moe_bias_update": (I, [P, P, I, I, I, F, P, P]),
    "moe_seq_balance_loss": (I, [P, P, I, P, I, I, I, F, P, P]),
    "moe_quantize_fp8": (I, [P, I, I, P, P, I, P]),
    "moe_quantize_weights_fp8": (I, [P, P, I, I, I, P, P, P]),
    "moe_permute_fp8": (I, [P, P, I, I, I, I, P, P, P, I, P]),
    "moe_grouped_swiglu_fp8": (I, [P, P, I, P, I, I, I, I, P, P, P, P, P, P, P, P, P, P]),
    "moe_grouped_swiglu_save": (I, [P, P, I, I, I, I, P, P, P, P, P, P, P, P, P]),
    "moe_wait_selftest": (I, [LL, P, P]),
    "moe_router_splits": (I, [I, I, I]),
    "moe_combine_backward": (I, [P, P, P, P, I, I, I, P, P, P]),
    "moe_swiglu_backward": (I, [P, P, P, I, I, P, P, P]),
    "moe_grouped_gemm": (I, [P, P, I, I, I, I, P, P, P, P]),
    "moe_grouped_gemm_wgrad": (I, [P, P, P, I, I, I, I, P, P, P]),
    "moe_grouped_gemm_kn": (I, [P, P, I, I, I, I, P, P, P, P, P]),
    "moe_router_backward": (I, [P, P, I, P, P, P, P, P, P, I, I, I, I, F, P, P, P, P, P]),
    "moe_combine_dx": (I, [P, P, I, P, P, I, I, P, P]),
}

_lib = None


class MoEError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {code} ({_STATUS_NAMES.get(code, 'unknown')})")
        self.code = code


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m expert_ffn_layer_affinity_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name, code):
    if code != MOE_OK:
        raise MoEError(name, code)
    return code


# ---------------------------------------------------------------- raw calls
def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_workspace_bytes(T, d, E, K, I) -> int:
    return lib().moe_workspace_bytes(T, d, E, K, I)


def moe_router_prepare(w_r, E, d, w_split, stream=None, check=True):
    r = lib().moe_router_prepare(_ptr(w_r), E, d, _ptr(w_split), _stream(stream))
    return _check("moe_router_prepare", r) if check else r


def moe_router_topk(x, w_split, scores_in, logit_offset, bias, T, d, E, K, n_groups,
                    topk_groups, route_scale, topk_idx, topk_gate, expert_load,
                    affinity_out, status_dev, ws, ws_bytes, stream=None, check=True,
                    n_shared_routed=0):
    r = lib().moe_router_topk(_ptr(x), _ptr(w_split), _ptr(scores_in), _ptr(logit_offset),
                              _ptr(bias), T, d, E, K, n_groups, topk_groups,
                              float(route_scale), n_shared_routed, _ptr(topk_idx), _ptr(topk_gate),
                              _ptr(expert_load), _ptr(affinity_out), _ptr(status_dev),
                              _ptr(ws), ws_bytes, _stream(stream))
    return _check("moe_router_topk", r) if check else r


def moe_permute(topk_idx, T, K, E, x, d, expert_offsets, row_of, tok_of, x_perm,
                status_dev, ws, ws_bytes, stream=None, check=True):
    r = lib().moe_permute(_ptr(topk_idx), T, K, E, _ptr(x), d, _ptr(expert_offsets),
                          _ptr(row_of), _ptr(tok_of), _ptr(x_perm), _ptr(status_dev),
                          _ptr(ws), ws_bytes, _stream(stream))
    return _check("moe_permute", r) if check else r


def moe_permute_static(topk_idx, T, K, E, x, d, expert_offsets, row_of, tok_of, x_perm,
                       status_dev, stream=None, check=True):
    """moe_permute without a workspace, for callers that cannot allocate
    device memory at call time; its scratch is a fixed 256 KiB array inside
    the library, shared by all calls (see include/moe.h)."""
    r = lib().moe_permute_static(_ptr(topk_idx), T, K, E, _ptr(x), d, _ptr(expert_offsets),
                                 _ptr(row_of), _ptr(tok_of), _ptr(x_perm), _ptr(status_dev),
                                 _stream(stream))
    return _check("moe_permute_static", r) if check else r


def moe_tile_expert_weights(w1, w3, w2, n_groups, I, d, w13_tiled, w2_tiled, stream=None,
                            check=True):
    """Box-contiguous copies of the expert weights (see include/moe.h)."""
    r = lib().moe_tile_expert_weights(_ptr(w1), _ptr(w3), _ptr(w2), n_groups, I, d,
                                      _ptr(w13_tiled), _ptr(w2_tiled), _stream(stream))
    return _check("moe_tile_expert_weights", r) if check else r


def moe_grouped_swiglu_tiled(a, group_offsets, n_groups, R, d, I, w13_tiled, w2_tiled, h, y,
                             status_dev, stream=None, check=True):
    r = lib().moe_grouped_swiglu_tiled(_ptr(a), _ptr(group_offsets), n_groups, R, d, I,
                                       _ptr(w13_tiled), _ptr(w2_tiled), _ptr(h), _ptr(y),
                                       _ptr(status_dev), _stream(stream))
    return _check("moe_grouped_swiglu_tiled", r) if check else r


def moe_grouped_swiglu(a, group_offsets, n_groups, R, d, I, w1, w3, w2, h, y, status_dev,
                       stream=None, check=True):
    r = lib().moe_grouped_swiglu(_ptr(a), _ptr(group_offsets), n_groups, R, d, I, _ptr(w1),
                                 _ptr(w3), _ptr(w2), _ptr(h), _ptr(y), _ptr(status_dev),
                                 _stream(stream))
    return _check("moe_grouped_swiglu", r) if check else r


def moe_replica_plan(load, E, n_redundant, check=True):
    """Host call: returns (slot_start [E+1], slots [E+n], expert_of_slot [E+n])
    as int32 CPU tensors for the given per-expert loads."""
    load = torch.as_tensor(load, dtype=torch.int32).contiguous().cpu()
    ss = torch.empty(E + 1, dtype=torch.int32)
    sl = torch.empty(E + n_redundant, dtype=torch.int32)
    eo = torch.empty(E + n_redundant, dtype=torch.int32)
    r = lib().moe_replica_plan(load.data_ptr(), E, n_redundant, ss.data_ptr(), sl.data_ptr(),
                               eo.data_ptr())
    if check:
        _check("moe_replica_plan", r)
        return ss, sl, eo
    return r


def moe_replica_remap(topk_idx, T, K, E, n_redundant, slot_start, slots, phys_idx, stream=None,
                      check=True):
    r = lib().moe_replica_remap(_ptr(topk_idx), T, K, E, n_redundant, _ptr(slot_start),
                                _ptr(slots), _ptr(phys_idx), _stream(stream))
    return _check("moe_replica_remap", r) if check else r


def moe_combine(y_perm, row_of, topk_gate, y_shared, T, K, d, out, stream=None, check=True):
    r = lib().moe_combine(_ptr(y_perm), _ptr(row_of), _ptr(topk_gate), _ptr(y_shared), T, K, d,
                          _ptr(out), _stream(stream))
    return _check("moe_combine", r) if check else r


def moe_seq_balance_loss(scores, topk_idx, ldk, seq_offsets, S, E, K, alpha, loss_out,
                         stream=None, check=True):
    r = lib().moe_seq_balance_loss(_ptr(scores), _ptr(topk_idx), ldk, _ptr(seq_offsets), S, E, K,
                                   float(alpha), _ptr(loss_out), _stream(stream))
    return _check("moe_seq_balance_loss", r) if check else r


def moe_bias_update(expert_load, bias, T, K, E, gamma, stats_out, stream=None, check=True):
    r = lib().moe_bias_update(_ptr(expert_load), _ptr(bias), T, K, E, float(gamma),
                              _ptr(stats_out), _stream(stream))
    return _check("moe_bias_update", r) if check else r


# ------------------------------------------------------------------ FP8 path
def moe_quantize_fp8(x, rows, cols, q_out, s_out, ld_s, stream=None, check=True):
    r = lib().moe_quantize_fp8(_ptr(x), rows, cols, _ptr(q_out), _ptr(s_out), ld_s,
                               _stream(stream))
    return _check("moe_quantize_fp8", r) if check else r


def moe_quantize_weights_fp8(w, w_pair, groups, rows, cols, q_out, s_out, stream=None,
                             check=True):
    r = lib().moe_quantize_weights_fp8(_ptr(w), _ptr(w_pair), groups, rows, cols, _ptr(q_out),
                                       _ptr(s_out), _stream(stream))
    return _check("moe_quantize_weights_fp8", r) if check else r


def moe_permute_fp8(q_in, s_in, ld_in, T, K, d, row_of, q_perm, s_perm, ld_out, stream=None,
                    check=True):
    r = lib().moe_permute_fp8(_ptr(q_in), _ptr(s_in), ld_in, T, K, d, _ptr(row_of), _ptr(q_perm),
                              _ptr(s_perm), ld_out, _stream(stream))
    return _check("moe_permute_fp8", r) if check else r


def moe_grouped_swiglu_fp8(a_q, a_s, ld_as, group_offsets, n_groups, R, d, I, w13_q, w13_s,
                           w2_q, w2_s, h, h_q, h_s, y, status_dev, stream=None, check=True):
    r = lib().moe_grouped_swiglu_fp8(_ptr(a_q), _ptr(a_s), ld_as, _ptr(group_offsets), n_groups,
                                     R, d, I, _ptr(w13_q), _ptr(w13_s), _ptr(w2_q), _ptr(w2_s),
                                     _ptr(h), _ptr(h_q), _ptr(h_s), _ptr(y), _ptr(status_dev),
                                     _stream(stream))
    return _check("moe_grouped_swiglu_fp8", r) if check else r


# ------------------------------------------------------------------ backward
def moe_grouped_swiglu_save(a, group_offsets, n_groups, R, d, I, w1, w3, w2, h, y, pre_a, pre_c,
                            status_dev, stream=None, check=True):
    r = lib().moe_grouped_swiglu_save(_ptr(a), _ptr(group_offsets), n_groups, R, d, I, _ptr(w1),
                                      _ptr(w3), _ptr(w2), _ptr(h), _ptr(y), _ptr(pre_a),
                                      _ptr(pre_c), _ptr(status_dev), _stream(stream))
    return _check("moe_grouped_swiglu_save", r) if check else r



def moe_combine_backward(dy, y_perm, row_of, gate, T, K, d, dy_perm, dgate, stream=None, check=True):
    r = lib().moe_combine_backward(_ptr(dy), _ptr(y_perm), _ptr(row_of), _ptr(gate), T, K, d,
                                   _ptr(dy_perm), _ptr(dgate), _stream(stream))
    return _check("moe_combine_backward", r) if check else r


def moe_swiglu_backward(dh, a, c, R, I, dac, h, stream=None, check=True):
    r = lib().moe_swiglu_backward(_ptr(dh), _ptr(a), _ptr(c), R, I, _ptr(dac), _ptr(h),
                                  _stream(stream))
    return _check("moe_swiglu_backward", r) if check else r


def moe_grouped_gemm(a, group_offsets, n_groups, R, K, N, w, out, status_dev, stream=None,
                     check=True):
    r = lib().moe_grouped_gemm(_ptr(a), _ptr(group_offsets), n_groups, R, K, N, _ptr(w), _ptr(out),
                               _ptr(status_dev), _stream(stream))
    return _check("moe_grouped_gemm", r) if check else r


def moe_grouped_gemm_wgrad(a, b, group_offsets, n_groups, R, M, N, out, status_dev, stream=None,
                           check=True):
    r = lib().moe_grouped_gemm_wgrad(_ptr(a), _ptr(b), _ptr(group_offsets), n_groups, R, M, N,
                                     _ptr(out), _ptr(status_dev), _stream(stream))
    return _check("moe_grouped_gemm_wgrad", r) if check else r


def moe_grouped_gemm_kn(a, group_offsets, n_groups, R, K, N, w0, w1, out, status_dev, stream=None,
                        check=True):
    r = lib().moe_grouped_gemm_kn(_ptr(a), _ptr(group_offsets), n_groups, R, K, N, _ptr(w0),
                                  _ptr(w1), _ptr(out), _ptr(status_dev), _stream(stream))
    return _check("moe_grouped_gemm_kn", r) if check else r


def moe_router_backward(dgate, topk_idx, ldk, affinity, w_r, x, row_of, tok_of, expert_offsets,
                        T, d, E, K, route_scale, du, du_row, dx_router, dw_r, stream=None,
                        check=True):
    r = lib().moe_router_backward(_ptr(dgate), _ptr(topk_idx), ldk, _ptr(affinity), _ptr(w_r),
                                  _ptr(x), _ptr(row_of), _ptr(tok_of), _ptr(expert_offsets), T, d,
                                  E, K, float(route_scale), _ptr(du), _ptr(du_row), _ptr(dx_router),
                                  _ptr(dw_r), _stream(stream))
    return _check("moe_router_backward", r) if check else r


def moe_combine_dx(dx_perm, row_of, K, dx_shared, dx_router, T, d, dx, stream=None, check=True):
    r = lib().moe_combine_dx(_ptr(dx_perm), _ptr(row_of), K, _ptr(dx_shared), _ptr(dx_router), T, d,
                             _ptr(dx), _stream(stream))
    return _check("moe_combine_dx", r) if check else r


def moe_wait_selftest(limit_ns, status_dev, stream=None, check=True):
    r = lib().moe_wait_selftest(int(limit_ns), _ptr(status_dev), _stream(stream))
    return _check("moe_wait_selftest", r) if check else r


def moe_router_splits(T, d, E):
    return int(lib().moe_router_splits(T, d, E))
