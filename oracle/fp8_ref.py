"""Plain CPU reference (the oracle) for the FP8 (E4M3) expert FFN with
fine-grained scaling.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package's smoke check and
the benchmark's CPU-baseline / reference arm may import this module.  The
product path never imports it and shares no code with it.

What the pages fix:

* All FP8 tensors use the E4M3 format; activations are scaled per 1 x 128
  tile, weights per 128 x 128 block; the tensor core's partial sums are moved
  to FP32 on the CUDA cores every Nc = 128 reduction elements.  Source: qwbw.cn
  essay on the report, the passage on the FP8 training framework ("对于激活采用
  1×128的瓦片分组缩放权重使用128×128块级分组缩放", "每完成Nc128个元素的矩阵乘累加
  之后把中间结果搬运到CUDA Core", "全部张量统一使用E4M3格式").
* Scales are kept per block or tile, and the accumulation precision matters.
  Source: "DeepSeek-V3 Technical Report：中英对照解读" (weigao.cc), section
  "6. FP8 Training", rows "Fine-grained quantization is used" and
  "Accumulation precision still matters".
* Gating stays in high precision (same qwbw.cn passage: "MoE门控…依然保留BF16
  或者FP32高精度"), so the router, the gates and the combine are those of the
  bf16 layer (moe_ref); only the expert GEMM inputs are FP8.

Readings of what the pages leave open (also listed in the design notes):

R9   Scale of a block = fp32(amax / 448), amax = the largest |value| of the
     block in fp32 (NaN ignored); an all-zero block gets scale 1.  Code =
     E4M3 rounding (nearest, ties to even, saturating at +-448) of
     fp32(value / scale); the value it stands for is code * scale.
R10  Promotion: each 128-deep slice of the reduction is summed by the tensor
     core, multiplied by (activation scale * weight scale) and added in fp32,
     slices in ascending order.  The oracle takes the exact sum of the
     dequantized products in fp64; promotion only adds rounding.
R11  Blocks: activation tiles run along the reduction dimension of each row
     (token); weight blocks are 128 output rows x 128 reduction columns of
     w1, w3 and w2 separately.  The shared experts' side-by-side weights have
     blocks that never straddle two experts (I is a multiple of 128).
R12  FP8 FFN: x is quantized once per token (1 x 128 over d); the SwiGLU
     output h = silu(a) * c is rounded to bf16 and then quantized (1 x 128
     over I) as the input of the down projection.

Function-level parity status: every function here is pinned by the CPU test
suite (the E4M3 grid against the format's own definition and PyTorch's
float8_e4m3fn conversion; quantization by closed forms and error bounds; the
GEMM by its block-promotion form and closed forms).
"""
from __future__ import annotations

import numpy as np

from .moe_ref import silu64

F32 = np.float32
F64 = np.float64

E4M3_MAX = 448.0
BLOCK = 128


# ---------------------------------------------------------------------------
# Rounding to a binary floating-point format (round to nearest, ties to even)
# ---------------------------------------------------------------------------
def round_to_format(x, mant_bits: int, emin: int, max_finite: float, saturate: bool):
    """Round every value of x (exactly, from float64) to the nearest number of
    a binary format with `mant_bits` stored mantissa bits and smallest normal
    exponent `emin` (subnormals below it), ties to even.  Results above
    max_finite become max_finite (saturate) or inf.  NaN stays NaN."""
    x = np.asarray(x, dtype=F64)
    ax = np.abs(x)
    _, ex = np.frexp(ax)                       # ax = m * 2**ex, m in [0.5, 1)
    e = np.maximum(ex.astype(np.int64) - 1, emin)
    quantum = np.ldexp(1.0, (e - mant_bits).astype(np.int32))
    with np.errstate(invalid="ignore"):
        q = np.round(ax / quantum) * quantum      # np.round: half to even
    if saturate:
        q = np.minimum(q, max_finite)
    else:
        q = np.where(q > max_finite, np.inf, q)
    q = np.where(np.isnan(ax), np.nan, q)
    return np.copysign(q, x)


def round_e4m3(x):
    """E4M3 (no infinities, max 448) with saturation to the largest finite."""
    return round_to_format(x, 3, -6, E4M3_MAX, saturate=True)


def round_bf16(x):
    """bf16 (8-bit exponent, 7 stored mantissa bits); overflow to inf."""
    return round_to_format(x, 7, -126, float((2.0 - 2.0 ** -7) * 2.0 ** 127), saturate=False)


def e4m3_code_value(code: int) -> float:
    """Value of one E4M3 byte: 1 sign, 4 exponent (bias 7), 3 mantissa bits;
    exponent 0 is subnormal (m * 2**-9); S.1111.111 is NaN."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_encode(v):
    """Byte code of E4M3 values (v must be on the grid; NaN -> 0x7F)."""
    v = np.asarray(v, dtype=F64)
    table = {}
    for c in range(256):
        val = e4m3_code_value(c)
        if not np.isnan(val) and not (val == 0.0 and c == 0x80):
            table[val] = c
    out = np.empty(v.shape, dtype=np.uint8)
    flat = v.reshape(-1)
    o = out.reshape(-1)
    for i, val in enumerate(flat):
        if np.isnan(val):
            o[i] = 0x7F
        elif val == 0.0:
            o[i] = 0x80 if np.signbit(val) else 0x00
        else:
            o[i] = table[float(val)]
    return out


# ---------------------------------------------------------------------------
# Quantization (readings R9, R11)
# ---------------------------------------------------------------------------
def _scale_of(amax32):
    amax32 = np.asarray(amax32, dtype=F32)
    with np.errstate(invalid="ignore", divide="ignore"):
        s = (amax32 / F32(E4M3_MAX)).astype(F32)
    return np.where(amax32 > 0, s, F32(1.0)).astype(F32)


def _quant_codes(x32, s32):
    with np.errstate(invalid="ignore", divide="ignore"):
        return round_e4m3((x32 / s32).astype(F32))


def quantize_act_1x128(X):
    """Per row, per 128 consecutive columns: (codes [rows, cols] as float64
    values on the E4M3 grid, scales fp32 [rows, cols/128])."""
    X = np.asarray(X, dtype=F64).astype(F32)
    rows, cols = X.shape
    assert cols % BLOCK == 0
    b = X.reshape(rows, cols // BLOCK, BLOCK)
    amax = np.fmax.reduce(np.abs(b), axis=2)
    s = _scale_of(amax)
    q = _quant_codes(b, s[:, :, None])
    return q.reshape(rows, cols), s


def quantize_w_128x128(W):
    """Per 128 x 128 block of W [N, K]: (codes [N, K] as float64 values,
    scales fp32 [N/128, K/128])."""
    W = np.asarray(W, dtype=F64).astype(F32)
    N, K = W.shape
    assert N % BLOCK == 0 and K % BLOCK == 0
    b = W.reshape(N // BLOCK, BLOCK, K // BLOCK, BLOCK)
    amax = np.fmax.reduce(np.fmax.reduce(np.abs(b), axis=3), axis=1)
    s = _scale_of(amax)
    q = _quant_codes(b, s[:, None, :, None])
    return q.reshape(N, K), s


def dequant_act(q, s):
    return np.asarray(q, dtype=F64) * np.repeat(np.asarray(s, dtype=F64), BLOCK, axis=1)


def dequant_w(q, s):
    s = np.asarray(s, dtype=F64)
    return np.asarray(q, dtype=F64) * np.repeat(np.repeat(s, BLOCK, axis=0), BLOCK, axis=1)


# ---------------------------------------------------------------------------
# GEMM and FFN (readings R10, R12)
# ---------------------------------------------------------------------------
def fp8_linear64(qa, sa, qw, sw):
    """Y = dequant(A) . dequant(W)^T in float64: the exact value the
    per-128 promoted FP8 GEMM approximates."""
    return dequant_act(qa, sa) @ dequant_w(qw, sw).T


def fp8_linear_promoted64(qa, sa, qw, sw):
    """The same product in the pages' promotion form: per 128-deep slice j,
    the code product qa_j . qw_j^T scaled by sa[:, j] x sw[:, j] and added.
    Used by the pins as an independent check of fp8_linear64."""
    qa = np.asarray(qa, dtype=F64)
    qw = np.asarray(qw, dtype=F64)
    sa = np.asarray(sa, dtype=F64)
    sw = np.asarray(sw, dtype=F64)
    rows, K = qa.shape
    N = qw.shape[0]
    y = np.zeros((rows, N), dtype=F64)
    for j in range(K // BLOCK):
        sl = slice(j * BLOCK, (j + 1) * BLOCK)
        part = qa[:, sl] @ qw[:, sl].T
        y += part * sa[:, j][:, None] * np.repeat(sw[:, j], BLOCK)[None, :]
    return y


def quantize_expert(W1, W3, W2):
    """((q1, s1), (q3, s3), (q2, s2)) of one expert (R11)."""
    return quantize_w_128x128(W1), quantize_w_128x128(W3), quantize_w_128x128(W2)


def swiglu_ffn64_fp8(X, qexp):
    """FFN of reading R12 for every row of X (values exactly representable in
    bf16 or fp32), with the expert's quantized weights qexp."""
    (q1, s1), (q3, s3), (q2, s2) = qexp
    qx, sx = quantize_act_1x128(X)
    a = fp8_linear64(qx, sx, q1, s1)
    c = fp8_linear64(qx, sx, q3, s3)
    h = round_bf16(silu64(a) * c)
    qh, sh = quantize_act_1x128(h)
    return fp8_linear64(qh, sh, q2, s2)


def split_shared(qexp, n_shared):
    """Per-expert slices of the side-by-side shared weights' codes and scales
    (blocks never straddle two experts, R11)."""
    (q1, s1), (q3, s3), (q2, s2) = qexp
    I = q1.shape[0] // n_shared
    nb = I // BLOCK
    out = []
    for j in range(n_shared):
        r = slice(j * I, (j + 1) * I)
        rb = slice(j * nb, (j + 1) * nb)
        out.append(((q1[r], s1[rb]), (q3[r], s3[rb]), (q2[:, r], s2[:, rb])))
    return out


def moe_output64_fp8(x, idx, gate, get_expert_q, shared_q, n_shared, tokens=None):
    """Layer output of reading R6 (moe_ref) with every expert FFN replaced by
    swiglu_ffn64_fp8.  get_expert_q(e) -> quantized expert (quantize_expert);
    shared_q = quantized side-by-side shared block or None."""
    x = np.asarray(x, dtype=F64)
    T = x.shape[0]
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    xs = x[tokens]
    out = np.zeros_like(xs)
    if shared_q is not None:
        for qe in split_shared(shared_q, n_shared):
            out += swiglu_ffn64_fp8(xs, qe)
    sub_idx = np.asarray(idx)[tokens]
    sub_gate = np.asarray(gate, dtype=F64)[tokens]
    for e in np.unique(sub_idx):
        rows, slots = np.nonzero(sub_idx == e)
        y = swiglu_ffn64_fp8(xs[rows], get_expert_q(int(e)))
        out[rows] += sub_gate[rows, slots][:, None] * y
    return out
