"""Pins of the FP8 oracle (CPU): the E4M3 grid against the format's definition
and PyTorch's float8_e4m3fn conversion, quantization by closed forms and the
format's error bound, and the GEMM reference by its block-promotion form."""
import numpy as np
import pytest
import torch

from oracle import fp8_ref as F8

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _torch_e4m3(x32):
    return torch.from_numpy(np.asarray(x32, dtype=np.float32)).to(torch.float8_e4m3fn).double().numpy()


def test_code_values_match_torch_format():
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mine = np.array([F8.e4m3_code_value(c) for c in range(256)])
    both_nan = np.isnan(codes) & np.isnan(mine)
    assert np.array_equal(np.isnan(codes), np.isnan(mine))
    assert np.array_equal(codes[~both_nan], mine[~both_nan])
    # the format's landmarks
    assert F8.e4m3_code_value(0x7E) == 448.0
    assert F8.e4m3_code_value(0x01) == 2.0 ** -9
    assert F8.e4m3_code_value(0x08) == 2.0 ** -6
    assert sum(np.isnan(mine)) == 2


def test_grid_points_are_fixed_points_and_encode_roundtrips():
    vals = np.array([F8.e4m3_code_value(c) for c in range(256)])
    vals = vals[~np.isnan(vals)]
    assert np.array_equal(F8.round_e4m3(vals), vals)
    codes = F8.e4m3_encode(vals)
    back = np.array([F8.e4m3_code_value(int(c)) for c in codes])
    assert np.array_equal(back, vals)


def test_round_e4m3_matches_torch_below_overflow():
    rng = np.random.default_rng(1)
    grid = np.unique(np.abs([F8.e4m3_code_value(c) for c in range(0x7F)]))
    mids = (grid[1:] + grid[:-1]) / 2                       # exact ties
    x = np.concatenate([
        rng.standard_normal(20000) * 50,
        rng.standard_normal(5000) * 2.0 ** -8,              # subnormal range
        mids, -mids, grid, mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20),
        [0.0, -0.0, 463.99, -463.99, 448.0, 2.0 ** -10, 2.0 ** -12],
    ]).astype(np.float32)
    x = x[np.abs(x) < 464]
    got = F8.round_e4m3(x)
    assert np.array_equal(got, _torch_e4m3(x))


def test_round_e4m3_ties_and_saturation_closed_forms():
    # ties go to the even mantissa
    assert F8.round_e4m3(1.0625) == 1.0          # between 1.000 and 1.125
    assert F8.round_e4m3(1.1875) == 1.25         # between 1.125 and 1.250
    assert F8.round_e4m3(2.0 ** -10) == 0.0      # half the smallest subnormal
    assert F8.round_e4m3(3 * 2.0 ** -10) == 2.0 ** -8   # 1.5 -> 2 subnormal steps
    # saturation: everything at or beyond 448 in magnitude becomes +-448
    big = np.array([448.0, 464.0, 470.0, 1e6, 3e38, -500.0, -1e30])
    assert np.array_equal(F8.round_e4m3(big), np.copysign(448.0, big))
    assert np.isnan(F8.round_e4m3(np.nan))


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1e-40]]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(F8.round_bf16(x), want)


def test_quantize_act_closed_forms():
    rows, cols = 3, 384
    X = np.zeros((rows, cols))
    # row 0, block 1: amax planted at 448 * 2**-3 -> scale 2**-3 exactly
    rng = np.random.default_rng(3)
    X[0, 128:256] = rng.uniform(-1, 1, 128) * 56.0
    X[0, 130] = -56.0
    # row 2, block 2: planted amax 448 * 2**5
    X[2, 256:384] = rng.uniform(-1, 1, 128) * 448 * 32
    X[2, 300] = 448 * 32
    q, s = F8.quantize_act_1x128(X)
    assert s.dtype == np.float32 and s.shape == (rows, cols // 128)
    assert s[0, 1] == 2.0 ** -3 and s[2, 2] == 2.0 ** 5
    # all-zero blocks: scale 1, codes 0
    for (r, j) in [(0, 0), (0, 2), (1, 0), (1, 1), (1, 2), (2, 0), (2, 1)]:
        assert s[r, j] == 1.0
        assert not q[r, j * 128:(j + 1) * 128].any()
    # codes of power-of-two-scaled blocks are the E4M3 rounding of x / s
    assert np.array_equal(q[0, 128:256], F8.round_e4m3(X[0, 128:256] / 2.0 ** -3))
    assert q[0, 130] == -448.0 and q[2, 300] == 448.0


def test_quantize_act_invariants_and_error_bound():
    rng = np.random.default_rng(4)
    X = (rng.standard_normal((37, 512)) * np.exp(rng.uniform(-6, 6, (37, 1)))).astype(np.float32)
    X[5, 200] = 0.0
    q, s = F8.quantize_act_1x128(X)
    blocks = X.reshape(37, 4, 128).astype(np.float64)
    qb = q.reshape(37, 4, 128)
    # the largest element of every block maps to +-448 exactly
    assert np.all(np.abs(qb).max(axis=2) == 448.0)
    # scale = fp32(amax / 448)
    amax = np.abs(blocks).max(axis=2).astype(np.float32)
    assert np.array_equal(s, (amax / np.float32(448)).astype(np.float32))
    # dequantization error within E4M3's half-ulp: 2**-4 relative (normal), 2**-10 * s (subnormal)
    err = np.abs(blocks - qb * s[:, :, None])
    scaled = np.abs(blocks) / s[:, :, None]
    bound = np.where(scaled >= 2.0 ** -6, 2.0 ** -4 * np.abs(blocks), 2.0 ** -10 * s[:, :, None])
    assert np.all(err <= bound * (1 + 1e-6) + 1e-300)


def test_quantize_w_block_layout():
    N, K = 384, 256
    rng = np.random.default_rng(5)
    W = rng.uniform(-1, 1, (N, K))
    for i in range(N // 128):
        for j in range(K // 128):
            blk = W[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            blk *= 448.0 * 2.0 ** (i - 2 * j)
            blk[(7 * i + 3) % 128, (5 * j + 1) % 128] = -448.0 * 2.0 ** (i - 2 * j)
    q, s = F8.quantize_w_128x128(W)
    assert s.shape == (3, 2)
    for i in range(3):
        for j in range(2):
            assert s[i, j] == 2.0 ** (i - 2 * j)
    assert np.array_equal(q, F8.round_e4m3(W / np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)))


def test_fp8_linear_forms_agree_and_closed_form():
    rng = np.random.default_rng(6)
    A = rng.standard_normal((19, 384))
    W = rng.standard_normal((256, 384)) * 0.02
    qa, sa = F8.quantize_act_1x128(A)
    qw, sw = F8.quantize_w_128x128(W)
    y1 = F8.fp8_linear64(qa, sa, qw, sw)
    y2 = F8.fp8_linear_promoted64(qa, sa, qw, sw)
    assert np.max(np.abs(y1 - y2)) <= 1e-12 * np.max(np.abs(y1))
    # closed form: unit codes, sa[r, j] = r + 1, sw[:, j] = 2**-j
    rows, K, N = 4, 384, 128
    qa1 = np.ones((rows, K)); qw1 = np.ones((N, K))
    sa1 = np.array([[r + 1.0] * 3 for r in range(rows)], dtype=np.float32)
    sw1 = np.array([[1.0, 0.5, 0.25]], dtype=np.float32)
    y = F8.fp8_linear64(qa1, sa1, qw1, sw1)
    want = np.array([128 * (r + 1) * (1 + 0.5 + 0.25) for r in range(rows)])
    assert np.array_equal(y, np.repeat(want[:, None], N, axis=1))
    # the quantized product is close to the exact one (E4M3 noise only)
    rel = np.linalg.norm(y1 - A @ W.T) / np.linalg.norm(A @ W.T)
    assert 1e-3 < rel < 0.08


def test_swiglu_fp8_reduces_to_grid_exact_gemm1():
    """With inputs already on the E4M3 grid and every block's amax at 448,
    quantization is the identity, so the gate/up products are exact."""
    rng = np.random.default_rng(7)
    grid = np.array([F8.e4m3_code_value(c) for c in range(0x7F)])
    X = rng.choice(grid, (8, 256)) * rng.choice([-1, 1], (8, 256)); X[:, 0] = 448; X[:, 128] = -448
    W = rng.choice(grid, (128, 256)) * rng.choice([-1, 1], (128, 256)); W[0, 0] = 448; W[0, 128] = 448
    qx, sx = F8.quantize_act_1x128(X)
    qw, sw = F8.quantize_w_128x128(W)
    assert np.all(sx == 1.0) and np.all(sw == 1.0)
    assert np.array_equal(qx, X) and np.array_equal(qw, W)
    assert np.array_equal(F8.fp8_linear64(qx, sx, qw, sw), X @ W.T)


def test_swiglu_fp8_close_to_bf16_oracle_and_shared_split():
    from oracle import moe_ref as R
    rng = np.random.default_rng(8)
    d, I = 256, 256
    X = rng.standard_normal((16, d))
    W1, W3 = rng.standard_normal((I, d)) * 0.05, rng.standard_normal((I, d)) * 0.05
    W2 = rng.standard_normal((d, I)) * 0.05
    y8 = F8.swiglu_ffn64_fp8(X, F8.quantize_expert(W1, W3, W2))
    y = R.swiglu_ffn64(X, W1, W3, W2)
    rel = R.rel_l2(y8, y)
    assert 1e-3 < rel < 0.15
    # two shared experts side by side == the sum of the two quantized separately
    W1b, W3b, W2b = rng.standard_normal((I, d)) * 0.05, rng.standard_normal((I, d)) * 0.05, rng.standard_normal((d, I)) * 0.05
    cat = F8.quantize_expert(np.vstack([W1, W1b]), np.vstack([W3, W3b]), np.hstack([W2, W2b]))
    parts = F8.split_shared(cat, 2)
    ysum = F8.swiglu_ffn64_fp8(X, F8.quantize_expert(W1, W3, W2)) + \
        F8.swiglu_ffn64_fp8(X, F8.quantize_expert(W1b, W3b, W2b))
    yparts = F8.swiglu_ffn64_fp8(X, parts[0]) + F8.swiglu_ffn64_fp8(X, parts[1])
    assert np.array_equal(ysum, yparts)
