"""FP8 (E4M3) path against the oracle: quantization bit for bit, the FP8
row gather exactly, the grouped FP8 SwiGLU experts within the tolerance of
fp32 promotion plus one bf16 rounding."""
import numpy as np
import pytest
import torch

import expert_ffn_layer_affinity_b300 as moe
from oracle import fp8_ref as F8
from oracle import moe_ref as ref
from _util import bf16_to_np64, sync_status

pytestmark = pytest.mark.gpu
DEV = "cuda"


def e4m3_values(q: torch.Tensor) -> np.ndarray:
    """float64 values of E4M3 bytes (decoded by PyTorch's float8_e4m3fn)."""
    return q.detach().cpu().contiguous().view(torch.float8_e4m3fn).double().numpy()


def same_values(a, b):
    """Equal as numbers, sign of zero included, NaN where NaN."""
    a, b = np.asarray(a), np.asarray(b)
    nan = np.isnan(a) & np.isnan(b)
    return bool(np.array_equal(np.isnan(a), np.isnan(b)) and
                np.array_equal(a[~nan], b[~nan]) and
                np.array_equal(np.signbit(a[~nan]), np.signbit(b[~nan])))


def seeded_rows(rows, cols, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 3)
    x = x.to(torch.bfloat16)
    if rows > 3 and cols >= 256:
        x[1, 128:256] = 0.0                      # an all-zero block: scale 1
        x[2, :128] = -0.0
        x[3, 5] = 3.0e38                         # a block with a huge amax
        x[3, 6:128] = 1e-30                      # ... whose other values flush to zero
    return x


@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 256), (300, 384), (1024, 7168),
                                       (5, 1152), (65, 2048)])   # a run of 8 blocks + 1; two runs
def test_quantize_rows_bit_exact(rows, cols):
    x = seeded_rows(rows, cols, 11 + rows)
    ld = rows + 5
    q = torch.zeros(rows, cols, dtype=torch.uint8, device=DEV)
    s = torch.full((cols // 128, ld), -1.0, device=DEV)
    moe.moe_quantize_fp8(x.to(DEV), rows, cols, q, s, ld)
    torch.cuda.synchronize()
    want_q, want_s = F8.quantize_act_1x128(bf16_to_np64(x))
    assert same_values(e4m3_values(q), want_q)
    got_s = s.cpu().numpy()
    assert np.array_equal(got_s[:, :rows].T.view(np.uint32), want_s.view(np.uint32))
    assert np.all(got_s[:, rows:] == -1.0)          # padding columns untouched


@pytest.mark.parametrize("pair", [False, True])
def test_quantize_weights_bit_exact(pair):
    G, rows, cols = 3, 256, 384
    g = torch.Generator().manual_seed(21 + pair)
    w = (torch.randn(G, rows, cols, generator=g) * 0.05).to(torch.bfloat16)
    w[1, :128, 128:256] *= 1000
    w2 = (torch.randn(G, rows, cols, generator=g) * 0.02).to(torch.bfloat16) if pair else None
    nm = 2 if pair else 1
    pitch = (nm * (cols // 128) + 3) // 4 * 4
    q = torch.zeros(G, nm * rows, cols, dtype=torch.uint8, device=DEV)
    s = torch.full((G, rows // 128, pitch), -1.0, device=DEV)
    moe.moe_quantize_weights_fp8(w.to(DEV), w2.to(DEV) if pair else None, G, rows, cols, q, s)
    torch.cuda.synchronize()
    qv = e4m3_values(q)
    sv = s.cpu().numpy()
    for gi in range(G):
        mats = [w[gi]] + ([w2[gi]] if pair else [])
        for which, m in enumerate(mats):
            wq, ws = F8.quantize_w_128x128(bf16_to_np64(m))
            got = qv[gi, which::nm] if pair else qv[gi]
            assert same_values(got, wq)
            got_s = sv[gi, :, which:nm * (cols // 128):nm]
            assert np.array_equal(got_s.view(np.uint32), ws.view(np.uint32))
    assert np.all(sv[:, :, nm * (cols // 128):] == -1.0)       # row padding untouched


def test_permute_fp8_exact():
    T, K, E, d = 333, 4, 8, 256
    g = torch.Generator().manual_seed(5)
    idx = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)]).to(torch.int32)
    _, row_of, _ = ref.permute(idx.numpy(), E)
    q = torch.randint(0, 256, (T, d), generator=g, dtype=torch.uint8)
    ld_in = T + 3
    s = torch.rand(d // 128, ld_in, generator=g)
    R = T * K
    ld_out = R + 7
    qp = torch.zeros(R, d, dtype=torch.uint8, device=DEV)
    sp = torch.full((d // 128, ld_out), -1.0, device=DEV)
    moe.moe_permute_fp8(q.to(DEV), s.to(DEV), ld_in, T, K, d, torch.from_numpy(row_of).to(DEV),
                        qp, sp, ld_out)
    torch.cuda.synchronize()
    want_q = np.zeros((R, d), dtype=np.uint8)
    want_s = np.full((d // 128, ld_out), -1.0, dtype=np.float32)
    for t in range(T):
        for k in range(K):
            want_q[row_of[t, k]] = q[t].numpy()
            want_s[:, row_of[t, k]] = s[:, t].numpy()
    assert np.array_equal(qp.cpu().numpy(), want_q)
    assert np.array_equal(sp.cpu().numpy(), want_s)


def run_fp8_experts(a, offsets, w1, w3, w2):
    """Quantize with the library and run the FP8 grouped experts."""
    R, d = a.shape
    G, I, _ = w1.shape
    r4 = lambda v: (v + 3) // 4 * 4  # noqa: E731
    ld_as = r4(R + 1)
    aq = torch.zeros(R, d, dtype=torch.uint8, device=DEV)
    as_ = torch.zeros(d // 128, ld_as, device=DEV)
    w13q = torch.zeros(G, 2 * I, d, dtype=torch.uint8, device=DEV)
    w13s = torch.zeros(G, I // 128, r4(2 * d // 128), device=DEV)
    w2q = torch.zeros(G, d, I, dtype=torch.uint8, device=DEV)
    w2s = torch.zeros(G, d // 128, r4(I // 128), device=DEV)
    h = torch.full((R, I), 7.0, dtype=torch.bfloat16, device=DEV)
    hq = torch.zeros(R, I, dtype=torch.uint8, device=DEV)
    hs = torch.zeros(I // 128, r4(R), device=DEV)
    y = torch.full((R, d), -3.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    moe.moe_quantize_fp8(a.to(DEV), R, d, aq, as_, ld_as)
    moe.moe_quantize_weights_fp8(w1.to(DEV), w3.to(DEV), G, I, d, w13q, w13s)
    moe.moe_quantize_weights_fp8(w2.to(DEV), None, G, d, I, w2q, w2s)
    moe.moe_grouped_swiglu_fp8(aq, as_, ld_as, offsets.to(DEV), G, R, d, I, w13q, w13s, w2q, w2s,
                               h, hq, hs, y, status)
    st = sync_status(status)
    return h.cpu(), y.cpu(), st


def oracle_experts(a, offsets, w1, w3, w2):
    """h (bf16-rounded) and y per reading R12, group by group, in fp64."""
    A = bf16_to_np64(a)
    R, d = A.shape
    G, I, _ = w1.shape
    H = np.zeros((R, I))
    Y = np.zeros((R, d))
    offs = offsets.numpy()
    for g in range(G):
        r0, r1 = offs[g], offs[g + 1]
        if r1 <= r0:
            continue
        qe = F8.quantize_expert(bf16_to_np64(w1[g]), bf16_to_np64(w3[g]), bf16_to_np64(w2[g]))
        (q1, s1), (q3, s3), _ = qe
        qx, sx = F8.quantize_act_1x128(A[r0:r1])
        H[r0:r1] = F8.round_bf16(ref.silu64(F8.fp8_linear64(qx, sx, q1, s1)) *
                                 F8.fp8_linear64(qx, sx, q3, s3))
        Y[r0:r1] = F8.swiglu_ffn64_fp8(A[r0:r1], qe)
    return H, Y


@pytest.mark.parametrize("sizes,d,I", [
    ([128], 256, 128),                        # one full-ish tile
    ([1], 256, 128),                          # one row
    ([0, 300, 37, 0, 256], 256, 128),         # empty groups, a ragged second tile, exact tile
    ([513, 64, 200], 512, 384),               # three h column tiles, two down column tiles
    ([90, 170], 384, 256),                    # d % 256 == 128: half of the last down tile is empty
    ([400, 31], 1024, 256),
    # decode-sized groups (fewer than 64 rows per group on average) take the
    # small-group orientation of the kernel
    ([3, 0, 7, 1, 30, 2], 256, 128),
    ([40] * 8, 512, 256),
    ([1, 63, 0, 0, 128], 384, 128),
])
def test_grouped_swiglu_fp8_vs_oracle(sizes, d, I):
    G = len(sizes)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(sizes)]), dtype=torch.int32)
    R = int(offsets[-1])
    g = torch.Generator().manual_seed(sum(sizes) + d + I)
    a = torch.randn(R, d, generator=g).to(torch.bfloat16)
    w1 = (torch.randn(G, I, d, generator=g) * 0.05).to(torch.bfloat16)
    w3 = (torch.randn(G, I, d, generator=g) * 0.05).to(torch.bfloat16)
    w2 = (torch.randn(G, d, I, generator=g) * 0.05).to(torch.bfloat16)
    h, y, st = run_fp8_experts(a, offsets, w1, w3, w2)
    assert st == 0
    H, Y = oracle_experts(a, offsets, w1, w3, w2)
    hg, yg = bf16_to_np64(h), bf16_to_np64(y)
    # h: fp32 promotion then one bf16 rounding on each side -> at most one bf16
    # step apart (2**-7 relative), nearly always equal
    dh = np.abs(hg - H)
    assert np.all(dh <= 2.0 ** -7 * np.abs(H) + 1e-5 * np.abs(H).max()), dh.max()
    assert np.mean(hg != H) < 0.02
    # y: the same h codes but where h differed by one step; bf16 output rounding
    assert ref.rel_l2(yg, Y) < 3e-3, ref.rel_l2(yg, Y)
    dy = np.abs(yg - Y)
    assert np.all(dy <= 2.0 ** -6 * np.abs(Y) + 2e-2 * np.abs(Y).max()), dy.max()


def test_grouped_swiglu_fp8_shared_form():
    """One group covering all rows (the shared-expert call), two experts side
    by side: equal to the sum of the two experts evaluated on their own."""
    T, d, I1 = 200, 256, 128
    g = torch.Generator().manual_seed(77)
    a = torch.randn(T, d, generator=g).to(torch.bfloat16)
    w1 = (torch.randn(1, 2 * I1, d, generator=g) * 0.05).to(torch.bfloat16)
    w3 = (torch.randn(1, 2 * I1, d, generator=g) * 0.05).to(torch.bfloat16)
    w2 = (torch.randn(1, d, 2 * I1, generator=g) * 0.05).to(torch.bfloat16)
    offsets = torch.tensor([0, T], dtype=torch.int32)
    _, y, st = run_fp8_experts(a, offsets, w1, w3, w2)
    assert st == 0
    qe = F8.quantize_expert(bf16_to_np64(w1[0]), bf16_to_np64(w3[0]), bf16_to_np64(w2[0]))
    want = sum(F8.swiglu_ffn64_fp8(bf16_to_np64(a), part) for part in F8.split_shared(qe, 2))
    assert ref.rel_l2(bf16_to_np64(y), want) < 3e-3


# ------------------------------------------------------------------ layer
from expert_ffn_layer_affinity_b300 import synth  # noqa: E402
from expert_ffn_layer_affinity_b300.layer import MoELayer  # noqa: E402
from _util import check_pass, HostExperts  # noqa: E402


def test_fp8_layer_tiny_all_tokens():
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    x = synth.make_tokens(cfg, 0, "cpu")
    layer = MoELayer(cfg, p, precision="fp8")
    out = layer.forward(x.cuda()).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    r = check_pass(cfg, p, x, layer, out, fp8=True)
    assert r["rel_l2"] < 3e-3
    # the FP8 layer stays near the bf16 reading of the same layer
    x64 = bf16_to_np64(x)
    host = HostExperts(p)
    want16 = ref.moe_output64(x64, r["idx64"], layer.gate[:, :cfg.K].cpu().numpy(), host,
                              host.shared(), cfg.n_shared)
    assert ref.rel_l2(bf16_to_np64(out), want16) < 0.1


@pytest.mark.parametrize("T", [1, 77, 300])
def test_fp8_layer_tiny_odd_token_counts(T):
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    layer = MoELayer(cfg, p, max_T=300, precision="fp8")
    x = synth.make_tokens(cfg, T, "cpu", T=T)
    out = layer.forward(x.cuda()).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    check_pass(cfg, p, x, layer, out, fp8=True)


def test_fp8_layer_mid_sampled_shared_stream():
    cfg = synth.CONFIGS["mid"]
    p = synth.make_params(cfg, "cpu")
    x = synth.make_tokens(cfg, 0, "cpu")
    layer = MoELayer(cfg, p, shared_stream=True, precision="fp8")
    out = layer.forward(x.cuda()).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    sample = np.random.default_rng(1).choice(cfg.T, 256, replace=False)
    r = check_pass(cfg, p, x, layer, out, sample=sample, fp8=True)
    assert r["rel_l2"] < 3e-3


def test_fp8_layer_serving_layouts_match_standard():
    """Shared-as-routed and redundant copies reorder the same FP8 work: the
    outputs equal the standard layout's (copies: bit for bit)."""
    cfg = synth.CONFIGS["tiny"]
    p = synth.make_params(cfg, "cpu")
    x = synth.make_tokens(cfg, 0, "cuda")
    base = MoELayer(cfg, p, precision="fp8").forward(x).clone()
    rep = MoELayer(cfg, p, precision="fp8", n_redundant=4)
    rep.forward(x)
    rep.plan_replicas(rep.load.cpu())
    out_rep = rep.forward(x).clone()
    sar = MoELayer(cfg, p, precision="fp8", shared_as_routed=True).forward(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(base.view(torch.int16), out_rep.view(torch.int16))
    assert ref.rel_l2(bf16_to_np64(sar), bf16_to_np64(base)) < 6e-3
