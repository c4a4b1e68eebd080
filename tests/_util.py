"""Conversions and comparison helpers shared by the tests (the layer's
arithmetic comes from the oracle only)."""
import numpy as np
import torch

from oracle import fp8_ref as f8ref
from oracle import moe_ref as ref


def bf16_to_np64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a bf16 tensor (widening bf16 to float64 is
    exact; tests/test_util_pins.py checks this against the oracle's
    bit-pattern decoding)."""
    return t.detach().cpu().to(torch.float64).numpy()


def f32_bits(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def sync_status(status: torch.Tensor) -> int:
    torch.cuda.synchronize()
    return int(status.item())


class HostExperts:
    """Oracle-side view of the expert weights: exact fp64 values fetched one
    expert at a time (the full V3 set does not fit comfortably in host RAM as
    fp64)."""

    def __init__(self, p):
        self.p = p

    def __call__(self, e):
        return (bf16_to_np64(self.p["w1"][e]), bf16_to_np64(self.p["w3"][e]),
                bf16_to_np64(self.p["w2"][e]))

    def shared(self):
        return (bf16_to_np64(self.p["ws1"]), bf16_to_np64(self.p["ws3"]),
                bf16_to_np64(self.p["ws2"]))

    def quantized(self, e):
        """The oracle's own E4M3 quantization of routed expert e."""
        return f8ref.quantize_expert(*self(e))

    def shared_quantized(self):
        return f8ref.quantize_expert(*self.shared())


def route_check(cfg, p, x, layer, bias=None):
    """The GPU's expert choice for every token of the pass against the
    oracle's fp64 routing (with the bias the GPU used).  Returns the oracle's
    x64, idx64, gate64, the near-tie masks kth / grp, the mismatch mask and
    `bad`: mismatched tokens that are not near-tie (must be empty)."""
    T = x.shape[0]
    x64 = bf16_to_np64(x)
    off = p["logit_offset"].cpu().numpy() if p["logit_offset"] is not None else None
    b = (bias if bias is not None else p["bias"]).cpu().numpy()
    s64 = ref.router_affinity64(x64, p["w_r"].cpu().numpy(), off)
    idx64, gate64 = ref.select_experts(s64, b.astype(np.float64), cfg.K, cfg.n_groups,
                                       cfg.topk_groups, cfg.route_scale, precision="fp64")
    kth, grp = ref.near_tie_tokens(s64, b, cfg.K, cfg.n_groups, cfg.topk_groups)
    gidx = layer.idx[:T, :cfg.K].cpu().numpy()
    mism = np.any(np.sort(gidx, 1) != np.sort(idx64, 1), axis=1)
    return dict(x64=x64, idx64=idx64, gate64=gate64, kth=kth, grp=grp, mism=mism,
                bad=np.nonzero(mism & ~(kth | grp))[0])


def check_pass(cfg, p, x, layer, out, sample=None, bias=None, fp8=False):
    """Compare one pass: routing on every token, output on `sample` tokens
    (against the FP8 reading of the experts when fp8=True)."""
    T = x.shape[0]
    rc = route_check(cfg, p, x, layer, bias)
    x64, idx64, gate64 = rc["x64"], rc["idx64"], rc["gate64"]
    kth, grp, mism = rc["kth"], rc["grp"], rc["mism"]
    assert len(rc["bad"]) == 0, rc["bad"][:10]
    tokens = np.arange(T) if sample is None else sample
    tokens = tokens[~mism[tokens]]
    host = HostExperts(p)
    if fp8:
        want = f8ref.moe_output64_fp8(x64, idx64, gate64, host.quantized,
                                      host.shared_quantized(), cfg.n_shared, tokens)
    else:
        want = ref.moe_output64(x64, idx64, gate64, host, host.shared(), cfg.n_shared, tokens)
    got = bf16_to_np64(out[torch.from_numpy(tokens).to(out.device)])
    err = ref.rel_l2(got, want)
    assert err < 1e-2, err
    return dict(rel_l2=err, mismatched_tokens=int(mism.sum()), near_tie=int((kth | grp).sum()),
                near_tie_kth=int(kth.sum()), near_tie_grp=int(grp.sum()),
                mismatched_kth=int((mism & kth).sum()), mismatched_grp_only=int((mism & grp & ~kth).sum()),
                checked_tokens=int(len(tokens)), idx64=idx64)


def output_sample(rc, n, seed):
    """Tokens whose layer output is checked: `n` seeded-random tokens of the
    pass plus every near-tie token (K-th gap or group gap below 1e-5 in the
    oracle's fp64 scores), minus the tokens whose experts differ (a counted
    near-tie flip: the GPU then ran other experts for them)."""
    T = len(rc["mism"])
    rnd = np.random.default_rng(seed).choice(T, min(n, T), replace=False)
    tok = np.union1d(rnd, np.nonzero(rc["kth"] | rc["grp"])[0])
    return tok[~rc["mism"][tok]]


def oracle_outputs(requests, host, n_shared):
    """The oracle's layer output (reading R6) for several passes that share
    one set of expert weights, in ONE call of the oracle on the stacked token
    rows (rows are independent, so this equals one call per pass; each
    expert's weights are then fetched once).  requests: list of
    (x64 rows, idx64 rows, gate64 rows).  Returns one array per request."""
    X = np.concatenate([r[0] for r in requests], axis=0)
    IDX = np.concatenate([r[1] for r in requests], axis=0)
    GATE = np.concatenate([r[2] for r in requests], axis=0)
    Y = ref.moe_output64(X, IDX, GATE, host, host.shared(), n_shared)
    out, a = [], 0
    for r in requests:
        out.append(Y[a:a + len(r[0])])
        a += len(r[0])
    return out


def describe(r) -> str:
    return (f"rel_l2={r['rel_l2']:.3e} checked={r['checked_tokens']} "
            f"near_tie kth={r['near_tie_kth']} grp={r['near_tie_grp']} "
            f"mismatched={r['mismatched_tokens']} (kth {r['mismatched_kth']}, "
            f"group-gap only {r['mismatched_grp_only']})")


def sign_rule_holds(load, b_before, b_after, T, K, E, gamma) -> bool:
    """Property of the bias feedback on any (load, bias) pair: each expert's
    bias moved by exactly one fp32 step of gamma in the direction of
    T*K - E*load, or not at all when the two are equal."""
    load = np.asarray(load, dtype=np.int64)
    b0 = np.asarray(b_before, dtype=np.float32)
    b1 = np.asarray(b_after, dtype=np.float32)
    g = np.float32(gamma)
    diff = T * K - E * load
    want = np.where(diff > 0, b0 + g, np.where(diff < 0, b0 - g, b0)).astype(np.float32)
    return bool(np.array_equal(want.view(np.uint32), b1.view(np.uint32)))


class Trajectory:
    """The oracle's own bias-feedback trajectory next to the GPU's: loads from
    the oracle's fp64 routing, updates by the oracle's fp32 rule.  The two are
    compared bit for bit until a near-tie token (counted) makes a load differ;
    after that the trajectories may legitimately part and only the sign-rule
    property of the GPU's own updates is checked."""

    def __init__(self, cfg, bias0):
        self.cfg = cfg
        self.b = np.asarray(bias0, dtype=np.float32).copy()
        self.diverged_at = None
        self.near_tie_mismatches = 0
        self.mismatches_kth = 0
        self.mismatches_grp_only = 0

    def step(self, step, T, s64, gpu_idx, gpu_load, gpu_b_before, gpu_b_after):
        c = self.cfg
        assert sign_rule_holds(gpu_load, gpu_b_before, gpu_b_after, T, c.K, c.E, c.gamma)
        if self.diverged_at is not None:
            return
        idx64, _ = ref.select_experts(s64, self.b.astype(np.float64), c.K, c.n_groups,
                                      c.topk_groups, c.route_scale, precision="fp64")
        kth, grp = ref.near_tie_tokens(s64, self.b, c.K, c.n_groups, c.topk_groups)
        mism = np.any(np.sort(gpu_idx, 1) != np.sort(idx64, 1), axis=1)
        assert not np.any(mism & ~(kth | grp)), np.nonzero(mism & ~(kth | grp))[0][:10]
        self.near_tie_mismatches += int(mism.sum())
        self.mismatches_kth += int((mism & kth).sum())
        self.mismatches_grp_only += int((mism & grp & ~kth).sum())
        load = ref.expert_load(idx64, c.E)
        new_b = ref.bias_update(load, self.b, T, c.K, c.E, c.gamma)
        if np.array_equal(load, np.asarray(gpu_load)):
            assert np.array_equal(new_b.view(np.uint32),
                                  np.asarray(gpu_b_after, dtype=np.float32).view(np.uint32))
        else:
            assert mism.any()
            self.diverged_at = step
        self.b = new_b
