"""Seeded synthetic inputs for the MoE layer: shapes, distributions and
seeds only.  This module holds none of the layer's arithmetic; the CUDA path
and the CPU reference both take the tensors it makes.

Workloads (sizes from the DeepSeek-V3 report's layer shape: 256 routed
experts, 8 active per token, 1 shared expert, hidden size 7168 -- qwbw.cn essay
on the report, "1个共享专家256个路由专家每个token激活8个路由专家"):

tiny     T=256,  d=256,  E=16,  K=2, 1 shared, I=128,  no group limit
mid      T=4096, d=2048, E=64,  K=6, 2 shared, I=1408, no group limit,
         Zipf(1.2) per-expert logit offset, 50 bias-feedback steps
v3       T=8192, d=7168, E=256, K=8, 1 shared, I=2048, 8 groups / 4 kept,
         route scale 2.5, bias N(0, 0.01)
v3_decode  the v3 layer at T in {64, 256, 1024}
v3_drift   the v3 layer, 100 steps of T=16384 tokens from 4 Gaussian
           clusters whose mixture weights rotate every 25 steps

Layouts (all row-major, the reduction dimension contiguous):
  x      bf16 [T, d]          w_r   fp32 [E, d]       bias fp32 [E]
  w1,w3  bf16 [E, I, d]       w2    bf16 [E, d, I]   (w1, w3 = views of w13 [2, E, I, d])
  ws1,ws3 bf16 [n_s*I, d]     ws2   bf16 [d, n_s*I]   (shared experts side by side)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    d: int
    E: int
    K: int
    n_shared: int
    I: int
    n_groups: int = 1
    topk_groups: int = 1
    route_scale: float = 1.0
    gamma: float = 1e-3
    bias_std: float = 0.0
    weight_std: float = 0.02
    router_std: float = 0.02
    zipf_s: float | None = None
    steps: int = 1
    clusters: int = 0
    rotate_every: int = 0
    seed: int = 0

    @property
    def R(self) -> int:
        return self.T * self.K

    def with_T(self, T: int) -> "LayerConfig":
        return replace(self, T=T)

    def expert_flops(self) -> float:
        """Dense-contraction FLOPs of the routed + shared experts per pass."""
        return 6.0 * self.d * self.I * self.T * (self.K + self.n_shared)

    def router_flops(self) -> float:
        return 2.0 * self.T * self.d * self.E


CONFIGS = {
    "tiny": LayerConfig("tiny", T=256, d=256, E=16, K=2, n_shared=1, I=128),
    "mid": LayerConfig("mid", T=4096, d=2048, E=64, K=6, n_shared=2, I=1408,
                       zipf_s=1.2, steps=50),
    "v3": LayerConfig("v3", T=8192, d=7168, E=256, K=8, n_shared=1, I=2048,
                      n_groups=8, topk_groups=4, route_scale=2.5, bias_std=0.01),
    "v3_decode": LayerConfig("v3_decode", T=1024, d=7168, E=256, K=8, n_shared=1,
                             I=2048, n_groups=8, topk_groups=4, route_scale=2.5,
                             bias_std=0.01),
    "v3_drift": LayerConfig("v3_drift", T=16384, d=7168, E=256, K=8, n_shared=1,
                            I=2048, n_groups=8, topk_groups=4, route_scale=2.5,
                            bias_std=0.01, steps=100, clusters=4, rotate_every=25),
    # V3 expert shape with 16 experts and 256 rows per expert: the profiling
    # case (1.4 GB of weights, larger than L2, small enough for a full capture)
    "v3_e16": LayerConfig("v3_e16", T=512, d=7168, E=16, K=8, n_shared=1, I=2048,
                          n_groups=8, topk_groups=4, route_scale=2.5, bias_std=0.01),
    # V3 token count and hidden size with 16 experts: the memory-bound calls see
    # V3-sized activations (x_perm ~0.94 GB, larger than L2) with ~3.5 GB on the device
    "v3_mem": LayerConfig("v3_mem", T=8192, d=7168, E=16, K=8, n_shared=1, I=2048,
                          n_groups=8, topk_groups=4, route_scale=2.5, bias_std=0.01),
}
DECODE_T = (64, 256, 1024)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device, dtype):
    """N(0, std^2) drawn in fp32, scaled in fp32, rounded once to dtype."""
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def zipf_logit_offset(E: int, s: float) -> torch.Tensor:
    """Per-expert logit skew for the `mid` workload: o[e] = -s*ln(e+1),
    centred to zero mean, so expert 0 is the most favoured (a Zipf(s) prior
    on expert popularity expressed in logit space)."""
    o = torch.tensor([-s * math.log(e + 1) for e in range(E)], dtype=torch.float64)
    return (o - o.mean()).to(torch.float32)


def _expert_seed(seed: int, e: int) -> int:
    return seed * 1000003 + 7919 + e


def make_expert(cfg: LayerConfig, e: int, device="cpu", seed: int | None = None):
    """(w1 [I, d], w3 [I, d], w2 [d, I]) of routed expert e, from its own seed,
    so any single expert can be made without the others."""
    seed = cfg.seed if seed is None else seed
    g = _gen(_expert_seed(seed, e), device)
    bf = torch.bfloat16
    w1 = _normal((cfg.I, cfg.d), cfg.weight_std, g, device, bf)
    w3 = _normal((cfg.I, cfg.d), cfg.weight_std, g, device, bf)
    w2 = _normal((cfg.d, cfg.I), cfg.weight_std, g, device, bf)
    return w1, w3, w2


def make_router(cfg: LayerConfig, device="cpu", seed: int | None = None):
    """(w_r fp32 [E, d], bias fp32 [E], logit offset [E] or None)."""
    seed = cfg.seed if seed is None else seed
    g = _gen(seed, device)
    w_r = _normal((cfg.E, cfg.d), cfg.router_std, g, device, torch.float32)
    if cfg.bias_std > 0:
        bias = _normal((cfg.E,), cfg.bias_std, g, device, torch.float32)
    else:
        bias = torch.zeros(cfg.E, dtype=torch.float32, device=device)
    off = zipf_logit_offset(cfg.E, cfg.zipf_s).to(device) if cfg.zipf_s else None
    return w_r, bias, off


def make_shared(cfg: LayerConfig, device="cpu", seed: int | None = None):
    """Shared experts side by side: ws1, ws3 [n_s*I, d], ws2 [d, n_s*I]."""
    seed = cfg.seed if seed is None else seed
    g = _gen(_expert_seed(seed, -1000), device)
    bf = torch.bfloat16
    n = cfg.n_shared * cfg.I
    return (_normal((n, cfg.d), cfg.weight_std, g, device, bf),
            _normal((n, cfg.d), cfg.weight_std, g, device, bf),
            _normal((cfg.d, n), cfg.weight_std, g, device, bf))


def make_params(cfg: LayerConfig, device="cpu", seed: int | None = None) -> dict:
    """Router and expert weights of one layer (router from `seed`, each
    routed expert and the shared block from seeds of their own)."""
    seed = cfg.seed if seed is None else seed
    p = {}
    p["w_r"], p["bias"], p["logit_offset"] = make_router(cfg, device, seed)
    bf = torch.bfloat16
    E, d, I = cfg.E, cfg.d, cfg.I
    # w1 and w3 side by side in one allocation (the grouped GEMM then fetches
    # matching rows of both with one copy); p["w13"] is that allocation
    w13 = torch.empty(2, E, I, d, dtype=bf, device=device)
    w1, w3 = w13[0], w13[1]
    w2 = torch.empty(E, d, I, dtype=bf, device=device)
    for e in range(E):
        w1[e], w3[e], w2[e] = make_expert(cfg, e, device, seed)
    p["w1"], p["w3"], p["w2"], p["w13"] = w1, w3, w2, w13
    p["ws1"], p["ws3"], p["ws2"] = make_shared(cfg, device, seed)
    return p


def cluster_weights(cfg: LayerConfig, step: int) -> list[float]:
    """Mixture weights of the drifting workload: (0.55, 0.15, 0.15, 0.15)
    rotated by one cluster every `rotate_every` steps."""
    base = [0.55] + [0.45 / (cfg.clusters - 1)] * (cfg.clusters - 1)
    r = (step // cfg.rotate_every) % cfg.clusters if cfg.rotate_every else 0
    return base[-r:] + base[:-r] if r else base


def make_tokens(cfg: LayerConfig, step: int = 0, device="cpu",
                seed: int | None = None, T: int | None = None) -> torch.Tensor:
    """Activations x bf16 [T, d] for one step (seed + 1 + step).

    Plain workloads: N(0, 1).  Clustered workload: 4 centres mu_c ~ N(0, I)
    (drawn from seed + 1000003), x = (mu_c + eps) / sqrt(2), eps ~ N(0, I),
    cluster chosen per token from the rotating mixture weights."""
    seed = cfg.seed if seed is None else seed
    T = cfg.T if T is None else T
    g = _gen(seed + 1 + step, device)
    if not cfg.clusters:
        return _normal((T, cfg.d), 1.0, g, device, torch.bfloat16)
    gc = _gen(seed + 1000003, device)
    mu = torch.randn(cfg.clusters, cfg.d, generator=gc, device=device)
    w = torch.tensor(cluster_weights(cfg, step), device=device)
    which = torch.multinomial(w, T, replacement=True, generator=g)
    eps = torch.randn(T, cfg.d, generator=g, device=device)
    return ((mu[which] + eps) * (1.0 / math.sqrt(2.0))).to(torch.bfloat16)


def make_affinities(T: int, E: int, step: int = 0, seed: int = 0, device="cpu",
                    skew: float = 0.0, quantum: float | None = None) -> torch.Tensor:
    """Synthetic fp32 affinity scores in (0, 1) for feeding the router's
    selection step directly.  `skew` adds a per-expert tilt (expert e gets
    +skew*(1 - 2e/(E-1)) before clamping) so the loads start unbalanced;
    `quantum` snaps scores to a grid to force exact ties."""
    g = _gen(seed * 7919 + 17 + step, device)
    s = torch.rand(T, E, generator=g, device=device, dtype=torch.float32)
    if skew:
        tilt = skew * (1.0 - 2.0 * torch.arange(E, device=device) / max(E - 1, 1))
        s = (s * 0.5 + 0.25 + tilt[None, :].float()).clamp(1e-4, 1 - 1e-4)
    if quantum:
        s = (torch.round(s / quantum) * quantum).clamp(quantum, 1.0)
    return s.contiguous()


def make_ffn_rows(R: int, d: int, seed: int = 0, device="cpu", std: float = 1.0):
    """bf16 [R, d] rows for testing an expert FFN / combine in isolation."""
    return _normal((R, d), std, _gen(seed + 31337, device), device, torch.bfloat16)


def make_groups(n_groups: int, total: int, seed: int = 0, empty_every: int = 0):
    """Ragged group sizes summing to `total` (some groups may be empty)."""
    g = _gen(seed + 4242, "cpu")
    w = torch.rand(n_groups, generator=g) ** 2
    if empty_every:
        w[::empty_every] = 0
    if float(w.sum()) == 0:
        w[0] = 1
    sizes = torch.floor(w / w.sum() * total).to(torch.int64)
    sizes[int(torch.argmax(w))] += total - int(sizes.sum())
    return sizes


def make_output_grad(cfg: LayerConfig, step: int = 0, device="cpu", seed: int | None = None,
                     T: int | None = None) -> torch.Tensor:
    """Upstream gradient dy bf16 [T, d] of a backward pass: N(0, 1), from a
    seed of its own (seed + 2000003 + step)."""
    seed = cfg.seed if seed is None else seed
    T = cfg.T if T is None else T
    g = _gen(seed + 2000003 + step, device)
    return _normal((T, cfg.d), 1.0, g, device, torch.bfloat16)
