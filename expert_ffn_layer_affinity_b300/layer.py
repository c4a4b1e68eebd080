"""A DeepSeekMoE layer driven through the C ABI: buffers are torch device
tensors, every step is one library call, nothing is computed in Python.

Step order of one pass (the bias changes only between passes; qwbw.cn essay
on the report, "训练的每一步结束之后统计整批样本各个专家的负载情况"):
  moe_router_topk -> [moe_replica_remap] -> moe_permute -> moe_grouped_swiglu
  (routed) -> moe_grouped_swiglu (shared) -> moe_combine ; then moe_bias_update.

Serving layouts from the report's deployment (qwbw.cn essay, "9个专家",
"32个冗余专家"):
  shared_as_routed  the shared experts travel as routed experts E.. with gate 1,
                    computed inside the routed grouped GEMM (no separate launch);
  n_redundant       extra physical copies of the most loaded experts, planned by
                    plan_replicas() from observed loads; tokens of a copied expert
                    are spread over its copies.
Physical expert weights are then laid out [E experts][copies][shared].

tiled_weights (default: on whenever it applies, i.e. a bf16 forward layer in
the standard layout with d % 128 == 0 and I % 64 == 0) keeps box-contiguous
copies of the routed and shared expert weights (moe_tile_expert_weights) and
runs the expert GEMMs on them (moe_grouped_swiglu_tiled): the same arithmetic
in the same order, so bit-identical outputs, with every staged weight box one
run of consecutive memory and the SwiGLU finished inside each epilogue warp.

precision="fp8" runs the expert GEMMs in E4M3 with fine-grained scaling
(qwbw.cn essay on the report, the FP8 training passage; weigao.cc section
"6. FP8 Training"): weights are quantized once per 128 x 128 block when the
layer is built (and again when replicas are re-placed), activations per
1 x 128 tile inside every pass:
  moe_router_topk -> moe_permute (maps only) -> moe_quantize_fp8 (x) ->
  moe_permute_fp8 -> moe_grouped_swiglu_fp8 (routed, shared) -> moe_combine.
Routing, gates and the combine are those of the bf16 path.
"""
from __future__ import annotations

import torch

from . import _lib as L
from .synth import LayerConfig


def _round4(v: int) -> int:
    return (v + 3) // 4 * 4


class MoELayer:
    def __init__(self, cfg: LayerConfig, params: dict, max_T: int | None = None,
                 device: str = "cuda", keep_affinity: bool = False,
                 shared_stream: bool = False, shared_as_routed: bool = False,
                 n_redundant: int = 0, precision: str = "bf16", training: bool = False,
                 tiled_weights: bool | None = None):
        if precision not in ("bf16", "fp8"):
            raise ValueError(f"precision must be 'bf16' or 'fp8', not {precision!r}")
        if training and (precision != "bf16" or shared_as_routed or n_redundant):
            raise NotImplementedError("training: bf16 precision and the standard layout only")
        # training keeps what the backward pass reads: the affinities and the
        # experts' pre-activations a = v.W1^T, c = v.W3^T
        self.training = training
        keep_affinity = keep_affinity or training
        self.cfg = cfg
        self.fp8 = precision == "fp8"
        self.device = torch.device(device)
        dev = self.device
        p = params
        E, d, I, ns = cfg.E, cfg.d, cfg.I, cfg.n_shared
        self.w_r = p["w_r"].to(dev).contiguous()
        self.bias = p["bias"].to(dev).clone().contiguous()
        self.ws1 = p["ws1"].to(dev).contiguous()
        self.ws3 = p["ws3"].to(dev).contiguous()
        self.ws2 = p["ws2"].to(dev).contiguous()
        lo = p.get("logit_offset")
        self.logit_offset = lo.to(dev).contiguous() if lo is not None else None
        self.shared_as_routed = shared_as_routed
        self.n_redundant = n_redundant
        self.ns_routed = ns if shared_as_routed else 0
        self.E_phys = E + n_redundant + self.ns_routed
        # w1 and w3 live in one allocation [2, E, I, d] so the grouped GEMM
        # fetches matching rows of both with a single copy
        w13 = p.get("w13")
        if (self.E_phys == E and w13 is not None and w13.device == dev
                and w13.is_contiguous()):
            self.w13 = w13
            self.w1, self.w3 = w13[0], w13[1]
            self.w2 = p["w2"].to(dev).contiguous()
        elif self.E_phys == E:
            self.w13 = torch.empty(2, E, I, d, dtype=torch.bfloat16, device=dev)
            self.w1, self.w3 = self.w13[0], self.w13[1]
            self.w1.copy_(p["w1"])
            self.w3.copy_(p["w3"])
            self.w2 = p["w2"].to(dev).contiguous()
        else:
            bf = torch.bfloat16
            self.w13 = torch.empty(2, self.E_phys, I, d, dtype=bf, device=dev)
            self.w1, self.w3 = self.w13[0], self.w13[1]
            self.w2 = torch.empty(self.E_phys, d, I, dtype=bf, device=dev)
            self.w1[:E].copy_(p["w1"])
            self.w3[:E].copy_(p["w3"])
            self.w2[:E].copy_(p["w2"])
            for r in range(n_redundant):           # until a plan exists: copies of expert 0
                self.w1[E + r].copy_(self.w1[0])
                self.w3[E + r].copy_(self.w3[0])
                self.w2[E + r].copy_(self.w2[0])
            for j in range(self.ns_routed):
                sl = slice(j * I, (j + 1) * I)
                self.w1[E + n_redundant + j].copy_(self.ws1[sl])
                self.w3[E + n_redundant + j].copy_(self.ws3[sl])
                self.w2[E + n_redundant + j].copy_(self.ws2[:, sl])
        self.slot_start = self.slots = None
        if n_redundant:                            # identity plan: no copy used yet
            self.slot_start = torch.arange(E + 1, dtype=torch.int32, device=dev)
            self.slots = torch.arange(E + n_redundant, dtype=torch.int32, device=dev)
        self.w_split = torch.empty(E, 3 * d, dtype=torch.bfloat16, device=dev)
        L.moe_router_prepare(self.w_r, E, d, self.w_split)
        # box-contiguous copies of the expert weights for the forward GEMMs
        # (moe_tile_expert_weights): the standard layout, whose boxes are
        # strided rows, stays for the backward pass and the other layouts
        can_tile = (d % 128 == 0 and I % 64 == 0 and not self.fp8 and not shared_as_routed
                    and not n_redundant and not training)
        self.tiled = can_tile if tiled_weights is None else bool(tiled_weights)
        if self.tiled and not can_tile:
            raise ValueError("tiled weights need bf16, the standard layout, d % 128 == 0 and "
                             "I % 64 == 0")
        if self.tiled:
            bf = torch.bfloat16
            self.w13_t = torch.empty(E, I // 64, d // 64, 128, 64, dtype=bf, device=dev)
            self.w2_t = torch.empty(E, d // 128, I // 64, 128, 64, dtype=bf, device=dev)
            L.moe_tile_expert_weights(self.w1, self.w3, self.w2, E, I, d, self.w13_t, self.w2_t)
            nI = ns * I
            self.ws13_t = torch.empty(1, nI // 64, d // 64, 128, 64, dtype=bf, device=dev)
            self.ws2_t = torch.empty(1, d // 128, nI // 64, 128, 64, dtype=bf, device=dev)
            L.moe_tile_expert_weights(self.ws1, self.ws3, self.ws2, 1, nI, d, self.ws13_t,
                                      self.ws2_t)
        if self.fp8:
            self._quantize_weights()
        self.keep_affinity = keep_affinity
        self.side = torch.cuda.Stream(device=dev) if shared_stream else None
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stats = torch.zeros(4, dtype=torch.float32, device=dev)
        self.T_cap = 0
        self._alloc(max_T or cfg.T)

    def _quantize_weights(self):
        """E4M3 copies of the expert weights: w1/w3 row-interleaved per
        expert with 128 x 128 block scales, w2 likewise; the shared block as
        one group."""
        c, dev = self.cfg, self.device
        E, d, I, nI = self.E_phys, c.d, c.I, c.n_shared * c.I
        u8, f32 = torch.uint8, torch.float32
        r4 = _round4
        self.w13_q = torch.empty(E, 2 * I, d, dtype=u8, device=dev)
        self.w13_s = torch.empty(E, I // 128, r4(2 * d // 128), dtype=f32, device=dev)
        self.w2_q = torch.empty(E, d, I, dtype=u8, device=dev)
        self.w2_s = torch.empty(E, d // 128, r4(I // 128), dtype=f32, device=dev)
        L.moe_quantize_weights_fp8(self.w1, self.w3, E, I, d, self.w13_q, self.w13_s)
        L.moe_quantize_weights_fp8(self.w2, None, E, d, I, self.w2_q, self.w2_s)
        self.ws13_q = torch.empty(1, 2 * nI, d, dtype=u8, device=dev)
        self.ws13_s = torch.empty(1, nI // 128, r4(2 * d // 128), dtype=f32, device=dev)
        self.ws2_q = torch.empty(1, d, nI, dtype=u8, device=dev)
        self.ws2_s = torch.empty(1, d // 128, r4(nI // 128), dtype=f32, device=dev)
        L.moe_quantize_weights_fp8(self.ws1, self.ws3, 1, nI, d, self.ws13_q, self.ws13_s)
        L.moe_quantize_weights_fp8(self.ws2, None, 1, d, nI, self.ws2_q, self.ws2_s)

    # ------------------------------------------------------------ buffers
    @property
    def K_slots(self) -> int:
        """Entries per token after selection (K, plus shared experts in the
        serving layout)."""
        return self.cfg.K + self.ns_routed

    def _alloc(self, T: int):
        c, dev = self.cfg, self.device
        K, E, d, I, ns = self.K_slots, c.E, c.d, c.I, c.n_shared
        R = T * K
        bf, i32 = torch.bfloat16, torch.int32
        self.idx = torch.empty(T, K, dtype=i32, device=dev)
        self.phys_idx = torch.empty(T, K, dtype=i32, device=dev) if self.n_redundant else None
        self.gate = torch.empty(T, K, dtype=torch.float32, device=dev)
        self.load = torch.zeros(E, dtype=i32, device=dev)
        self.offsets = torch.zeros(self.E_phys + 1, dtype=i32, device=dev)
        self.row_of = torch.empty(T, K, dtype=i32, device=dev)
        self.tok_of = torch.empty(R, dtype=i32, device=dev)
        self.x_perm = torch.empty(R, d, dtype=bf, device=dev)
        self.h = torch.empty(R, I, dtype=bf, device=dev)
        self.y_perm = torch.empty(R, d, dtype=bf, device=dev)
        if not self.shared_as_routed:
            self.h_sh = torch.empty(T, ns * I, dtype=bf, device=dev)
            self.y_sh = torch.empty(T, d, dtype=bf, device=dev)
        else:
            self.h_sh = self.y_sh = None
        self.out = torch.empty(T, d, dtype=bf, device=dev)
        self.affinity = (torch.empty(T, E, dtype=torch.float32, device=dev)
                         if self.keep_affinity else None)
        if self.training:
            self.pre_a = torch.empty(R, I, dtype=bf, device=dev)
            self.pre_c = torch.empty(R, I, dtype=bf, device=dev)
            self.pre_a_sh = torch.empty(T, ns * I, dtype=bf, device=dev)
            self.pre_c_sh = torch.empty(T, ns * I, dtype=bf, device=dev)
        self.ws_bytes = L.moe_workspace_bytes(T, d, self.E_phys, K, I)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.shared_offsets = torch.tensor([0, T], dtype=i32, device=dev)
        if self.fp8:
            u8, f32 = torch.uint8, torch.float32
            self.x_perm = None
            # rows of activation scales: leading dimensions rounded to 4 floats
            self.ld_xs, self.ld_xsp = _round4(T), _round4(R)
            self.xq = torch.empty(T, d, dtype=u8, device=dev)
            self.xs = torch.empty(d // 128, self.ld_xs, dtype=f32, device=dev)
            self.xq_perm = torch.empty(R, d, dtype=u8, device=dev)
            self.xs_perm = torch.empty(d // 128, self.ld_xsp, dtype=f32, device=dev)
            self.hq = torch.empty(R, I, dtype=u8, device=dev)
            self.hs = torch.empty(I // 128, _round4(R), dtype=f32, device=dev)
            if not self.shared_as_routed:
                self.hq_sh = torch.empty(T, ns * I, dtype=u8, device=dev)
                self.hs_sh = torch.empty(ns * I // 128, _round4(T), dtype=f32, device=dev)
        self.T_cap = T
        self._shared_T = T

    def _ensure(self, T: int):
        if T > self.T_cap:
            self._alloc(T)
        if T != self._shared_T:
            self.shared_offsets.copy_(torch.tensor([0, T], dtype=torch.int32))
            self._shared_T = T

    # ------------------------------------------------------------ replicas
    def plan_replicas(self, load) -> torch.Tensor:
        """Re-place the redundant copies from observed per-expert loads (a host
        plan, then a copy of each planned expert's weights into its slot).
        Returns the logical expert of every slot."""
        E = self.cfg.E
        ss, sl, eo = L.moe_replica_plan(load, E, self.n_redundant)
        for r in range(self.n_redundant):
            e = int(eo[E + r])
            self.w1[E + r].copy_(self.w1[e])
            self.w3[E + r].copy_(self.w3[e])
            self.w2[E + r].copy_(self.w2[e])
            if self.fp8:
                for t in (self.w13_q, self.w13_s, self.w2_q, self.w2_s):
                    t[E + r].copy_(t[e])
        self.slot_start = ss.to(self.device)
        self.slots = sl.to(self.device)
        return eo

    # ------------------------------------------------------------- steps
    def route(self, x: torch.Tensor, stream=None):
        c = self.cfg
        T = x.shape[0]
        self._ensure(T)
        aff = self.affinity[:T] if self.affinity is not None else None
        L.moe_router_topk(x, self.w_split, None, self.logit_offset, self.bias, T, c.d, c.E,
                          c.K, c.n_groups, c.topk_groups, c.route_scale, self.idx,
                          self.gate, self.load, aff, self.status, self.ws, self.ws_bytes,
                          stream, n_shared_routed=self.ns_routed)

    def forward(self, x: torch.Tensor, stream=None, marks: dict | None = None,
                out: torch.Tensor | None = None) -> torch.Tensor:
        """One layer pass over x bf16 [T, d]; returns the bf16 [T, d] output:
        `out` when given, else a view of an internal buffer valid until the
        next call.

        `marks`, if given, maps call names ("route", "permute", "routed",
        "shared", "combine") to a pair of CUDA events recorded around that
        call on the stream it runs on."""
        c = self.cfg
        T = x.shape[0]
        K = self.K_slots
        R = T * K
        self._fwd_T = T                               # what a backward call differentiates
        main = torch.cuda.current_stream() if stream is None else stream

        def mark(name, i, s=main):
            if marks is not None and name in marks:
                marks[name][i].record(s)

        mark("route", 0)
        self.route(x, stream)
        idx = self.idx
        if self.n_redundant:
            L.moe_replica_remap(self.idx, T, K, c.E, self.n_redundant, self.slot_start,
                                self.slots, self.phys_idx, stream)
            idx = self.phys_idx
        mark("route", 1)
        if self.fp8:
            return self._forward_fp8(x, idx, stream, mark, out)
        mark("permute", 0)
        L.moe_permute(idx, T, K, self.E_phys, x, c.d, self.offsets, self.row_of, self.tok_of,
                      self.x_perm, self.status, self.ws, self.ws_bytes, stream)
        mark("permute", 1)
        separate_shared = not self.shared_as_routed

        def shared(s):
            if self.training:
                L.moe_grouped_swiglu_save(x, self.shared_offsets, 1, T, c.d, c.n_shared * c.I,
                                          self.ws1, self.ws3, self.ws2, self.h_sh, self.y_sh,
                                          self.pre_a_sh, self.pre_c_sh, self.status, s)
            elif self.tiled:
                L.moe_grouped_swiglu_tiled(x, self.shared_offsets, 1, T, c.d, c.n_shared * c.I,
                                           self.ws13_t, self.ws2_t, self.h_sh, self.y_sh,
                                           self.status, s)
            else:
                L.moe_grouped_swiglu(x, self.shared_offsets, 1, T, c.d, c.n_shared * c.I, self.ws1,
                                     self.ws3, self.ws2, self.h_sh, self.y_sh, self.status, s)

        if self.side is not None and separate_shared:
            self.side.wait_stream(main)
            mark("shared", 0, self.side)
            shared(self.side)
            mark("shared", 1, self.side)
        mark("routed", 0)
        if self.training:
            L.moe_grouped_swiglu_save(self.x_perm, self.offsets, self.E_phys, R, c.d, c.I, self.w1,
                                      self.w3, self.w2, self.h, self.y_perm, self.pre_a,
                                      self.pre_c, self.status, stream)
        elif self.tiled:
            L.moe_grouped_swiglu_tiled(self.x_perm, self.offsets, self.E_phys, R, c.d, c.I,
                                       self.w13_t, self.w2_t, self.h, self.y_perm, self.status,
                                       stream)
        else:
            L.moe_grouped_swiglu(self.x_perm, self.offsets, self.E_phys, R, c.d, c.I, self.w1,
                                 self.w3, self.w2, self.h, self.y_perm, self.status, stream)
        mark("routed", 1)
        if self.side is not None and separate_shared:
            main.wait_stream(self.side)
        elif separate_shared:
            mark("shared", 0)
            shared(stream)
            mark("shared", 1)
        dst = self.out[:T] if out is None else out
        mark("combine", 0)
        L.moe_combine(self.y_perm, self.row_of, self.gate, self.y_sh, T, K, c.d, dst, stream)
        mark("combine", 1)
        return dst

    def _forward_fp8(self, x, idx, stream, mark, out):
        c = self.cfg
        T = x.shape[0]
        K = self.K_slots
        R = T * K
        Tc, Rc = self.ld_xs, self.ld_xsp
        main = torch.cuda.current_stream() if stream is None else stream
        mark("permute", 0)
        L.moe_permute(idx, T, K, self.E_phys, None, c.d, self.offsets, self.row_of, self.tok_of,
                      None, self.status, self.ws, self.ws_bytes, stream)
        L.moe_quantize_fp8(x, T, c.d, self.xq, self.xs, Tc, stream)
        L.moe_permute_fp8(self.xq, self.xs, Tc, T, K, c.d, self.row_of, self.xq_perm,
                          self.xs_perm, Rc, stream)
        mark("permute", 1)
        separate_shared = not self.shared_as_routed
        nI = c.n_shared * c.I

        def shared(s):
            L.moe_grouped_swiglu_fp8(self.xq, self.xs, Tc, self.shared_offsets, 1, T, c.d, nI,
                                     self.ws13_q, self.ws13_s, self.ws2_q, self.ws2_s,
                                     self.h_sh, self.hq_sh, self.hs_sh, self.y_sh, self.status, s)

        if self.side is not None and separate_shared:
            self.side.wait_stream(main)
            mark("shared", 0, self.side)
            shared(self.side)
            mark("shared", 1, self.side)
        mark("routed", 0)
        L.moe_grouped_swiglu_fp8(self.xq_perm, self.xs_perm, Rc, self.offsets, self.E_phys, R,
                                 c.d, c.I, self.w13_q, self.w13_s, self.w2_q, self.w2_s, self.h,
                                 self.hq, self.hs, self.y_perm, self.status, stream)
        mark("routed", 1)
        if self.side is not None and separate_shared:
            main.wait_stream(self.side)
        elif separate_shared:
            mark("shared", 0)
            shared(stream)
            mark("shared", 1)
        dst = self.out[:T] if out is None else out
        mark("combine", 0)
        L.moe_combine(self.y_perm, self.row_of, self.gate, self.y_sh, T, K, c.d, dst, stream)
        mark("combine", 1)
        return dst

    def bias_update(self, T: int, stream=None, group=None, stats_out=None):
        """Sign-rule bias update from this pass's loads.  With a process
        group, the loads of all ranks are summed first (each rank routed its
        own T tokens), so every replica applies the same update for the
        global batch of T * world_size tokens."""
        c = self.cfg
        T_total = T
        if group is not None:
            from .dist import allreduce_loads
            T_total = allreduce_loads(self.load, group)
            T_total *= T
        stats = self.stats if stats_out is None else stats_out
        L.moe_bias_update(self.load, self.bias, T_total, c.K, c.E, c.gamma, stats, stream)
        self.updates = getattr(self, "updates", 0) + 1

    # ------------------------------------------------------------ state
    def state_dict(self) -> dict:
        """The layer's mutable state: the per-expert bias, the number of bias
        updates applied, and the replica plan of a serving layout (host
        tensors; synchronises the device)."""
        st = {"bias": self.bias.detach().cpu().clone(), "updates": getattr(self, "updates", 0)}
        if self.n_redundant:
            st["slot_start"] = self.slot_start.cpu().clone()
            st["slots"] = self.slots.cpu().clone()
        return st

    def load_state_dict(self, st: dict) -> None:
        """Restore a state_dict(): the bias bit for bit, then the replica plan
        (re-placing the copies' weights)."""
        if st["bias"].shape != self.bias.shape or st["bias"].dtype != self.bias.dtype:
            raise ValueError("bias of a different shape or type")
        self.bias.copy_(st["bias"])
        self.updates = int(st.get("updates", 0))
        if self.n_redundant:
            if "slot_start" not in st:
                raise ValueError("state without the replica plan of this serving layout")
            ss, sl = st["slot_start"], st["slots"]
            E = self.cfg.E
            owner = torch.repeat_interleave(torch.arange(E, dtype=torch.int32),
                                            (ss[1:] - ss[:-1]).to(torch.int64))
            used = sl[:int(ss[E])]
            # re-place the copies exactly as recorded: copy r serves the expert
            # whose slot range holds physical id E + r (an unused copy stays)
            for r in range(self.n_redundant):
                at = (used == E + r).nonzero()
                if at.numel() == 0:
                    continue
                e = int(owner[int(at[0])])
                self.w1[E + r].copy_(self.w1[e])
                self.w3[E + r].copy_(self.w3[e])
                self.w2[E + r].copy_(self.w2[e])
                if self.fp8:
                    for t in (self.w13_q, self.w13_s, self.w2_q, self.w2_s):
                        t[E + r].copy_(t[e])
            self.slot_start = ss.to(self.device)
            self.slots = sl.to(self.device)

    def save_state(self, path: str) -> None:
        torch.save(self.state_dict(), path)

    def load_state(self, path: str) -> None:
        self.load_state_dict(torch.load(path, map_location="cpu", weights_only=True))

    def step(self, x: torch.Tensor, stream=None, group=None, marks=None,
             stats_out=None, out: torch.Tensor | None = None) -> torch.Tensor:
        y = self.forward(x, stream, marks, out)
        self.bias_update(x.shape[0], stream, group, stats_out)
        return y

    def capture_step(self, x: torch.Tensor, stats_out=None,
                     out: torch.Tensor | None = None) -> "StepGraph":
        """One step (forward on x, then the bias update from its loads)
        captured in a CUDA graph: replay() relaunches all of the step's
        kernels with one host call, on the same x, out and stats_out buffers
        and the layer's own buffers (the bias it reads is the one the previous
        replay or step left).  Steps of small batches are bound by the host's
        per-call launch cost; a replay removes it.  Run one forward pass
        before capturing (first calls set up kernel attributes).  Single
        process only (a process group's load all-reduce is not captured)."""
        g = torch.cuda.CUDAGraph()
        n = getattr(self, "updates", 0)
        with torch.cuda.graph(g):
            self.forward(x, out=out)
            self.bias_update(x.shape[0], stats_out=stats_out)
        self.updates = n                  # capturing ran nothing
        return StepGraph(self, g, self.out[:x.shape[0]] if out is None else out)

    def device_status(self) -> int:
        return int(self.status.item())

    # ------------------------------------------------------------- backward
    def _alloc_backward(self, T: int):
        c = self.cfg
        E, d, I, K, nI = c.E, c.d, c.I, c.K, c.n_shared * c.I
        R = T * K
        dev, bf, f32 = self.device, torch.bfloat16, torch.float32
        self.bwd = dict(
            T=T,
            dy_perm=torch.empty(R, d, dtype=bf, device=dev),
            dgate=torch.empty(T, K, dtype=f32, device=dev),
            a=None if self.training else torch.empty(R, I, dtype=bf, device=dev),
            c=None if self.training else torch.empty(R, I, dtype=bf, device=dev),
            dh=torch.empty(R, I, dtype=bf, device=dev),
            dac=torch.empty(R, 2 * I, dtype=bf, device=dev),
            dx_perm=torch.empty(R, d, dtype=bf, device=dev),
            dw2=torch.empty(E, d, I, dtype=f32, device=dev),
            dw13=torch.empty(E, 2 * I, d, dtype=f32, device=dev),
            a_s=None if self.training else torch.empty(T, nI, dtype=bf, device=dev),
            c_s=None if self.training else torch.empty(T, nI, dtype=bf, device=dev),
            dh_s=torch.empty(T, nI, dtype=bf, device=dev),
            dac_s=torch.empty(T, 2 * nI, dtype=bf, device=dev),
            dx_s=torch.empty(T, d, dtype=bf, device=dev),
            dws2=torch.empty(1, d, nI, dtype=f32, device=dev),
            dws13=torch.empty(1, 2 * nI, d, dtype=f32, device=dev),
            du=torch.empty(T, K, dtype=f32, device=dev),
            du_row=torch.empty(max(R, 1), dtype=f32, device=dev),
            dx_router=torch.empty(T, d, dtype=f32, device=dev),
            dw_r=torch.empty(E, d, dtype=f32, device=dev),
            dx=torch.empty(T, d, dtype=bf, device=dev),
        )

    def backward(self, x: torch.Tensor, dy: torch.Tensor, stream=None,
                 marks: dict | None = None, dx_out: torch.Tensor | None = None) -> dict:
        """Gradients of <dy, layer(x)> for the experts the last forward(x)
        chose (that pass's routing, gates, dispatch order and expert outputs
        are reused; the bias and the selection take no gradient).  Needs a
        layer built with training=True (or keep_affinity=True), bf16
        precision and the standard layout.

        Expert pre-activations a = v.W1^T and c = v.W3^T come from the
        forward pass when the layer was built with training=True (else they
        are recomputed), the data gradients read the weights in their
        forward layout, the weight
        gradients reduce over each expert's tokens on the tensor cores (fp32
        results), and every step is one library call.  Returns views of
        internal buffers valid until the next call: dx bf16 [T, d], dw_r fp32
        [E, d], dw13 fp32 [E, 2I, d] (dW1 rows 0..I-1, dW3 rows I..2I-1 of each
        expert), dw2 fp32 [E, d, I], dws13 fp32 [2 nI, d], dws2 fp32 [d, nI],
        dgate fp32 [T, K], du fp32 [T, K].

        `dx_out`, if given, receives dx (bf16 [T, d]) instead of an internal
        buffer.  `marks`, if given, maps part names ("bwd_combine", "bwd_routed_dgrad",
        "bwd_routed_wgrad", "bwd_shared", "bwd_router", "bwd_dx") to a pair
        of CUDA events recorded around that part."""
        if self.fp8 or self.shared_as_routed or self.n_redundant:
            raise NotImplementedError("backward: bf16 precision and the standard layout only")
        if self.affinity is None:
            raise ValueError("backward needs the forward's affinities: build with training=True "
                             "(or keep_affinity=True to recompute the expert pre-activations)")
        c = self.cfg
        E, d, I, K, nI = c.E, c.d, c.I, c.K, c.n_shared * c.I
        T = x.shape[0]
        R = T * K
        if getattr(self, "_fwd_T", None) != T:
            raise ValueError("backward(x, dy) must follow forward(x) on the same tokens")
        if dy.shape != x.shape or dy.dtype != torch.bfloat16 or not dy.is_contiguous():
            raise ValueError("dy must be a contiguous bf16 tensor shaped like x")
        if getattr(self, "bwd", None) is None or self.bwd["T"] < T:
            self._alloc_backward(T)
        b = self.bwd
        st, s = self.status, stream
        main = torch.cuda.current_stream() if stream is None else stream

        def mark(name, i):
            if marks is not None and name in marks:
                marks[name][i].record(main)

        mark("bwd_combine", 0)
        # combine backward: dY_perm = g dy, dgate = <dy, y_perm>
        L.moe_combine_backward(dy, self.y_perm, self.row_of, self.gate, T, K, d, b["dy_perm"],
                               b["dgate"], s)
        mark("bwd_combine", 1)
        mark("bwd_routed_dgrad", 0)
        # routed experts: recompute a and c, dh = dY W2, SwiGLU backward,
        # dv = [da | dc] [W1 ; W3]
        if self.training:
            pa, pc = self.pre_a, self.pre_c
        else:
            pa, pc = b["a"], b["c"]
            L.moe_grouped_gemm(self.x_perm, self.offsets, E, R, d, I, self.w1, pa, st, s)
            L.moe_grouped_gemm(self.x_perm, self.offsets, E, R, d, I, self.w3, pc, st, s)
        L.moe_grouped_gemm_kn(b["dy_perm"], self.offsets, E, R, d, I, self.w2, None, b["dh"], st, s)
        L.moe_swiglu_backward(b["dh"], pa, pc, R, I, b["dac"], None, s)
        L.moe_grouped_gemm_kn(b["dac"], self.offsets, E, R, 2 * I, d, self.w1, self.w3,
                              b["dx_perm"], st, s)
        mark("bwd_routed_dgrad", 1)
        mark("bwd_routed_wgrad", 0)
        # weight gradients: dW2 = dY^T h, [dW1 ; dW3] = [da | dc]^T v per expert,
        # straight from the dispatch-order buffers
        L.moe_grouped_gemm_wgrad(b["dy_perm"], self.h, self.offsets, E, R, d, I, b["dw2"], st, s)
        L.moe_grouped_gemm_wgrad(b["dac"], self.x_perm, self.offsets, E, R, 2 * I, d, b["dw13"],
                                 st, s)
        mark("bwd_routed_wgrad", 1)
        mark("bwd_shared", 0)
        # shared experts: one group of all T tokens with gate 1
        so = self.shared_offsets
        if self.training:
            pa, pc = self.pre_a_sh, self.pre_c_sh
        else:
            pa, pc = b["a_s"], b["c_s"]
            L.moe_grouped_gemm(x, so, 1, T, d, nI, self.ws1, pa, st, s)
            L.moe_grouped_gemm(x, so, 1, T, d, nI, self.ws3, pc, st, s)
        L.moe_grouped_gemm_kn(dy, so, 1, T, d, nI, self.ws2, None, b["dh_s"], st, s)
        L.moe_swiglu_backward(b["dh_s"], pa, pc, T, nI, b["dac_s"], None, s)
        L.moe_grouped_gemm_kn(b["dac_s"], so, 1, T, 2 * nI, d, self.ws1, self.ws3, b["dx_s"], st, s)
        L.moe_grouped_gemm_wgrad(dy, self.h_sh, so, 1, T, d, nI, b["dws2"], st, s)
        L.moe_grouped_gemm_wgrad(b["dac_s"], x, so, 1, T, 2 * nI, d, b["dws13"], st, s)
        mark("bwd_shared", 1)
        mark("bwd_router", 0)
        # router: gates -> raw affinities -> logits -> w_r and x
        L.moe_router_backward(b["dgate"], self.idx, K, self.affinity, self.w_r, x, self.row_of,
                              self.tok_of, self.offsets, T, d, E, K, c.route_scale, b["du"],
                              b["du_row"], b["dx_router"], b["dw_r"], s)
        mark("bwd_router", 1)
        mark("bwd_dx", 0)
        dx = b["dx"][:T] if dx_out is None else dx_out
        L.moe_combine_dx(b["dx_perm"], self.row_of, K, b["dx_s"], b["dx_router"], T, d, dx, s)
        mark("bwd_dx", 1)
        return dict(dx=dx, dw_r=b["dw_r"], dw13=b["dw13"], dw2=b["dw2"],
                    dws13=b["dws13"][0], dws2=b["dws2"][0], dgate=b["dgate"][:T], du=b["du"][:T])


class StepGraph:
    """A layer step captured by MoELayer.capture_step."""

    def __init__(self, layer: "MoELayer", graph: torch.cuda.CUDAGraph, out: torch.Tensor):
        self.layer, self.graph, self.out = layer, graph, out

    def replay(self) -> torch.Tensor:
        """Runs the captured step on the current stream's device work queue;
        returns the output buffer it writes."""
        self.graph.replay()
        self.layer.updates = getattr(self.layer, "updates", 0) + 1
        return self.out


class HostPipeline:
    """Layer steps on activations that live in (pinned) host memory, with the
    copies overlapped: while step i computes, step i+1's input is copied in
    on one stream and step i-1's output is copied out on another (PCIe runs
    both directions at once).  Every step still moves its whole input to the
    device and its whole output back; device buffers are double-buffered and
    ordered with events.  Usage: pipe.step(i, x_host, out_host) for i = 0, 1,
    ...; pipe.finish() orders the caller's stream after the last copy out.

    With train=True (a layer built with training=True) a step also copies in
    the output gradient dy_host, runs forward, backward and the bias update,
    and copies out dx into out_host; the weight gradients stay on the device
    (returned by layer.backward into the layer's buffers)."""

    def __init__(self, layer: MoELayer, T: int, train: bool = False):
        self.layer = layer
        self.train = train
        dev = layer.device
        d = layer.cfg.d
        self.h2d = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)
        self.x_dev = [torch.empty(T, d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.out_dev = [torch.empty(T, d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.dy_dev = ([torch.empty(T, d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
                       if train else None)
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_done = [torch.cuda.Event() for _ in range(2)]
        self.ev_out = [torch.cuda.Event() for _ in range(2)]

    def step(self, i: int, x_host: torch.Tensor, out_host: torch.Tensor, group=None,
             stats_out=None, dy_host: torch.Tensor | None = None) -> None:
        b = i % 2
        comp = torch.cuda.current_stream()
        self.h2d.wait_event(self.ev_done[b])         # step i-2 no longer reads x_dev[b]
        with torch.cuda.stream(self.h2d):
            self.x_dev[b].copy_(x_host, non_blocking=True)
            if self.train:
                self.dy_dev[b].copy_(dy_host, non_blocking=True)
        self.ev_in[b].record(self.h2d)
        comp.wait_event(self.ev_in[b])
        comp.wait_event(self.ev_out[b])              # step i-2's output has left out_dev[b]
        if self.train:
            self.layer.forward(self.x_dev[b])
            self.layer.backward(self.x_dev[b], self.dy_dev[b], dx_out=self.out_dev[b])
            self.layer.bias_update(self.x_dev[b].shape[0], group=group, stats_out=stats_out)
        else:
            self.layer.step(self.x_dev[b], group=group, stats_out=stats_out, out=self.out_dev[b])
        self.ev_done[b].record(comp)
        self.d2h.wait_event(self.ev_done[b])
        with torch.cuda.stream(self.d2h):
            out_host.copy_(self.out_dev[b], non_blocking=True)
        self.ev_out[b].record(self.d2h)

    def finish(self) -> None:
        torch.cuda.current_stream().wait_stream(self.d2h)
