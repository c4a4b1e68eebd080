"""A DeepSeekMoE layer driven through the C ABI: buffers are torch device
tensors, every step is one library call, nothing is computed in Python.

Step order of one pass (the bias changes only between passes; qwbw.cn essay
on the report, "训练的每一步结束之后统计整批样本各个专家的负载情况"):
  moe_router_topk -> moe_permute -> moe_grouped_swiglu (routed)
  -> moe_grouped_swiglu (shared) -> moe_combine ; then moe_bias_update.
"""
from __future__ import annotations

import torch

from . import _lib as L
from .synth import LayerConfig


class MoELayer:
    def __init__(self, cfg: LayerConfig, params: dict, max_T: int | None = None,
                 device: str = "cuda", keep_affinity: bool = False,
                 shared_stream: bool = False):
        self.cfg = cfg
        self.device = torch.device(device)
        dev = self.device
        p = params
        self.w_r = p["w_r"].to(dev).contiguous()
        self.bias = p["bias"].to(dev).clone().contiguous()
        self.w1 = p["w1"].to(dev).contiguous()
        self.w3 = p["w3"].to(dev).contiguous()
        self.w2 = p["w2"].to(dev).contiguous()
        self.ws1 = p["ws1"].to(dev).contiguous()
        self.ws3 = p["ws3"].to(dev).contiguous()
        self.ws2 = p["ws2"].to(dev).contiguous()
        lo = p.get("logit_offset")
        self.logit_offset = lo.to(dev).contiguous() if lo is not None else None
        E, d = cfg.E, cfg.d
        self.w_split = torch.empty(E, 3 * d, dtype=torch.bfloat16, device=dev)
        L.moe_router_prepare(self.w_r, E, d, self.w_split)
        self.keep_affinity = keep_affinity
        self.side = torch.cuda.Stream(device=dev) if shared_stream else None
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stats = torch.zeros(4, dtype=torch.float32, device=dev)
        self.T_cap = 0
        self._alloc(max_T or cfg.T)

    # ------------------------------------------------------------ buffers
    def _alloc(self, T: int):
        c, dev = self.cfg, self.device
        K, E, d, I, ns = c.K, c.E, c.d, c.I, c.n_shared
        R = T * K
        bf, i32 = torch.bfloat16, torch.int32
        self.idx = torch.empty(T, K, dtype=i32, device=dev)
        self.gate = torch.empty(T, K, dtype=torch.float32, device=dev)
        self.load = torch.zeros(E, dtype=i32, device=dev)
        self.offsets = torch.zeros(E + 1, dtype=i32, device=dev)
        self.row_of = torch.empty(T, K, dtype=i32, device=dev)
        self.tok_of = torch.empty(R, dtype=i32, device=dev)
        self.x_perm = torch.empty(R, d, dtype=bf, device=dev)
        self.h = torch.empty(R, I, dtype=bf, device=dev)
        self.y_perm = torch.empty(R, d, dtype=bf, device=dev)
        self.h_sh = torch.empty(T, ns * I, dtype=bf, device=dev)
        self.y_sh = torch.empty(T, d, dtype=bf, device=dev)
        self.out = torch.empty(T, d, dtype=bf, device=dev)
        self.affinity = (torch.empty(T, E, dtype=torch.float32, device=dev)
                         if self.keep_affinity else None)
        self.ws_bytes = L.moe_workspace_bytes(T, d, E, K, I)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.shared_offsets = torch.tensor([0, T], dtype=i32, device=dev)
        self.T_cap = T
        self._shared_T = T

    def _ensure(self, T: int):
        if T > self.T_cap:
            self._alloc(T)
        if T != self._shared_T:
            self.shared_offsets.copy_(torch.tensor([0, T], dtype=torch.int32))
            self._shared_T = T

    # ------------------------------------------------------------- steps
    def route(self, x: torch.Tensor, stream=None):
        c = self.cfg
        T = x.shape[0]
        self._ensure(T)
        aff = self.affinity[:T] if self.affinity is not None else None
        L.moe_router_topk(x, self.w_split, None, self.logit_offset, self.bias, T, c.d, c.E,
                          c.K, c.n_groups, c.topk_groups, c.route_scale, self.idx, self.gate,
                          self.load, aff, self.status, self.ws, self.ws_bytes, stream)

    def forward(self, x: torch.Tensor, stream=None, marks: dict | None = None) -> torch.Tensor:
        """One layer pass over x bf16 [T, d]; returns the bf16 [T, d] output
        (a view of an internal buffer, valid until the next call).

        `marks`, if given, maps call names ("route", "permute", "routed",
        "shared", "combine") to a pair of CUDA events recorded around that
        call on the stream it runs on."""
        c = self.cfg
        T = x.shape[0]
        R = T * c.K
        main = torch.cuda.current_stream() if stream is None else stream

        def mark(name, i, s=main):
            if marks is not None and name in marks:
                marks[name][i].record(s)

        mark("route", 0)
        self.route(x, stream)
        mark("route", 1)
        mark("permute", 0)
        L.moe_permute(self.idx, T, c.K, c.E, x, c.d, self.offsets, self.row_of, self.tok_of,
                      self.x_perm, self.status, self.ws, self.ws_bytes, stream)
        mark("permute", 1)
        if self.side is not None:
            self.side.wait_stream(main)
            mark("shared", 0, self.side)
            L.moe_grouped_swiglu(x, self.shared_offsets, 1, T, c.d, c.n_shared * c.I, self.ws1,
                                 self.ws3, self.ws2, self.h_sh, self.y_sh, self.status,
                                 self.side)
            mark("shared", 1, self.side)
        mark("routed", 0)
        L.moe_grouped_swiglu(self.x_perm, self.offsets, c.E, R, c.d, c.I, self.w1, self.w3,
                             self.w2, self.h, self.y_perm, self.status, stream)
        mark("routed", 1)
        if self.side is not None:
            main.wait_stream(self.side)
        else:
            mark("shared", 0)
            L.moe_grouped_swiglu(x, self.shared_offsets, 1, T, c.d, c.n_shared * c.I, self.ws1,
                                 self.ws3, self.ws2, self.h_sh, self.y_sh, self.status, stream)
            mark("shared", 1)
        mark("combine", 0)
        L.moe_combine(self.y_perm, self.row_of, self.gate, self.y_sh, T, c.K, c.d,
                      self.out[:T], stream)
        mark("combine", 1)
        return self.out[:T]

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

    def step(self, x: torch.Tensor, stream=None, group=None, marks=None,
             stats_out=None) -> torch.Tensor:
        out = self.forward(x, stream, marks)
        self.bias_update(x.shape[0], stream, group, stats_out)
        return out

    def device_status(self) -> int:
        return int(self.status.item())
