"""The five calls of the forward pass chained over caller-owned device buffers.

PyTorch provides device memory and the stream; each step runs in the
library's kernels.  Buffers are allocated once (static shapes), so a forward
call is graph-capturable after a first eager call."""
from __future__ import annotations

import torch

from . import _lib as L

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8, "e2m1": torch.uint8}


class MoeLayer:
    """Buffers and calls for one problem.  Weights are slot-indexed tensors on the
    device: w13 [P+S, 2I, H], w2 [P+S, H, I] (e4m3: uint8 codes with fp32 block
    scales w13_s [P+S, 2I/128, H/128], w2_s [P+S, H/128, I/128]; e2m1: the same
    with two codes per byte, w13 [P+S, 2I, H/2], w2 [P+S, H, I/2]).  With e4m3
    or e2m1 weights the grouped activations xg, hg are e4m3 with 1x128 scales."""

    def __init__(self, problem: L.Problem, act: str, wt: str, out: str, w13, w2, w13_s=None, w2_s=None,
                 phys_to_log=None, device="cuda"):
        self.p = problem
        self.act, self.wt, self.out_dt = act, wt, out
        st = L.moe_check_problem(problem)
        if st != L.MOE_OK:
            raise L.MoeError(st, "problem")
        p = problem
        dev = torch.device(device)
        self.w13, self.w2, self.w13_s, self.w2_s = w13, w2, w13_s, w2_s
        self.p2l = phys_to_log
        S = p.has_shared
        rows = L.moe_grouped_rows(p)
        self.rows = rows
        i32 = dict(dtype=torch.int32, device=dev)
        self.ids = torch.empty((p.T, p.K), **i32)
        self.w = torch.empty((p.T, p.K), dtype=torch.float32, device=dev)
        self.masked_m = torch.empty(p.P + S, **i32)
        self.offsets = torch.empty(p.P + S + 1, **i32)
        self.row_of = torch.empty((p.T, p.K + S), **i32)
        self.src_of = torch.full((rows,), -1, **i32)
        f8 = wt in ("e4m3", "e2m1")
        gd = TORCH_DTYPE[wt]
        yd = torch.float32 if wt == "f32" else torch.bfloat16
        self.xg = torch.empty((rows, p.H), dtype=gd, device=dev)
        self.hg = torch.empty((rows, p.I), dtype=gd, device=dev)
        self.yg = torch.empty((rows, p.H), dtype=yd, device=dev)
        self.xg_s = torch.empty((rows, p.H // 128), dtype=torch.float32, device=dev) if f8 else None
        self.hg_s = torch.empty((rows, p.I // 128), dtype=torch.float32, device=dev) if f8 else None
        self.out = torch.empty((p.T, p.H), dtype=TORCH_DTYPE[out], device=dev)
        self.err = torch.zeros(1, **i32)
        nbytes = max(L.moe_workspace_bytes(p), 256)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    # -- the steps --------------------------------------------------------------
    def route(self, logits, stream=None):
        L.moe_route_topk(self.p, logits, self.ids, self.w, stream)

    def route_grouped(self, logits, n_group, topk_group, bias=None, renormalize=True, scale=1.0, stream=None):
        """DeepSeek-style grouped top-k (sigmoid, bias for the choice only) in place of route()."""
        L.moe_route_grouped_topk(self.p, logits, bias, n_group, topk_group, self.ids, self.w,
                                 renormalize=renormalize, scale=scale, stream=stream)

    def permute(self, x, stream=None):
        L.moe_permute(self.p, self.ids, x, self.p2l, self.masked_m, self.offsets, self.row_of, self.src_of,
                      self.xg, self.xg_s, self.err, self.ws, stream)

    def swiglu(self, stream=None):
        L.moe_grouped_swiglu_gemm(self.p, self.xg, self.xg_s, self.w13, self.w13_s, self.masked_m, self.offsets,
                                  self.hg, self.hg_s, self.err, self.ws, stream)

    def down(self, stream=None):
        L.moe_grouped_down_gemm(self.p, self.hg, self.hg_s, self.w2, self.w2_s, self.masked_m, self.offsets,
                                self.yg, self.err, self.ws, stream)

    def ffn(self, stream=None):
        """gate/up + SwiGLU and down in one launch (moe_grouped_ffn); same outputs as swiglu() + down()."""
        L.moe_grouped_ffn(self.p, self.xg, self.xg_s, self.w13, self.w13_s, self.w2, self.w2_s, self.masked_m,
                          self.offsets, self.hg, self.hg_s, self.yg, self.err, self.ws, stream)

    def combine(self, stream=None):
        L.moe_combine(self.p, self.yg, self.row_of, self.w, self.out, stream)

    def route_permute(self, logits, x, stream=None):
        """route() + permute() in one call (moe_route_permute; one launch for small batches)."""
        L.moe_route_permute(self.p, logits, x, self.p2l, self.ids, self.w, self.masked_m, self.offsets, self.row_of,
                            self.src_of, self.xg, self.xg_s, self.err, self.ws, stream)

    def ffn_combine(self, stream=None):
        """gate/up, down and combine in one call (moe_ffn_combine); same outputs as swiglu() + down() + combine()."""
        L.moe_ffn_combine(self.p, self.xg, self.xg_s, self.w13, self.w13_s, self.w2, self.w2_s, self.masked_m,
                          self.offsets, self.row_of, self.w, self.hg, self.hg_s, self.yg, self.out, self.err, self.ws,
                          stream)

    def forward(self, x, logits, stream=None, fused=False):
        """route -> permute -> gate/up -> down -> combine; returns self.out.  fused=True makes the
        same pass with the fused calls: route_permute() and ffn_combine()."""
        if fused:
            self.route_permute(logits, x, stream)
            self.ffn_combine(stream)
            return self.out
        self.route(logits, stream)
        self.permute(x, stream)
        self.swiglu(stream)
        self.down(stream)
        self.combine(stream)
        return self.out
