"""Helpers shared by the GPU parity tests: inputs on the device, the problem
struct of a workload, and the error measure max|err| / max|ref|."""
from __future__ import annotations

import numpy as np
import torch

import moe_inputs as mi
import oracle
import routed_expert_layer_moe_gb300 as moe

TOL = {"f32": 1e-4, "bf16": 1e-2, "e4m3": 3e-2}  # by the type of the GEMM operands (e4m3 also for e2m1 weights)


def problem_of(cfg) -> moe.Problem:
    return moe.Problem.make(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, P=cfg.P, M_max=cfg.M_max,
                            has_shared=cfg.S, act=cfg.act, wt=cfg.wt, out=cfg.out, layout=cfg.layout)


def to_dev(a: np.ndarray | None, dev="cuda"):
    """numpy storage array -> device tensor (uint16 arrays become bf16)."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def to_host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def real(a: np.ndarray, dtype: str, scales=None) -> np.ndarray:
    """fp64 values of a stored activation array ([rows, cols], 1x128 e4m3 groups)."""
    return oracle.dequant(a, dtype, scales, 1)


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got, np.float64)
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


class Workload:
    """Host inputs of one workload, the oracle's routing, and device tensors."""

    def __init__(self, cfg, seed=0, logits=None, x=None, weights=None):
        self.cfg = cfg
        x0, lg0 = mi.activations(cfg, seed)
        self.x = x0 if x is None else x
        self.logits = lg0 if logits is None else logits
        if weights is None:
            self.w13, self.w13_s = mi.expert_weights(cfg, "w13", seed=seed)
            self.w2, self.w2_s = mi.expert_weights(cfg, "w2", seed=seed)
        else:
            self.w13, self.w13_s, self.w2, self.w2_s = weights
        self.ids, self.w = oracle.route(self.logits, cfg.K)
        self.p2l = None
        if cfg.redundant:
            counts = np.bincount(self.ids.ravel(), minlength=cfg.E)
            self.p2l = mi.replica_map(counts, cfg.E, cfg.redundant)
        self.order = mi.slot_experts(cfg, self.p2l)
        self.problem = problem_of(cfg)

    def device_weights(self):
        """Slot-indexed weights on the device (replicas are copies, gathered on the device)."""
        idx = torch.from_numpy(self.order).cuda()

        def slots(a):
            if a is None:
                return None
            t = to_dev(a)
            return t if len(self.order) == t.shape[0] and (self.order == np.arange(len(self.order))).all() \
                else t.index_select(0, idx).contiguous()

        return slots(self.w13), slots(self.w13_s), slots(self.w2), slots(self.w2_s)

    def layer(self) -> moe.MoeLayer:
        w13, w13s, w2, w2s = self.device_weights()
        p2l = None if self.p2l is None else torch.from_numpy(self.p2l).cuda()
        return moe.MoeLayer(self.problem, self.cfg.act, self.cfg.wt, self.cfg.out, w13, w2, w13s, w2s,
                            phys_to_log=p2l)
