"""Seeded synthetic workloads for the routed-expert MoE layer.

This module describes the five workloads (shapes, dtypes, layouts, value
distributions) and draws their inputs with the counter-based generator in
``gen.c``.  It holds none of the layer's arithmetic: it does not route,
dispatch, run an expert or combine.  The CPU oracle and the CUDA path both
read the arrays it returns.

Storage conventions (shared by every consumer):
  * bf16 arrays are ``uint16`` bit patterns; e4m3 arrays are ``uint8`` codes;
    e2m1 (FP4) weights are ``uint8`` bytes of two codes along the reduced
    dimension (even column in the low nibble), so their last dim is halved.
  * Expert weights are stored transposed, rows contiguous along the reduced
    dimension: ``w13 [n_exp, 2I, H]`` = gate rows (W1^T) then up rows (W3^T);
    ``w2 [n_exp, H, I]`` (W2^T).  e4m3 weights carry fp32 scales per 128x128
    block: ``w13_s [n_exp, 2I/128, H/128]``, ``w2_s [n_exp, H/128, I/128]``;
    e2m1 weights carry the same block scales.
  * With a shared expert it is logical expert ``E`` (the last one).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libmoe_inputs.so")
_lib = None

# tensor stream ids of the generator
STREAM_X, STREAM_LOGITS, STREAM_WG, STREAM_W13, STREAM_W2, STREAM_W13S, STREAM_W2S = 1, 2, 3, 4, 5, 6, 7


@dataclasses.dataclass(frozen=True)
class MoeConfig:
    name: str
    T: int            # tokens
    H: int            # hidden size
    I: int            # expert intermediate size
    E: int            # logical routed experts
    K: int            # experts per token
    shared: int       # 1 = one always-on shared expert
    act: str          # dtype of x as given to the layer: f32 | bf16 (e4m3 activations are quantised by the dispatch)
    gemm: str         # arithmetic type of the expert GEMMs: f32 | bf16 | e4m3
    out: str          # output dtype: f32 | bf16
    layout: str       # masked | contig
    M_max: int        # rows per slot of the masked layout (0 for contig)
    redundant: int    # extra physical slots filled with replicas of hot experts
    router: str       # wg (logits = x @ W_g) | normal (logits ~ N(0,1)) | zipf (N(0,1) + Zipf bias)
    wg_std: float
    w_std: float
    zipf_s: float = 0.0
    description: str = ""
    wq: str = ""      # weight storage type when it differs from `gemm` ("e2m1": FP4 weights, e4m3 activations)

    @property
    def wt(self) -> str:
        """Type of the stored expert weights."""
        return self.wq or self.gemm

    @property
    def P(self) -> int:
        return self.E + self.redundant

    @property
    def S(self) -> int:
        return self.shared

    @property
    def n_exp(self) -> int:
        """Logical experts including the shared one."""
        return self.E + self.shared

    @property
    def rows(self) -> int:
        """Rows of the grouped activation buffers."""
        if self.layout == "masked":
            return (self.P + self.S) * self.M_max
        return self.T * self.K + self.S * self.T

    @property
    def h_dtype(self) -> str:
        return self.gemm

    @property
    def y_dtype(self) -> str:
        return "f32" if self.gemm == "f32" else "bf16"

    def replace(self, **kw) -> "MoeConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": MoeConfig(
        "tiny", T=16, H=64, I=128, E=8, K=2, shared=0, act="f32", gemm="f32", out="f32",
        layout="masked", M_max=16, redundant=0, router="wg", wg_std=0.1, w_std=0.05,
        description="tiny MoE layer T=16 H=64 I=128 E=8 K=2, fp32"),
    "mixtral_decode": MoeConfig(
        "mixtral_decode", T=32, H=4096, I=14336, E=8, K=2, shared=0, act="bf16", gemm="bf16",
        out="bf16", layout="masked", M_max=32, redundant=0, router="wg", wg_std=0.02, w_std=0.02,
        description="Mixtral-8x7B-shaped decode layer T=32 H=4096 I=14336 E=8 K=2, bf16, masked [8,32,4096]"),
    "dsv3_decode": MoeConfig(
        "dsv3_decode", T=128, H=7168, I=2048, E=256, K=8, shared=1, act="bf16", gemm="e4m3",
        out="bf16", layout="masked", M_max=128, redundant=0, router="normal", wg_std=0.0, w_std=0.02,
        description="DeepSeek-V3-shaped decode layer T=128 H=7168 I=2048 E=256+1 shared K=8, "
                    "e4m3 128x128-block weights, 1x128 activations, masked [257,128,7168]"),
    "skew_eplb": MoeConfig(
        "skew_eplb", T=256, H=7168, I=2048, E=256, K=8, shared=1, act="bf16", gemm="e4m3",
        out="bf16", layout="masked", M_max=256, redundant=32, router="zipf", wg_std=0.0, w_std=0.02,
        zipf_s=1.2,
        description="Zipf(1.2)-skewed routing with 32 EPLB replicas (288 slots + shared), "
                    "DeepSeek-V3 shapes, T=256, masked [289,256,7168]"),
    "prefill": MoeConfig(
        "prefill", T=8192, H=4096, I=1024, E=512, K=10, shared=0, act="bf16", gemm="e4m3",
        out="bf16", layout="contig", M_max=0, redundant=0, router="normal", wg_std=0.0, w_std=0.02,
        description="prefill grouped layer T=8192 H=4096 I=1024 E=512 K=10, e4m3, contiguous layout"),
    "dsv4_fp4_decode": MoeConfig(
        "dsv4_fp4_decode", T=128, H=7168, I=2048, E=384, K=6, shared=1, act="bf16", gemm="e4m3",
        out="bf16", layout="masked", M_max=128, redundant=0, router="normal", wg_std=0.0, w_std=0.02, wq="e2m1",
        description="DS-V4-Pro-shaped decode layer with FP4 experts T=128 H=7168 I=2048 E=384+1 shared K=6, "
                    "e2m1 128x128-block weights, e4m3 1x128 activations, masked [385,128,7168]"),
}

CONFIG_ORDER = ["tiny", "mixtral_decode", "dsv3_decode", "skew_eplb", "prefill"]


def build(verbose: bool = False) -> str:
    """Compile gen.c into libmoe_inputs.so next to this file."""
    src = os.path.join(_HERE, "gen.c")
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", _LIB_PATH, src, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    src = os.path.join(_HERE, "gen.c")
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        build()
    lib = ctypes.CDLL(_LIB_PATH)
    u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    for name in ("mg_normal_f64", "mg_normal_f32", "mg_normal_bf16", "mg_uniform_f64"):
        getattr(lib, name).argtypes = [u64, u64, u64, i64, dbl, dbl, vp]
        getattr(lib, name).restype = None
    lib.mg_weights_e4m3.argtypes = [u64, u64, u64, i64, i64, i64, i64, dbl, vp, vp]
    lib.mg_weights_e2m1.argtypes = [u64, u64, u64, i64, i64, i64, i64, dbl, vp, vp]
    lib.mg_weights_bf16.argtypes = [u64, u64, i64, i64, i64, i64, dbl, vp]
    lib.mg_weights_f32.argtypes = [u64, u64, i64, i64, i64, i64, dbl, vp]
    lib.mg_num_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def normal(seed: int, stream: int, shape, mean=0.0, std=1.0, dtype="f64", offset: int = 0) -> np.ndarray:
    """Counter-based N(mean, std^2) draws; dtype f64 | f32 | bf16 (uint16 bits)."""
    lib = _load()
    n = int(np.prod(shape))
    if dtype == "f64":
        out = np.empty(n, np.float64)
        lib.mg_normal_f64(seed, stream, offset, n, mean, std, out.ctypes.data)
    elif dtype == "f32":
        out = np.empty(n, np.float32)
        lib.mg_normal_f32(seed, stream, offset, n, mean, std, out.ctypes.data)
    elif dtype == "bf16":
        out = np.empty(n, np.uint16)
        lib.mg_normal_bf16(seed, stream, offset, n, mean, std, out.ctypes.data)
    else:
        raise ValueError(dtype)
    return out.reshape(shape)


def uniform(seed: int, stream: int, shape, lo=0.0, hi=1.0, offset: int = 0) -> np.ndarray:
    lib = _load()
    n = int(np.prod(shape))
    out = np.empty(n, np.float64)
    lib.mg_uniform_f64(seed, stream, offset, n, lo, hi, out.ctypes.data)
    return out.reshape(shape)


def bf16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (input preparation helper)."""
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def expert_weights(cfg: MoeConfig, which: str, e0: int = 0, ne: int | None = None, seed: int = 0):
    """Weights of logical experts [e0, e0+ne) of ``w13`` or ``w2``.

    Returns (data, scales); scales is None unless the weights are e4m3 or e2m1."""
    lib = _load()
    ne = cfg.n_exp - e0 if ne is None else ne
    if which == "w13":
        N, Kd, ws, ss = 2 * cfg.I, cfg.H, STREAM_W13, STREAM_W13S
    elif which == "w2":
        N, Kd, ws, ss = cfg.H, cfg.I, STREAM_W2, STREAM_W2S
    else:
        raise ValueError(which)
    if cfg.wt == "e2m1":
        q = np.empty((ne, N, Kd // 2), np.uint8)
        s = np.empty((ne, N // 128, Kd // 128), np.float32)
        lib.mg_weights_e2m1(seed, ws, ss, e0, ne, N, Kd, cfg.w_std, q.ctypes.data, s.ctypes.data)
        return q, s
    if cfg.gemm == "e4m3":
        q = np.empty((ne, N, Kd), np.uint8)
        s = np.empty((ne, N // 128, Kd // 128), np.float32)
        lib.mg_weights_e4m3(seed, ws, ss, e0, ne, N, Kd, cfg.w_std, q.ctypes.data, s.ctypes.data)
        return q, s
    if cfg.gemm == "bf16":
        w = np.empty((ne, N, Kd), np.uint16)
        lib.mg_weights_bf16(seed, ws, e0, ne, N, Kd, cfg.w_std, w.ctypes.data)
        return w, None
    w = np.empty((ne, N, Kd), np.float32)
    lib.mg_weights_f32(seed, ws, e0, ne, N, Kd, cfg.w_std, w.ctypes.data)
    return w, None


def activations(cfg: MoeConfig, seed: int = 0):
    """x [T,H] (f32, or bf16 bits) and router logits [T,E] fp32.

    Router logits: 'wg' -> fp32(x @ W_g) evaluated in fp64 with W_g [H,E] drawn
    N(0, wg_std^2) (bf16 when x is bf16); 'normal' -> N(0,1);
    'zipf' -> N(0,1) - s*ln(e+1), expert 0 the hottest."""
    T, H, E = cfg.T, cfg.H, cfg.E
    if cfg.act == "f32":
        x = normal(seed, STREAM_X, (T, H), dtype="f32")
        xf = x.astype(np.float64)
    else:
        x = normal(seed, STREAM_X, (T, H), dtype="bf16")
        xf = bf16_bits_to_f64(x)
    if cfg.router == "wg":
        if cfg.act == "f32":
            wg = normal(seed, STREAM_WG, (H, E), std=cfg.wg_std, dtype="f32").astype(np.float64)
        else:
            wg = bf16_bits_to_f64(normal(seed, STREAM_WG, (H, E), std=cfg.wg_std, dtype="bf16"))
        logits = (xf @ wg).astype(np.float32)
    elif cfg.router == "normal":
        logits = normal(seed, STREAM_LOGITS, (T, E), dtype="f32")
    elif cfg.router == "zipf":
        bias = -cfg.zipf_s * np.log(np.arange(E, dtype=np.float64) + 1.0)
        logits = (normal(seed, STREAM_LOGITS, (T, E)) + bias[None, :]).astype(np.float32)
    else:
        raise ValueError(cfg.router)
    return x, logits


def replica_map(counts: np.ndarray, E: int, n_redundant: int) -> np.ndarray:
    """physical_to_logical map: slots 0..E-1 hold experts 0..E-1; the next
    n_redundant slots hold the hottest experts by count (descending, ties to the
    lower expert index).  ``counts`` is the per-logical-expert routing count of
    the batch, supplied by the caller."""
    counts = np.asarray(counts, dtype=np.int64)
    order = sorted(range(E), key=lambda e: (-int(counts[e]), e))
    return np.array(list(range(E)) + order[:n_redundant], dtype=np.int32)


def slot_experts(cfg: MoeConfig, p2l: np.ndarray | None) -> np.ndarray:
    """Logical expert held by each of the P+S slots (shared expert last)."""
    base = np.arange(cfg.E, dtype=np.int64) if p2l is None else np.asarray(p2l, np.int64)
    if cfg.shared:
        base = np.concatenate([base, [cfg.E]])
    return base


def num_threads() -> int:
    return int(_load().mg_num_threads())
