"""CPU oracle of the routed-expert MoE layer (fp64, plain loops in ``oracle.c``).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The CUDA library and its
binding never import it, and it imports nothing from them.

Every function is a thin ctypes wrapper; the arithmetic, with its citations,
is in ``oracle.c``.  Array conventions are those of ``moe_inputs``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

DT = {"f32": 0, "bf16": 1, "e4m3": 2, "e2m1": 3}


class _Mat(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("scale_rows", ctypes.c_int32), ("data", ctypes.c_void_p),
                ("scales", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


def build(verbose: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", _LIB_PATH, src, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    src = os.path.join(_HERE, "oracle.c")
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        build()
    lib = ctypes.CDLL(_LIB_PATH)
    i32, i64, vp, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
    mp = ctypes.POINTER(_Mat)
    lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_decode.restype = dbl
    lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e2m1_decode.restype = dbl
    lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_bf16_encode.argtypes = [dbl]
    lib.orc_bf16_encode.restype = ctypes.c_uint16
    lib.orc_e4m3_decode_array.argtypes = [i64, vp, vp]
    lib.orc_e4m3_encode_array.argtypes = [i64, vp, vp]
    lib.orc_bf16_encode_array.argtypes = [i64, vp, vp]
    lib.orc_route.argtypes = [i32, i32, i32, vp, vp, vp]
    lib.orc_route_grouped.argtypes = [i32, i32, i32, vp, vp, i32, i32, i32, dbl, vp, vp]
    lib.orc_eplb_rebalance.argtypes = [i32, i32, i32, vp, vp, vp, vp]
    lib.orc_token_tiles.argtypes = [i32, vp, i32]
    lib.orc_token_tiles.restype = i64
    lib.orc_pad_waste.argtypes = [i32, i32]
    lib.orc_pad_waste.restype = dbl
    lib.orc_eplb_rebalance.restype = i32
    lib.orc_eplb_invert.argtypes = [i32, i32, vp, i32, vp, vp]
    lib.orc_eplb_invert.restype = i32
    lib.orc_layout.argtypes = [i32] * 7 + [vp] * 7
    lib.orc_layout.restype = i32
    lib.orc_quant_rows_e4m3.argtypes = [i64, i32, vp, vp, vp]
    lib.orc_grouped_swiglu.argtypes = [i32, i32, i32, i32, i32, mp, mp, vp, vp, i32, vp, vp]
    lib.orc_grouped_down.argtypes = [i32, i32, i32, i32, i32, mp, mp, vp, vp, i32, vp]
    lib.orc_combine.argtypes = [i32, i32, i32, i32, mp, vp, vp, i32, vp, vp]
    lib.orc_layer_tokens.argtypes = [i32] * 6 + [vp, mp, i32, mp, mp, i32, i32, i32, i32, vp, vp, vp]
    lib.orc_num_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().orc_num_threads())


# ---- codecs ----------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load().orc_e4m3_decode_array(codes.size, codes.ctypes.data, out.ctypes.data)
    return out


def e2m1_decode(codes) -> np.ndarray:
    """Values of 4-bit E2M1 codes (one code per array element, 0..15)."""
    codes = np.asarray(codes)
    lib = _load()
    table = np.array([lib.orc_e2m1_decode(c) for c in range(16)], np.float64)
    return table[codes.astype(np.int64) & 15]


def e2m1_decode_packed(data) -> np.ndarray:
    """Values of packed E2M1 bytes [..., n] -> [..., 2n] (even column = low nibble)."""
    b = np.asarray(data, np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), np.float64)
    out[..., 0::2] = e2m1_decode(b & 15)
    out[..., 1::2] = e2m1_decode(b >> 4)
    return out


def e4m3_encode(values) -> np.ndarray:
    v = _c(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().orc_e4m3_encode_array(v.size, v.ctypes.data, out.ctypes.data)
    return out


def bf16_encode(values) -> np.ndarray:
    v = _c(values, np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().orc_bf16_encode_array(v.size, v.ctypes.data, out.ctypes.data)
    return out


def bf16_decode(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def quant_rows_e4m3(x) -> tuple[np.ndarray, np.ndarray]:
    """1x128 group quantisation of fp32 rows: (codes [n,H], scales [n,H/128])."""
    x = _c(x, np.float32)
    n, H = x.shape
    q = np.empty((n, H), np.uint8)
    s = np.empty((n, H // 128), np.float32)
    _load().orc_quant_rows_e4m3(n, H, x.ctypes.data, q.ctypes.data, s.ctypes.data)
    return q, s


# ---- matrices --------------------------------------------------------------

def _mat(data, dtype: str, scales=None, scale_rows: int = 1, keep=None):
    """A 2-D view (rows = product of leading dims) of a stored tensor (e2m1:
    packed, the logical row is twice the stored last dim)."""
    cols = data.shape[-1] * (2 if dtype == "e2m1" else 1)
    rows = data.size // data.shape[-1]
    m = _Mat(DT[dtype], scale_rows, data.ctypes.data, 0 if scales is None else scales.ctypes.data, rows, cols)
    if keep is not None:
        keep.extend([data, scales])
    return m


def _np_dtype(dtype: str):
    return {"f32": np.float32, "bf16": np.uint16, "e4m3": np.uint8, "e2m1": np.uint8}[dtype]


def dequant(data, dtype: str, scales=None, scale_rows: int = 1) -> np.ndarray:
    """Real values of a stored 2-D (or batched) tensor, fp64."""
    if dtype == "f32":
        return np.asarray(data, np.float64)
    if dtype == "bf16":
        return bf16_decode(data)
    v = e2m1_decode_packed(data) if dtype == "e2m1" else e4m3_decode(data)
    shp = v.shape
    v2 = v.reshape(-1, shp[-1])
    s = np.asarray(scales, np.float64).reshape(-1, shp[-1] // 128)
    s_full = np.repeat(np.repeat(s, scale_rows, axis=0), 128, axis=1)
    return (v2 * s_full).reshape(shp)


# ---- the steps --------------------------------------------------------------

def route(logits, K: int):
    """a1: ids [T,K] int32 and fp64 weights [T,K]."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float64)
    _load().orc_route(T, E, K, logits.ctypes.data, ids.ctypes.data, w.ctypes.data)
    return ids, w


def route_grouped(logits, K: int, n_group: int, topk_group: int, bias=None, renormalize: bool = True,
                  scale: float = 1.0):
    """Sigmoid scores, bias-corrected grouped top-K: ids [T,K] int32, fp64 weights [T,K]."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    if E % n_group or not (1 <= topk_group <= n_group) or K > (E // n_group) * topk_group:
        raise ValueError("inconsistent grouped routing")
    b = None if bias is None else _c(bias, np.float32)
    ids = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float64)
    _load().orc_route_grouped(T, E, K, logits.ctypes.data, None if b is None else b.ctypes.data, n_group,
                              topk_group, int(renormalize), float(scale), ids.ctypes.data, w.ctypes.data)
    return ids, w


def eplb_invert(p2l, E: int, R: int | None = None):
    """physical_to_logical -> (logical_to_physical [E,R], logical_replica_count [E], max replicas)."""
    p2l = _c(p2l, np.int32)
    P = p2l.size
    R = P if R is None else R
    l2p = np.empty((E, R), np.int32)
    rc = np.empty(E, np.int32)
    r = _load().orc_eplb_invert(P, E, p2l.ctypes.data, R, l2p.ctypes.data, rc.ctypes.data)
    if r < 0:
        raise ValueError("invalid physical_to_logical map (code %d)" % r)
    return l2p[:, :max(r, 1)], rc, r


def eplb_rebalance(window, E: int, p2l=None):
    """Load window [W,P] (+ current map) -> (logical load [E] int64, new physical_to_logical [P])."""
    win = _c(window, np.int32)
    W, P = win.shape
    if P - E > E:
        raise ValueError("more extra slots than experts")
    m = None if p2l is None else _c(p2l, np.int32)
    load = np.empty(E, np.int64)
    new = np.empty(P, np.int32)
    r = _load().orc_eplb_rebalance(P, E, W, win.ctypes.data, None if m is None else m.ctypes.data,
                                   load.ctypes.data, new.ctypes.data)
    if r < 0:
        raise ValueError("invalid physical_to_logical map")
    return load, new


def token_tiles(masked_m, BM: int = 128) -> int:
    """Token tiles the grouped GEMMs issue: sum over slots of ceil(masked_m / BM)."""
    mm = _c(masked_m, np.int32)
    return int(_load().orc_token_tiles(mm.size, mm.ctypes.data, BM))


def pad_waste(M_e: int, BM: int) -> float:
    """MMA work over useful work for one expert of M_e rows in BM-row tiles."""
    return float(_load().orc_pad_waste(M_e, BM))


def layout(cfg, ids, p2l=None):
    """a2 integer outputs: dict(slot_of, masked_m, offsets, row_of, src_of, status)."""
    ids = _c(ids, np.int32)
    T, K = ids.shape
    P, S = cfg.P, cfg.S
    masked = 1 if cfg.layout == "masked" else 0
    slot_of = np.empty((T, K), np.int32)
    masked_m = np.empty(P + S, np.int32)
    offsets = np.empty(P + S + 1, np.int32)
    row_of = np.empty((T, K + S), np.int32)
    src_of = np.full(cfg.rows, -1, np.int32)
    p2l_c = None if p2l is None else _c(p2l, np.int32)
    st = _load().orc_layout(T, K, cfg.E, P, S, masked, cfg.M_max, ids.ctypes.data,
                            None if p2l_c is None else p2l_c.ctypes.data, slot_of.ctypes.data,
                            masked_m.ctypes.data, offsets.ctypes.data, row_of.ctypes.data, src_of.ctypes.data)
    return dict(slot_of=slot_of, masked_m=masked_m, offsets=offsets, row_of=row_of, src_of=src_of, status=st)


def grouped_swiglu(cfg, xg, xg_s, w13, w13_s, masked_m, offsets):
    """a3 over the grouped layout; returns (hg, hg_scales or None) in cfg.h_dtype.

    xg: [rows, H] in cfg.gemm dtype (e4m3 with [rows, H/128] scales);
    w13: slot-indexed [P+S, 2I, H]."""
    keep = []
    masked = 1 if cfg.layout == "masked" else 0
    gd, wd = cfg.gemm, cfg.wt
    xg_m = _mat(_c(xg, _np_dtype(gd)), gd, None if xg_s is None else _c(xg_s, np.float32), 1, keep)
    w_m = _mat(_c(w13, _np_dtype(wd)), wd, None if w13_s is None else _c(w13_s, np.float32), 128, keep)
    mm = _c(masked_m, np.int32)
    off = _c(offsets, np.int32)
    hg = np.zeros((cfg.rows, cfg.I), _np_dtype(cfg.h_dtype))
    hs = np.zeros((cfg.rows, cfg.I // 128), np.float32) if cfg.h_dtype == "e4m3" else None
    _load().orc_grouped_swiglu(mm.size, cfg.H, cfg.I, masked, cfg.M_max, ctypes.byref(xg_m), ctypes.byref(w_m),
                               mm.ctypes.data, off.ctypes.data, DT[cfg.h_dtype], hg.ctypes.data,
                               None if hs is None else hs.ctypes.data)
    return hg, hs


def grouped_down(cfg, hg, hg_s, w2, w2_s, masked_m, offsets):
    """a4 over the grouped layout; returns yg [rows, H] in cfg.y_dtype."""
    keep = []
    masked = 1 if cfg.layout == "masked" else 0
    gd, wd = cfg.gemm, cfg.wt
    h_m = _mat(_c(hg, _np_dtype(gd)), gd, None if hg_s is None else _c(hg_s, np.float32), 1, keep)
    w_m = _mat(_c(w2, _np_dtype(wd)), wd, None if w2_s is None else _c(w2_s, np.float32), 128, keep)
    mm = _c(masked_m, np.int32)
    off = _c(offsets, np.int32)
    yg = np.zeros((cfg.rows, cfg.H), _np_dtype(cfg.y_dtype))
    _load().orc_grouped_down(mm.size, cfg.H, cfg.I, masked, cfg.M_max, ctypes.byref(h_m), ctypes.byref(w_m),
                             mm.ctypes.data, off.ctypes.data, DT[cfg.y_dtype], yg.ctypes.data)
    return yg


def combine(cfg, yg, row_of, w):
    """a5: (out [T,H] in cfg.out dtype, fp64 unrounded sum)."""
    keep = []
    y_m = _mat(_c(yg, _np_dtype(cfg.y_dtype)), cfg.y_dtype, None, 1, keep)
    ro = _c(row_of, np.int32)
    wf = _c(w, np.float32)
    T = ro.shape[0]
    out = np.zeros((T, cfg.H), _np_dtype(cfg.out))
    exact = np.zeros((T, cfg.H), np.float64)
    _load().orc_combine(T, cfg.H, cfg.K, cfg.S, ctypes.byref(y_m), ro.ctypes.data, wf.ctypes.data,
                        DT[cfg.out], out.ctypes.data, exact.ctypes.data)
    return out, exact


def layer(cfg, x, logits, w13, w13_s, w2, w2_s, tokens=None):
    """The whole layer token by token from logical weights [E+S, ...].

    Returns (out rows in cfg.out dtype, fp64 unrounded rows) for ``tokens``
    (default: all T tokens, in order)."""
    keep = []
    T = cfg.T
    toks = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
    gd, wd = cfg.gemm, cfg.wt
    x_m = _mat(_c(x, _np_dtype(cfg.act)), cfg.act, None, 1, keep)
    w13_m = _mat(_c(w13, _np_dtype(wd)), wd, None if w13_s is None else _c(w13_s, np.float32), 128, keep)
    w2_m = _mat(_c(w2, _np_dtype(wd)), wd, None if w2_s is None else _c(w2_s, np.float32), 128, keep)
    lg = _c(logits, np.float32)
    out = np.zeros((toks.size, cfg.H), _np_dtype(cfg.out))
    exact = np.zeros((toks.size, cfg.H), np.float64)
    act_dt = DT["e4m3"] if gd == "e4m3" else DT[cfg.act]
    _load().orc_layer_tokens(T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.S, lg.ctypes.data, ctypes.byref(x_m), act_dt,
                             ctypes.byref(w13_m), ctypes.byref(w2_m), DT[cfg.h_dtype], DT[cfg.y_dtype],
                             DT[cfg.out], toks.size, toks.ctypes.data, out.ctypes.data, exact.ctypes.data)
    return out, exact


def dispatch_values(cfg, x, row_of, rows=None):
    """a2 value output: the grouped activation buffer the dispatch writes.

    Row row_of[t,k] holds x[t] (quantised with the 1x128 rule when the GEMMs
    are e4m3).  Unwritten rows are left as zeros.  Returns (xg, xg_scales)."""
    rows = cfg.rows if rows is None else rows
    ro = np.asarray(row_of)
    T = ro.shape[0]
    if cfg.gemm == "e4m3":
        xf = bf16_decode(x).astype(np.float32) if cfg.act == "bf16" else np.asarray(x, np.float32)
        q, s = quant_rows_e4m3(xf)
        xg = np.zeros((rows, cfg.H), np.uint8)
        xs = np.zeros((rows, cfg.H // 128), np.float32)
        for t in range(T):
            for r in ro[t]:
                if 0 <= r < rows:
                    xg[r] = q[t]
                    xs[r] = s[t]
        return xg, xs
    xg = np.zeros((rows, cfg.H), _np_dtype(cfg.act))
    for t in range(T):
        for r in ro[t]:
            if 0 <= r < rows:
                xg[r] = x[t]
    return xg, None
