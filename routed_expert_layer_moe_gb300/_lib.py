"""ctypes binding of libmoe_gb300.so (the C ABI declared in include/moe.h).

Argument marshalling only: tensors become device pointers, the stream becomes
a cudaStream_t.  Every step runs in the library's CUDA kernels; there is no
other implementation to fall back to, so a missing library is an error."""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_WORKSPACE = 0, -1, -2, -3, -4
MOE_F32, MOE_BF16, MOE_E4M3, MOE_E2M1 = 0, 1, 2, 3
MOE_LAYOUT_MASKED, MOE_LAYOUT_CONTIG = 0, 1
MOE_FLAG_OVERFLOW, MOE_FLAG_BAD_EXPERT, MOE_FLAG_BAD_MAP, MOE_FLAG_TIMEOUT = 1, 2, 4, 8
MOE_STATS_CTAS = 256                        # issue counters at the start of the workspace (include/moe.h)
MOE_STATS_BYTES = 2 * MOE_STATS_CTAS * 2 * 4

DTYPES = {"f32": MOE_F32, "bf16": MOE_BF16, "e4m3": MOE_E4M3, "e2m1": MOE_E2M1}
LAYOUTS = {"masked": MOE_LAYOUT_MASKED, "contig": MOE_LAYOUT_CONTIG}

# every symbol include/moe.h declares
EXPORTS = ["moe_version", "moe_status_string", "moe_grouped_rows", "moe_workspace_bytes", "moe_check_problem",
           "moe_gemm_tile_rows",
           "moe_route_topk", "moe_route_grouped_topk", "moe_permute", "moe_permute_no_workspace",
           "moe_grouped_swiglu_gemm", "moe_grouped_down_gemm", "moe_grouped_ffn", "moe_combine",
           "moe_route_permute", "moe_ffn_combine",
           "moe_eplb_record", "moe_eplb_rebalance", "moe_eplb_invert", "moe_selftest_bounded_wait"]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (where, status_string(status), status))


class Problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "H", "I", "E", "K", "P", "M_max", "has_shared", "act", "wt", "out", "layout")]

    @classmethod
    def make(cls, T, H, I, E, K, P=None, M_max=0, has_shared=0, act="bf16", wt="bf16", out="bf16",
             layout="masked") -> "Problem":
        return cls(T, H, I, E, K, E if P is None else P, M_max, has_shared, DTYPES[act], DTYPES[wt], DTYPES[out],
                   LAYOUTS[layout])

    def __repr__(self):
        return "Problem(%s)" % ", ".join("%s=%d" % (n, getattr(self, n)) for n, _ in self._fields_)


_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("%s is missing: build it with routed_expert_layer_moe_gb300.build.build() "
                          "(or __graft_entry__.build()); there is no other implementation" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    pp = ctypes.POINTER(Problem)
    L.moe_version.restype = i32
    L.moe_status_string.argtypes = [i32]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_grouped_rows.argtypes = [pp]
    L.moe_grouped_rows.restype = i64
    L.moe_workspace_bytes.argtypes = [pp]
    L.moe_workspace_bytes.restype = sz
    L.moe_check_problem.argtypes = [pp]
    L.moe_check_problem.restype = i32
    L.moe_gemm_tile_rows.argtypes = [pp, i32]
    L.moe_gemm_tile_rows.restype = i32
    L.moe_route_topk.argtypes = [pp, vp, vp, vp, vp]
    L.moe_route_topk.restype = i32
    L.moe_route_grouped_topk.argtypes = [pp, vp, vp, i32, i32, i32, ctypes.c_float, vp, vp, vp]
    L.moe_route_grouped_topk.restype = i32
    L.moe_permute.argtypes = [pp] + [vp] * 11 + [sz, vp]
    L.moe_permute.restype = i32
    L.moe_permute_no_workspace.argtypes = [pp] + [vp] * 11
    L.moe_permute_no_workspace.restype = i32
    L.moe_grouped_swiglu_gemm.argtypes = [pp] + [vp] * 10 + [sz, vp]
    L.moe_grouped_swiglu_gemm.restype = i32
    L.moe_grouped_down_gemm.argtypes = [pp] + [vp] * 9 + [sz, vp]
    L.moe_grouped_down_gemm.restype = i32
    L.moe_grouped_ffn.argtypes = [pp] + [vp] * 13 + [sz, vp]
    L.moe_grouped_ffn.restype = i32
    L.moe_route_permute.argtypes = [pp] + [vp] * 13 + [sz, vp]
    L.moe_route_permute.restype = i32
    L.moe_ffn_combine.argtypes = [pp] + [vp] * 16 + [sz, vp]
    L.moe_ffn_combine.restype = i32
    L.moe_combine.argtypes = [pp, vp, vp, vp, vp, vp]
    L.moe_combine.restype = i32
    L.moe_eplb_record.argtypes = [pp, vp, i64, i32, vp, vp]
    L.moe_eplb_record.restype = i32
    L.moe_eplb_rebalance.argtypes = [pp, vp, i32, vp, vp, vp, vp, vp]
    L.moe_eplb_rebalance.restype = i32
    L.moe_selftest_bounded_wait.argtypes = [i64, vp, vp]
    L.moe_selftest_bounded_wait.restype = i32
    L.moe_eplb_invert.argtypes = [i32, i32, vp, i32, vp, vp]
    L.moe_eplb_invert.restype = i32
    _lib = L
    return L


def status_string(s: int) -> str:
    return lib().moe_status_string(s).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def moe_version() -> int:
    return lib().moe_version()


def moe_check_problem(p: Problem) -> int:
    return lib().moe_check_problem(ctypes.byref(p))


def moe_gemm_tile_rows(p: Problem, step: int) -> int:
    return lib().moe_gemm_tile_rows(ctypes.byref(p), step)


def moe_grouped_rows(p: Problem) -> int:
    return lib().moe_grouped_rows(ctypes.byref(p))


def moe_workspace_bytes(p: Problem) -> int:
    return lib().moe_workspace_bytes(ctypes.byref(p))


def moe_route_topk(p: Problem, logits, ids, w, stream=None) -> None:
    _check(lib().moe_route_topk(ctypes.byref(p), _ptr(logits), _ptr(ids), _ptr(w), _stream(stream)),
           "moe_route_topk")


def moe_route_grouped_topk(p: Problem, logits, bias, n_group: int, topk_group: int, ids, w, renormalize=True,
                           scale: float = 1.0, stream=None) -> None:
    _check(lib().moe_route_grouped_topk(ctypes.byref(p), _ptr(logits), _ptr(bias), n_group, topk_group,
                                        int(bool(renormalize)), float(scale), _ptr(ids), _ptr(w), _stream(stream)),
           "moe_route_grouped_topk")


def moe_permute(p: Problem, ids, x, phys_to_log, masked_m, offsets, row_of, src_of, xg, xg_scales, err_flag,
                workspace, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().moe_permute(ctypes.byref(p), _ptr(ids), _ptr(x), _ptr(phys_to_log), _ptr(masked_m),
                             _ptr(offsets), _ptr(row_of), _ptr(src_of), _ptr(xg), _ptr(xg_scales),
                             _ptr(err_flag), _ptr(workspace), nbytes, _stream(stream)), "moe_permute")


def moe_permute_no_workspace(p: Problem, ids, x, phys_to_log, masked_m, offsets, row_of, src_of, xg, xg_scales,
                             err_flag, stream=None) -> None:
    """moe_permute without a workspace argument, for callers that cannot allocate
    device memory; its scratch is a fixed array inside the library (see moe.h)."""
    _check(lib().moe_permute_no_workspace(ctypes.byref(p), _ptr(ids), _ptr(x), _ptr(phys_to_log), _ptr(masked_m),
                                          _ptr(offsets), _ptr(row_of), _ptr(src_of), _ptr(xg), _ptr(xg_scales),
                                          _ptr(err_flag), _stream(stream)), "moe_permute_no_workspace")


def moe_grouped_swiglu_gemm(p: Problem, xg, xg_scales, w13, w13_scales, masked_m, offsets, hg, hg_scales,
                            err_flag, workspace, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().moe_grouped_swiglu_gemm(ctypes.byref(p), _ptr(xg), _ptr(xg_scales), _ptr(w13), _ptr(w13_scales),
                                         _ptr(masked_m), _ptr(offsets), _ptr(hg), _ptr(hg_scales), _ptr(err_flag),
                                         _ptr(workspace), nbytes, _stream(stream)), "moe_grouped_swiglu_gemm")


def moe_grouped_down_gemm(p: Problem, hg, hg_scales, w2, w2_scales, masked_m, offsets, yg, err_flag, workspace,
                          stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().moe_grouped_down_gemm(ctypes.byref(p), _ptr(hg), _ptr(hg_scales), _ptr(w2), _ptr(w2_scales),
                                       _ptr(masked_m), _ptr(offsets), _ptr(yg), _ptr(err_flag), _ptr(workspace),
                                       nbytes, _stream(stream)), "moe_grouped_down_gemm")


def moe_grouped_ffn(p: Problem, xg, xg_scales, w13, w13_scales, w2, w2_scales, masked_m, offsets, hg, hg_scales, yg,
                    err_flag, workspace, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().moe_grouped_ffn(ctypes.byref(p), _ptr(xg), _ptr(xg_scales), _ptr(w13), _ptr(w13_scales), _ptr(w2),
                                 _ptr(w2_scales), _ptr(masked_m), _ptr(offsets), _ptr(hg), _ptr(hg_scales), _ptr(yg),
                                 _ptr(err_flag), _ptr(workspace), nbytes, _stream(stream)), "moe_grouped_ffn")


def moe_route_permute(p: Problem, logits, x, phys_to_log, ids, w, masked_m, offsets, row_of, src_of, xg, xg_scales,
                      err_flag, workspace, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().moe_route_permute(ctypes.byref(p), _ptr(logits), _ptr(x), _ptr(phys_to_log), _ptr(ids), _ptr(w),
                                   _ptr(masked_m), _ptr(offsets), _ptr(row_of), _ptr(src_of), _ptr(xg),
                                   _ptr(xg_scales), _ptr(err_flag), _ptr(workspace), nbytes, _stream(stream)),
           "moe_route_permute")


def moe_ffn_combine(p: Problem, xg, xg_scales, w13, w13_scales, w2, w2_scales, masked_m, offsets, row_of, w, hg,
                    hg_scales, yg, out, err_flag, workspace, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().moe_ffn_combine(ctypes.byref(p), _ptr(xg), _ptr(xg_scales), _ptr(w13), _ptr(w13_scales), _ptr(w2),
                                 _ptr(w2_scales), _ptr(masked_m), _ptr(offsets), _ptr(row_of), _ptr(w), _ptr(hg),
                                 _ptr(hg_scales), _ptr(yg), _ptr(out), _ptr(err_flag), _ptr(workspace), nbytes,
                                 _stream(stream)), "moe_ffn_combine")


def moe_combine(p: Problem, yg, row_of, w, out, stream=None) -> None:
    _check(lib().moe_combine(ctypes.byref(p), _ptr(yg), _ptr(row_of), _ptr(w), _ptr(out), _stream(stream)),
           "moe_combine")


def moe_eplb_record(p: Problem, masked_m, pass_index: int, window: int, load_window, stream=None) -> None:
    _check(lib().moe_eplb_record(ctypes.byref(p), _ptr(masked_m), int(pass_index), int(window), _ptr(load_window),
                                 _stream(stream)), "moe_eplb_record")


def moe_eplb_rebalance(p: Problem, load_window, window: int, phys_to_log, logical_load, new_phys_to_log, err_flag,
                       stream=None) -> None:
    _check(lib().moe_eplb_rebalance(ctypes.byref(p), _ptr(load_window), int(window), _ptr(phys_to_log),
                                    _ptr(logical_load), _ptr(new_phys_to_log), _ptr(err_flag), _stream(stream)),
           "moe_eplb_rebalance")


def moe_selftest_bounded_wait(cycles: int, err_flag, stream=None) -> None:
    _check(lib().moe_selftest_bounded_wait(int(cycles), _ptr(err_flag), _stream(stream)), "moe_selftest_bounded_wait")


def moe_eplb_invert(p2l, E: int, R: int):
    """Host helper: (logical_to_physical [E,R], logical_replica_count [E], max replicas)."""
    import numpy as np
    p2l = np.ascontiguousarray(p2l, dtype=np.int32)
    l2p = np.empty((E, R), np.int32)
    rc = np.empty(E, np.int32)
    r = lib().moe_eplb_invert(p2l.size, E, p2l.ctypes.data, R, l2p.ctypes.data, rc.ctypes.data)
    if r < 0:
        raise MoeError(r, "moe_eplb_invert")
    return l2p, rc, r
