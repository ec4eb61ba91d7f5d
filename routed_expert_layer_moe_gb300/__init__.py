"""Single-GPU forward pass of one routed Mixture-of-Experts layer on GB300.

The compute lives in ``libmoe_gb300.so`` (hand-written CUDA for sm_103a,
C ABI in ``include/moe.h``); this package is its ctypes binding plus a
buffer-owning helper that chains the five calls."""
from ._lib import (EXPORTS, LIB_PATH, MOE_E2M1, MOE_E4M3, MOE_BF16, MOE_F32, MOE_FLAG_BAD_EXPERT,
                   MOE_FLAG_BAD_MAP, MOE_FLAG_OVERFLOW, MOE_FLAG_TIMEOUT, MOE_LAYOUT_CONTIG, MOE_LAYOUT_MASKED, MOE_ERR_CUDA,
                   MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_OK, MOE_STATS_BYTES, MOE_STATS_CTAS,
                   MoeError, Problem, lib,
                   moe_check_problem, moe_combine, moe_ffn_combine, moe_gemm_tile_rows, moe_eplb_invert, moe_eplb_rebalance, moe_eplb_record,
                   moe_grouped_down_gemm, moe_grouped_ffn, moe_grouped_rows, moe_grouped_swiglu_gemm, moe_permute,
                   moe_permute_no_workspace, moe_route_grouped_topk, moe_route_permute, moe_route_topk, moe_selftest_bounded_wait,
                   moe_version,
                   moe_workspace_bytes, status_string)
from .layer import MoeLayer

__all__ = [n for n in dir() if not n.startswith("_")]
