"""The C ABI on the host: the library loads, exports every symbol include/moe.h
declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import routed_expert_layer_moe_gb300 as moe
from routed_expert_layer_moe_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    moe_build.build()


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol():
    L = moe.lib()
    declared = header_functions()
    assert set(declared) == set(moe.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name
    assert moe.moe_version() >> 16 == 1


def test_problem_checks_without_gpu():
    ok = moe.Problem.make(T=32, H=4096, I=14336, E=8, K=2, M_max=32)
    assert moe.moe_check_problem(ok) == moe.MOE_OK
    assert moe.moe_grouped_rows(ok) == 8 * 32
    assert moe.moe_workspace_bytes(ok) > 0
    bad = [
        dict(T=-1), dict(K=0), dict(K=9), dict(E=0), dict(P=7), dict(M_max=0), dict(E=2000, P=2000),
        dict(has_shared=1, M_max=16),
    ]
    for b in bad:
        kw = dict(T=32, H=4096, I=14336, E=8, K=2, M_max=32)
        kw.update(b)
        assert moe.moe_check_problem(moe.Problem.make(**kw)) == moe.MOE_ERR_INVALID, b
    # valid shapes this build does not run
    assert moe.moe_check_problem(moe.Problem.make(T=4, H=100, I=128, E=8, K=2, M_max=4)) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_check_problem(
        moe.Problem.make(T=4, H=128, I=128, E=8, K=2, M_max=4, act="f32", wt="bf16", out="f32")) == \
        moe.MOE_ERR_UNSUPPORTED


def test_null_pointers_rejected_before_launch():
    L = moe.lib()
    p = moe.Problem.make(T=4, H=128, I=128, E=8, K=2, M_max=4)
    r = L.moe_route_topk(ctypes.byref(p), None, None, None, None)
    assert r == moe.MOE_ERR_INVALID
    r = L.moe_combine(ctypes.byref(p), None, None, None, None, None)
    assert r == moe.MOE_ERR_INVALID
    r = L.moe_permute(ctypes.byref(p), *([None] * 11), 0, None)
    assert r == moe.MOE_ERR_INVALID
    r = L.moe_grouped_swiglu_gemm(ctypes.byref(p), *([None] * 10), 0, None)
    assert r == moe.MOE_ERR_INVALID
    r = L.moe_grouped_down_gemm(ctypes.byref(p), *([None] * 9), 0, None)
    assert r == moe.MOE_ERR_INVALID
    # empty batch: nothing to route
    p0 = moe.Problem.make(T=0, H=128, I=128, E=8, K=2, M_max=4)
    assert L.moe_route_topk(ctypes.byref(p0), None, None, None, None) == moe.MOE_OK


def test_workspace_too_small_rejected():
    L = moe.lib()
    p = moe.Problem.make(T=4, H=128, I=128, E=8, K=2, M_max=4)
    fake = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    r = L.moe_permute(ctypes.byref(p), fake, fake, None, fake, fake, fake, fake, fake, None, fake, fake, 1, None)
    assert r == moe.MOE_ERR_WORKSPACE


def test_host_eplb_invert_matches_oracle():
    rng = np.random.default_rng(0)
    for _ in range(50):
        E = int(rng.integers(1, 9))
        P = E + int(rng.integers(0, 5))
        p2l = np.concatenate([np.arange(E), rng.integers(0, E, P - E)]).astype(np.int32)
        rng.shuffle(p2l)
        l2p, rc, r = moe.moe_eplb_invert(p2l, E, P)
        ol2p, orc, oref = oracle.eplb_invert(p2l, E, P)
        assert r == oref and (rc == orc).all() and (l2p[:, :r] == ol2p[:, :r]).all()
    with pytest.raises(moe.MoeError):
        moe.moe_eplb_invert([0, 5], 2, 2)


def documented_scratch_bytes(T, K, E, P):
    """The dispatch scratch as the header states it: bitmask (+4), word prefixes, the slot of
    each record, the compact replica list, starts and counts, each rounded up to 256 bytes."""
    W = (T + 31) // 32
    up = lambda b: (b + 255) // 256 * 256
    return up(4 * P * W + 4) + up(4 * P * W) + up(4 * T * K) + up(4 * P) + up(4 * E) + up(4 * E)


@pytest.mark.parametrize("T,K,E,P", [(8192, 10, 512, 512), (256, 8, 256, 288), (1100, 4, 64, 72), (1, 1, 8, 8),
                                     (4096, 4, 64, 64)])
def test_documented_scratch_formula_matches_library(T, K, E, P):
    # fp32 problems: the GEMMs need no workspace, so moe_workspace_bytes is the dispatch's scratch alone
    p = moe.Problem.make(T=T, H=128, I=128, E=E, K=K, P=P, layout="contig", act="f32", wt="f32", out="f32")
    assert moe.moe_check_problem(p) == moe.MOE_OK
    assert moe.moe_workspace_bytes(p) == documented_scratch_bytes(T, K, E, P)


def test_no_workspace_call_rejects_beyond_four_mib_without_gpu():
    # the size check comes before any device call; the stated prefill figure is ~1.3 MiB
    assert abs(documented_scratch_bytes(8192, 10, 512, 512) / 2**20 - 1.3) < 0.05
    L = moe.lib()
    fake = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    T = 32
    while documented_scratch_bytes(T, 8, 1024, 1024) <= (4 << 20):
        T += 32
    p = moe.Problem.make(T=T, H=128, I=128, E=1024, K=8, layout="contig", act="f32", wt="f32", out="f32")
    r = L.moe_permute_no_workspace(ctypes.byref(p), fake, fake, None, fake, fake, fake, fake, fake, None, fake, None)
    assert r == moe.MOE_ERR_WORKSPACE


def documented_tile_rows(T, H, K, P, wt, step):
    """The header's rule for moe_gemm_tile_rows: 0 for fp32 experts (CUDA-core GEMM); for FP8 / FP4
    experts 256 with at least 128 rows per slot on average (T * K / P; for step 4 only when H is
    a multiple of 256), else 64; 128 for bf16 experts."""
    if wt == "f32":
        return 0
    if wt in ("e4m3", "e2m1"):
        return 256 if T * K / P >= 128 and (step == 3 or H % 256 == 0) else 64
    return 128


@pytest.mark.parametrize("T,H,I,E,K,P,S,wt,act,layout", [
    (8192, 4096, 1024, 512, 10, 512, 0, "e4m3", "bf16", "contig"),    # prefill: SM pairs for both GEMMs
    (8192, 4224, 1024, 512, 10, 512, 0, "e4m3", "bf16", "contig"),    # H not a multiple of 256: down on one CTA (64)
    (1024, 2048, 1024, 8, 1, 8, 0, "e2m1", "bf16", "contig"),         # exactly 128 rows per slot, FP4
    (1016, 2048, 1024, 8, 1, 8, 0, "e2m1", "bf16", "contig"),         # just below
    (128, 7168, 2048, 256, 8, 256, 1, "e4m3", "bf16", "masked"),      # DeepSeek-V3-shaped decode
    (32, 4096, 14336, 8, 2, 8, 0, "bf16", "bf16", "masked"),          # Mixtral-shaped decode (bf16)
    (8192, 4096, 1024, 64, 2, 64, 0, "bf16", "bf16", "contig"),       # bf16 prefill-sized: no pairs
    (16, 64, 128, 8, 2, 8, 0, "f32", "f32", "masked"),                # fp32: CUDA cores
])
def test_gemm_tile_rows_follow_the_header_rule(T, H, I, E, K, P, S, wt, act, layout):
    out = "f32" if wt == "f32" else "bf16"
    p = moe.Problem.make(T=T, H=H, I=I, E=E, K=K, P=P, M_max=T if layout == "masked" else 0, has_shared=S,
                         act=act, wt=wt, out=out, layout=layout)
    assert moe.moe_check_problem(p) == moe.MOE_OK
    for step in (3, 4):
        assert moe.moe_gemm_tile_rows(p, step) == documented_tile_rows(T, H, K, P, wt, step), step
    assert moe.moe_gemm_tile_rows(p, 5) == 0  # only steps 3 and 4 have a GEMM tile
