"""moe_permute_no_workspace against the oracle and against moe_permute.

The no-workspace call exists for callers that cannot allocate device memory
where they run the layer: an inference-engine plugin that must not allocate
inside its enqueue step, code running while its stream is captured into a
CUDA graph (cudaMalloc cannot be recorded by a capture), or a framework whose
device memory is all owned by its own pool.  Its scratch is a fixed array
inside the library instead of a caller workspace, and it must write exactly
what moe_permute writes.

Only batches above 4096 records (or above 256 with a replica map and a large
slot bitmask) take the multi-kernel dispatch that uses scratch memory (slot
bitmask, word prefixes, each record's slot, the replica tables); the cases
here are of that size.  They run back to back, a larger problem between two
smaller ones, so that bitmask words or prefixes left in the shared array by
the previous call would show up in the next one.

This file is collected last, so a run that stops at the first failure has run
every other test first.  It needs nothing from the other tests and passes on
its own in a fresh process."""
import numpy as np
import pytest
import torch

import oracle
import routed_expert_layer_moe_gb300 as moe
from cases import SMALL
from gpu_util import Workload, to_dev, to_host

pytestmark = pytest.mark.gpu

SENT_I32 = -7


@pytest.fixture(scope="module", autouse=True)
def built():
    from routed_expert_layer_moe_gb300 import build
    build.build()


def case(name):
    """Workloads that take the scratch-using dispatch (each above 4096 records)."""
    if name == "map_1100":  # 4400 records with a replica map: tables, mark, one-CTA scan, scatter
        b = SMALL["e4m3_eplb_zipf"]
        return b.replace(name=name, T=1100, H=256, I=128, E=64, K=4, M_max=1100, redundant=8)
    if name == "contig_4096":  # 16384 records, 64 slots x 128 bitmask words: the many-CTA slot scan
        b = SMALL["e4m3_contig"]
        return b.replace(name=name, T=4096, H=256, I=128, E=64, K=4)
    if name == "bf16_shared_1500":  # 6000 records, bf16 copies, a shared expert, masked rows
        b = SMALL["e4m3_masked_shared"]
        return b.replace(name=name, T=1500, H=256, I=128, E=48, K=4, M_max=1500, gemm="bf16")
    raise KeyError(name)


def outputs(L):
    """Fresh output buffers of a layer's dispatch, filled with sentinels."""
    p = L.p
    rows = L.rows
    dev = L.ids.device
    i32 = dict(dtype=torch.int32, device=dev)
    f8 = L.wt in ("e4m3", "e2m1")
    return dict(masked_m=torch.full((p.P + p.has_shared,), SENT_I32, **i32),
                offsets=torch.full((p.P + p.has_shared + 1,), SENT_I32, **i32),
                row_of=torch.full((p.T, p.K + p.has_shared), SENT_I32, **i32),
                src_of=torch.full((rows,), SENT_I32, **i32),
                xg=torch.full((rows, p.H), 0x5A, dtype=torch.uint8, device=dev) if f8
                else torch.full((rows, p.H), -3.0, dtype=L.xg.dtype, device=dev),
                xg_s=torch.full((rows, p.H // 128), -3.0, dtype=torch.float32, device=dev) if f8 else None,
                err=torch.zeros(1, **i32))


def with_workspace(L, x):
    o = outputs(L)
    moe.moe_permute(L.p, L.ids, x, L.p2l, o["masked_m"], o["offsets"], o["row_of"], o["src_of"], o["xg"], o["xg_s"],
                    o["err"], L.ws)
    return o


def without_workspace(L, x):
    o = outputs(L)
    moe.moe_permute_no_workspace(L.p, L.ids, x, L.p2l, o["masked_m"], o["offsets"], o["row_of"], o["src_of"],
                                 o["xg"], o["xg_s"], o["err"])
    return o


def check_against_oracle(wl, got):
    """Counts, offsets, row maps and dispatched rows equal the oracle's, bit for bit;
    padding rows keep their sentinels."""
    cfg = wl.cfg
    lay = oracle.layout(cfg, wl.ids, wl.p2l)
    assert lay["status"] == 0
    assert int(to_host(got["err"])[0]) == 0
    assert (to_host(got["masked_m"]) == lay["masked_m"]).all()
    assert (to_host(got["offsets"]) == lay["offsets"]).all()
    assert (to_host(got["row_of"]) == lay["row_of"]).all()
    valid = lay["src_of"] >= 0
    src = to_host(got["src_of"])
    assert (src[valid] == lay["src_of"][valid]).all()
    assert (src[~valid] == SENT_I32).all()
    xg, xgs = oracle.dispatch_values(cfg, wl.x, lay["row_of"])
    gx = to_host(got["xg"])
    assert (gx[valid] == xg[valid]).all()
    if cfg.gemm == "e4m3":
        assert (to_host(got["xg_s"])[valid] == xgs[valid]).all()
        assert (gx[~valid] == 0x5A).all()


def test_no_workspace_matches_oracle_and_workspace_call_back_to_back():
    # The largest problem runs between two smaller ones, and each problem runs twice in a
    # row: every call finds the previous call's bitmask, prefixes and slots still in the
    # library's scratch array and must not depend on them.
    loaded = {}
    for name in ("map_1100", "map_1100", "contig_4096", "bf16_shared_1500", "map_1100", "contig_4096"):
        if name not in loaded:
            wl = Workload(case(name))
            L = wl.layer()
            L.ids.copy_(torch.from_numpy(np.ascontiguousarray(wl.ids, np.int32)))
            loaded[name] = (wl, L, to_dev(wl.x))
        wl, L, x = loaded[name]
        got = without_workspace(L, x)
        ref = with_workspace(L, x)
        torch.cuda.synchronize()
        check_against_oracle(wl, got)
        for key in ref:  # the same bytes as the call with a caller workspace
            if ref[key] is None:
                assert got[key] is None
                continue
            assert (to_host(got[key]) == to_host(ref[key])).all(), (name, key)


def test_no_workspace_decode_batch():
    # a decode-sized batch (one-CTA layout, no scratch) through the same entry point
    wl = Workload(SMALL["e4m3_eplb_zipf"])
    L = wl.layer()
    L.ids.copy_(torch.from_numpy(np.ascontiguousarray(wl.ids, np.int32)))
    got = without_workspace(L, to_dev(wl.x))
    torch.cuda.synchronize()
    check_against_oracle(wl, got)


def test_no_workspace_rejects_problems_beyond_its_scratch():
    # 8*P*ceil(T/32) bytes alone exceed the 4 MiB array for this batch
    p = moe.Problem.make(T=65536, H=4096, I=1024, E=1024, K=8, layout="contig", act="bf16", wt="e4m3", out="bf16")
    fake = torch.empty(16, dtype=torch.int32, device="cuda")  # never read: the size check comes first
    with pytest.raises(moe.MoeError) as e:
        moe.moe_permute_no_workspace(p, fake, fake, None, fake, fake, fake, fake, fake, fake, fake)
    assert e.value.status == moe.MOE_ERR_WORKSPACE
