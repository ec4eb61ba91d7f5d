"""moe_permute_no_workspace against moe_permute.

The no-workspace call exists for callers that cannot allocate device memory
where they run the layer: an inference-engine plugin that must not allocate
inside its enqueue step, code running while its stream is captured into a
CUDA graph (cudaMalloc cannot be recorded by a capture), or a framework whose
device memory is all owned by its own pool.  Its scratch is a fixed array
inside the library instead of a caller workspace, and it must write exactly
what moe_permute writes.

This file is collected last, so a run that stops at the first failure has run
every other test first.  It needs nothing from the other tests and passes on
its own in a fresh process."""
import numpy as np
import pytest
import torch

import routed_expert_layer_moe_gb300 as moe
from cases import SMALL
from gpu_util import Workload, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from routed_expert_layer_moe_gb300 import build
    build.build()


def outputs(L, xg_bytes_fill=0x5A):
    """Fresh output buffers of a layer's dispatch, filled with sentinels."""
    p = L.p
    rows = L.rows
    dev = L.ids.device
    i32 = dict(dtype=torch.int32, device=dev)
    o = dict(masked_m=torch.full((p.P + p.has_shared,), -7, **i32),
             offsets=torch.full((p.P + p.has_shared + 1,), -7, **i32),
             row_of=torch.full((p.T, p.K + p.has_shared), -7, **i32),
             src_of=torch.full((rows,), -7, **i32),
             xg=torch.full((rows, p.H), xg_bytes_fill, dtype=torch.uint8, device=dev) if L.wt in ("e4m3", "e2m1")
             else torch.full((rows, p.H), -3.0, dtype=L.xg.dtype, device=dev),
             xg_s=torch.full((rows, p.H // 128), -3.0, dtype=torch.float32, device=dev) if L.wt in ("e4m3", "e2m1") else None,
             err=torch.zeros(1, **i32))
    return o


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


def test_no_workspace_matches_workspace_call_twice_in_a_row():
    # Two different problems back to back: the second call finds the first
    # call's data still in the library's scratch array and must not depend on it.
    for name in ("e4m3_eplb_zipf", "bf16_masked", "e4m3_eplb_zipf"):
        wl = Workload(SMALL[name])
        L = wl.layer()
        L.ids.copy_(torch.from_numpy(np.ascontiguousarray(wl.ids, np.int32)))
        x = to_dev(wl.x)
        ref = with_workspace(L, x)
        got = without_workspace(L, x)
        torch.cuda.synchronize()
        for key in ref:
            if ref[key] is None:
                assert got[key] is None
                continue
            assert (to_host(got[key]) == to_host(ref[key])).all(), (name, key)  # integers and bytes: bit-exact
        assert int(to_host(got["err"])[0]) == 0


def test_no_workspace_rejects_problems_beyond_its_scratch():
    # 8*P*ceil(T/32) bytes alone exceed the 4 MiB array for this batch
    p = moe.Problem.make(T=65536, H=4096, I=1024, E=1024, K=8, layout="contig", act="bf16", wt="e4m3", out="bf16")
    fake = torch.empty(16, dtype=torch.int32, device="cuda")  # never read: the size check comes first
    with pytest.raises(moe.MoeError) as e:
        moe.moe_permute_no_workspace(p, fake, fake, None, fake, fake, fake, fake, fake, fake, fake)
    assert e.value.status == moe.MOE_ERR_WORKSPACE
