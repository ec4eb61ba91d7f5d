"""Each C-ABI call on the GPU against the fp64 oracle, on the reduced workloads.

Integer outputs (ids, counts, offsets, row maps, quantised activations) must be
bit-exact; values within max|err|/max|ref| of 1e-2 (bf16), 3e-2 (e4m3) or 1e-4
(fp32).  Inputs of each call come from the generator or the oracle, never from
another GPU call."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import routed_expert_layer_moe_gb300 as moe
from cases import SMALL
from gpu_util import TOL, Workload, real, rel_err, to_dev, to_host

pytestmark = pytest.mark.gpu

NAMES = list(SMALL)
SENT_I32 = -7


@pytest.fixture(scope="module", autouse=True)
def built():
    from routed_expert_layer_moe_gb300 import build
    build.build()
    torch.cuda.init()


@pytest.fixture(scope="module")
def workloads():
    return {n: Workload(SMALL[n]) for n in NAMES}


def oracle_layout(wl):
    lay = oracle.layout(wl.cfg, wl.ids, wl.p2l)
    assert lay["status"] == 0
    return lay


# ---- a1 route -----------------------------------------------------------------

@pytest.mark.parametrize("name", NAMES)
def test_route(workloads, name):
    wl = workloads[name]
    L = wl.layer()
    L.route(to_dev(wl.logits))
    torch.cuda.synchronize()
    assert (to_host(L.ids) == wl.ids).all()
    np.testing.assert_allclose(to_host(L.w), wl.w, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("T,E,K", [(1, 8, 2), (37, 512, 10), (5, 256, 8), (64, 1024, 32), (3, 33, 32),
                                   (300, 128, 4), (7, 97, 32), (9, 96, 3),
                                   (2048, 512, 10), (2100, 128, 32), (2050, 97, 1), (2048, 96, 8)])
def test_route_shapes_and_ties(T, E, K):
    cfg = SMALL["tiny"].replace(T=T, E=E, K=K, M_max=T)
    logits = mi.normal(1, 77, (T, E), dtype="f32")
    logits[0, :] = 0.5                      # a token whose logits all tie
    if T > 2:
        logits[2, ::3] = logits[2, 1]       # many exact ties in another
    if T > 1:
        logits[1, ::max(1, E // 40)] = logits[1].max() + 1.0  # about 40 tied at the top
    ids, w = oracle.route(logits, K)
    p = moe.Problem.make(T=T, H=64, I=128, E=E, K=K, M_max=T, act="f32", wt="f32", out="f32")
    gids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    gw = torch.empty((T, K), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(p, to_dev(logits), gids, gw)
    torch.cuda.synchronize()
    assert (to_host(gids) == ids).all()
    np.testing.assert_allclose(to_host(gw), w, rtol=2e-6, atol=1e-7)


# ---- a2 permute -----------------------------------------------------------------

def run_permute(wl, ids=None):
    L = wl.layer()
    ids = wl.ids if ids is None else ids
    L.ids.copy_(torch.from_numpy(np.ascontiguousarray(ids, np.int32)))
    for t in (L.masked_m, L.offsets, L.row_of, L.src_of):
        t.fill_(SENT_I32)
    if L.xg.dtype == torch.uint8:
        L.xg.fill_(0x5A)
        L.xg_s.fill_(-3.0)
    else:
        L.xg.fill_(-3.0)
    L.err.zero_()
    L.permute(to_dev(wl.x))
    torch.cuda.synchronize()
    return L


@pytest.mark.parametrize("name", NAMES)
def test_permute(workloads, name):
    wl = workloads[name]
    cfg = wl.cfg
    L = run_permute(wl)
    lay = oracle_layout(wl)
    assert int(to_host(L.err)[0]) == 0
    assert (to_host(L.masked_m) == lay["masked_m"]).all()
    assert (to_host(L.offsets) == lay["offsets"]).all()
    assert (to_host(L.row_of) == lay["row_of"]).all()
    valid = lay["src_of"] >= 0
    src = to_host(L.src_of)
    assert (src[valid] == lay["src_of"][valid]).all()
    assert (src[~valid] == SENT_I32).all()  # padding rows untouched
    xg, xgs = oracle.dispatch_values(cfg, wl.x, lay["row_of"])
    gx = to_host(L.xg)
    assert (gx[valid] == xg[valid]).all()  # copies and e4m3 codes bit-exact
    if cfg.gemm == "e4m3":
        assert (to_host(L.xg_s)[valid] == xgs[valid]).all()
        assert (gx[~valid] == 0x5A).all()
    else:
        assert (real(gx[~valid], cfg.gemm) == -3.0).all()


@pytest.mark.parametrize("base,shared", [("e4m3_contig", 0), ("e4m3_masked_shared", 1), ("bf16_masked", 0)])
def test_permute_large_bitmask(base, shared):
    """A batch whose slot bitmask has >= 8192 words (4096 tokens x 64 slots) takes the
    many-CTA slot scan; counts, offsets, row maps and the dispatched rows (copies, e4m3 codes
    and their scales) stay bit-exact, padding rows untouched."""
    cfg = SMALL[base].replace(T=4096, H=256, I=128, E=64, K=4, shared=shared,
                              M_max=(4096 if SMALL[base].layout == "masked" else 0))
    wl = Workload(cfg)
    L = run_permute(wl)
    lay = oracle_layout(wl)
    assert int(to_host(L.err)[0]) == 0
    check_layout(L, wl, lay)


def check_layout(L, wl, lay, values=True):
    cfg = wl.cfg
    assert (to_host(L.masked_m) == lay["masked_m"]).all()
    assert (to_host(L.offsets) == lay["offsets"]).all()
    assert (to_host(L.row_of) == lay["row_of"]).all()
    valid = lay["src_of"] >= 0
    src = to_host(L.src_of)
    assert (src[valid] == lay["src_of"][valid]).all()
    assert (src[~valid] == SENT_I32).all()
    if values:
        xg, xgs = oracle.dispatch_values(cfg, wl.x, lay["row_of"])
        gx = to_host(L.xg)
        assert (gx[valid] == xg[valid]).all()
        if cfg.gemm == "e4m3":
            assert (to_host(L.xg_s)[valid] == xgs[valid]).all()
            assert (gx[~valid] == 0x5A).all()  # padding rows untouched
        else:
            assert (real(gx[~valid], cfg.gemm) == -3.0).all()


# T*K = 256: the largest batch of the one-launch permute (without a map); 4096: the largest of
# the one-CTA layout + copy; 4100: the mark / scan / scatter sequence (single-CTA scan: 64
# slots x 33 words)
@pytest.mark.parametrize("T", [64, 1024, 1025])
@pytest.mark.parametrize("base", ["e4m3_eplb_zipf", "e4m3_masked_shared", "bf16_masked", "e4m3_contig"])
def test_permute_both_paths(base, T):
    """Each permute path gives the oracle's layout and dispatched values, with and without a
    replica map and a shared expert."""
    b = SMALL[base]
    E = 64
    cfg = b.replace(T=T, H=256, I=128, E=E, K=4,
                    M_max=(T if b.layout == "masked" else 0),
                    redundant=(8 if b.redundant else 0))
    wl = Workload(cfg)
    L = run_permute(wl)
    lay = oracle_layout(wl)
    assert int(to_host(L.err)[0]) == 0
    check_layout(L, wl, lay)


@pytest.mark.parametrize("T", [40, 300, 1100])
def test_permute_duplicate_expert(T):
    """A token that names one expert twice: the record with the larger k is not placed
    (row -1, MOE_FLAG_BAD_EXPERT) and the counts leave it out; every other record is placed
    as the oracle places the batch without it."""
    cfg = SMALL["e4m3_masked_shared"].replace(T=T, M_max=T)
    wl = Workload(cfg)
    ids = wl.ids.copy()
    ids[3, 2] = ids[3, 0]
    L = run_permute(wl, ids)
    assert int(to_host(L.err)[0]) & moe.MOE_FLAG_BAD_EXPERT
    ro = to_host(L.row_of)
    assert ro[3, 2] == -1 and ro[3, 0] >= 0
    # expected rows by brute force: in each slot the placed records in ascending token order
    placed = np.ones(ids.shape, bool)
    placed[3, 2] = False
    want = np.full(ids.shape, -1, np.int64)
    fill = np.zeros(cfg.E, np.int64)
    for t in range(T):
        for k in range(cfg.K):
            if placed[t, k]:
                e = ids[t, k]
                want[t, k] = e * cfg.M_max + fill[e]
                fill[e] += 1
    assert (ro[:, :cfg.K] == want).all()
    assert (ro[:, cfg.K] == cfg.E * cfg.M_max + np.arange(T)).all()  # the shared expert's rows
    mm = to_host(L.masked_m)
    assert (mm[:cfg.E] == fill).all() and mm[cfg.E] == T


@pytest.mark.parametrize("T", [40, 2100])
def test_permute_pages_replica_map(T):
    """The EPLB page's example map [0, 1, 2, 3, 0, 1] (experts 0 and 1 in two slots each):
    records go round-robin by token index to the replicas, as the oracle places them."""
    cfg = SMALL["bf16_masked"].replace(T=T, E=4, K=2, M_max=T, redundant=2)
    wl = Workload(cfg)
    p2l = np.array([0, 1, 2, 3, 0, 1], np.int32)
    L = wl.layer()
    L.p2l = torch.from_numpy(p2l).cuda()
    L.ids.copy_(torch.from_numpy(np.ascontiguousarray(wl.ids, np.int32)))
    for t in (L.masked_m, L.offsets, L.row_of, L.src_of):
        t.fill_(SENT_I32)
    L.err.zero_()
    L.permute(to_dev(wl.x))
    torch.cuda.synchronize()
    lay = oracle.layout(cfg, wl.ids, p2l)
    assert lay["status"] == 0 and int(to_host(L.err)[0]) == 0
    assert (to_host(L.masked_m) == lay["masked_m"]).all()
    assert (to_host(L.row_of) == lay["row_of"]).all()
    assert to_host(L.masked_m)[4] > 0 and to_host(L.masked_m)[5] > 0  # the replicas take rows


@pytest.mark.parametrize("T", [40, 1100])
def test_permute_bad_replica_map(T):
    """A physical_to_logical map in which expert 0 has no slot and expert 1 has more than
    P-E+1: MOE_FLAG_BAD_MAP, the records of both experts are not placed, the rest are."""
    cfg = SMALL["e4m3_eplb_zipf"].replace(T=T, M_max=T)
    wl = Workload(cfg)
    P, E = cfg.P, cfg.E
    p2l = np.concatenate([np.arange(E), np.ones(P - E, np.int32)]).astype(np.int32)
    p2l[0] = 1  # expert 0 held by no slot; expert 1 by P-E+2 slots
    L = wl.layer()
    L.p2l = torch.from_numpy(p2l).cuda()
    L.ids.copy_(torch.from_numpy(np.ascontiguousarray(wl.ids, np.int32)))
    for t in (L.masked_m, L.offsets, L.row_of, L.src_of):
        t.fill_(SENT_I32)
    L.err.zero_()
    L.permute(to_dev(wl.x))
    torch.cuda.synchronize()
    assert int(to_host(L.err)[0]) & moe.MOE_FLAG_BAD_MAP
    ro = to_host(L.row_of)[:, :cfg.K]
    bad = (wl.ids == 0) | (wl.ids == 1)
    assert (ro[bad] == -1).all() and (ro[~bad] >= 0).all()
    mm = to_host(L.masked_m)
    assert mm[:P].sum() == (~bad).sum()


def test_permute_empty_and_one_hot():
    cfg = SMALL["e4m3_masked_shared"]
    wl = Workload(cfg)
    # every token on experts 0..K-1: the other slots stay empty
    ids = np.tile(np.arange(cfg.K, dtype=np.int32), (cfg.T, 1))
    L = run_permute(wl, ids)
    mm = to_host(L.masked_m)
    assert (mm[:cfg.K] == cfg.T).all() and (mm[cfg.K:cfg.P] == 0).all() and mm[cfg.P] == cfg.T
    lay = oracle.layout(cfg, ids, None)
    assert (to_host(L.row_of) == lay["row_of"]).all()


def test_permute_overflow_sets_flag_without_stray_writes():
    cfg = SMALL["bf16_masked"].replace(M_max=5)
    wl = Workload(cfg)
    L = run_permute(wl)
    lay = oracle.layout(cfg, wl.ids, None)
    assert lay["status"] == -2
    assert int(to_host(L.err)[0]) & moe.MOE_FLAG_OVERFLOW
    assert (to_host(L.masked_m) == lay["masked_m"]).all()  # true counts are reported
    ro = to_host(L.row_of)
    ranks_ok = lay["row_of"] % cfg.M_max < cfg.M_max
    # records past M_max are not placed
    for t in range(cfg.T):
        for k in range(cfg.K):
            s = wl.ids[t, k]
            rank = (lay["row_of"][t, k] - s * cfg.M_max)
            assert ro[t, k] == (lay["row_of"][t, k] if rank < cfg.M_max else -1)
    assert ranks_ok.all()


def test_permute_bad_ids_flagged():
    cfg = SMALL["bf16_masked"]
    wl = Workload(cfg)
    ids = wl.ids.copy()
    ids[3, 0] = cfg.E + 4
    L = run_permute(wl, ids)
    assert int(to_host(L.err)[0]) & moe.MOE_FLAG_BAD_EXPERT
    assert to_host(L.row_of)[3, 0] == -1


# ---- a3 / a4 grouped GEMMs -------------------------------------------------------------

def gemm_inputs(wl):
    cfg = wl.cfg
    lay = oracle_layout(wl)
    xg, xgs = oracle.dispatch_values(cfg, wl.x, lay["row_of"])
    o = wl.order
    w13, w2 = wl.w13[o], wl.w2[o]
    w13s = None if wl.w13_s is None else wl.w13_s[o]
    w2s = None if wl.w2_s is None else wl.w2_s[o]
    return lay, xg, xgs, w13, w13s, w2, w2s


@pytest.mark.parametrize("name", NAMES)
def test_grouped_swiglu(workloads, name):
    check_grouped_swiglu(workloads[name])


def check_grouped_swiglu(wl):
    cfg = wl.cfg
    lay, xg, xgs, w13, w13s, w2, w2s = gemm_inputs(wl)
    hg_ref, hgs_ref = oracle.grouped_swiglu(cfg, xg, xgs, w13, w13s, lay["masked_m"], lay["offsets"])
    L = wl.layer()
    L.xg.copy_(to_dev(xg))
    if xgs is not None:
        L.xg_s.copy_(to_dev(xgs))
    L.masked_m.copy_(to_dev(lay["masked_m"]))
    L.offsets.copy_(to_dev(lay["offsets"]))
    if L.hg.dtype == torch.uint8:
        L.hg.fill_(0x5A)
    else:
        L.hg.fill_(-3.0)
    L.swiglu()
    torch.cuda.synchronize()
    assert int(to_host(L.err)[0]) == 0
    valid = lay["src_of"] >= 0
    got = real(to_host(L.hg)[valid], cfg.gemm, None if hgs_ref is None else to_host(L.hg_s)[valid])
    ref = real(hg_ref[valid], cfg.gemm, None if hgs_ref is None else hgs_ref[valid])
    assert rel_err(got, ref) <= TOL[cfg.gemm]
    pad = to_host(L.hg)[~valid]
    assert (pad == 0x5A).all() if cfg.gemm == "e4m3" else (real(pad, cfg.gemm) == -3.0).all()


@pytest.mark.parametrize("name", NAMES)
def test_grouped_down(workloads, name):
    check_grouped_down(workloads[name])


def check_grouped_down(wl):
    cfg = wl.cfg
    lay, xg, xgs, w13, w13s, w2, w2s = gemm_inputs(wl)
    hg, hgs = oracle.grouped_swiglu(cfg, xg, xgs, w13, w13s, lay["masked_m"], lay["offsets"])
    yg_ref = oracle.grouped_down(cfg, hg, hgs, w2, w2s, lay["masked_m"], lay["offsets"])
    L = wl.layer()
    L.hg.copy_(to_dev(hg))
    if hgs is not None:
        L.hg_s.copy_(to_dev(hgs))
    L.masked_m.copy_(to_dev(lay["masked_m"]))
    L.offsets.copy_(to_dev(lay["offsets"]))
    L.yg.fill_(-3.0)
    L.down()
    torch.cuda.synchronize()
    assert int(to_host(L.err)[0]) == 0
    valid = lay["src_of"] >= 0
    got = real(to_host(L.yg)[valid], cfg.y_dtype)
    ref = real(yg_ref[valid], cfg.y_dtype)
    assert rel_err(got, ref) <= TOL[cfg.gemm]
    assert (real(to_host(L.yg)[~valid], cfg.y_dtype) == -3.0).all()


@pytest.mark.parametrize("name", NAMES)
def test_grouped_ffn_one_launch(workloads, name):
    """moe_grouped_ffn: gate/up and down in one launch.  yg within tolerance of the oracle's
    two steps; hg, its scales and yg bit-identical to the two separate calls; padding rows
    untouched."""
    wl = workloads[name]
    cfg = wl.cfg
    lay, xg, xgs, w13, w13s, w2, w2s = gemm_inputs(wl)
    hg_ref, hgs_ref = oracle.grouped_swiglu(cfg, xg, xgs, w13, w13s, lay["masked_m"], lay["offsets"])
    yg_ref = oracle.grouped_down(cfg, hg_ref, hgs_ref, w2, w2s, lay["masked_m"], lay["offsets"])

    def run(fused):
        L = wl.layer()
        L.xg.copy_(to_dev(xg))
        if xgs is not None:
            L.xg_s.copy_(to_dev(xgs))
        L.masked_m.copy_(to_dev(lay["masked_m"]))
        L.offsets.copy_(to_dev(lay["offsets"]))
        L.yg.fill_(-3.0)
        if fused:
            L.ffn()
        else:
            L.swiglu()
            L.down()
        torch.cuda.synchronize()
        assert int(to_host(L.err)[0]) == 0
        return to_host(L.hg), None if L.hg_s is None else to_host(L.hg_s), to_host(L.yg)

    hs, hss, ys = run(False)
    hf, hfs, yf = run(True)
    valid = lay["src_of"] >= 0
    assert (hf[valid] == hs[valid]).all()
    if hss is not None:
        assert (hfs[valid] == hss[valid]).all()
    assert (yf[valid] == ys[valid]).all()
    assert (real(yf[~valid], cfg.y_dtype) == -3.0).all()
    assert rel_err(real(yf[valid], cfg.y_dtype), real(yg_ref[valid], cfg.y_dtype)) <= TOL[cfg.gemm]


def routing_with_counts(counts, T, K):
    """ids [T, K] in which expert e is chosen by exactly counts[e] distinct tokens (sum(counts) =
    T * K, every count <= T): the experts, largest count first, take consecutive runs of tokens
    cyclically, so each token gets K distinct experts."""
    assert sum(counts) == T * K and max(counts) <= T
    per_token = [[] for _ in range(T)]
    ptr = 0
    for e in sorted(range(len(counts)), key=lambda e: -counts[e]):
        for i in range(counts[e]):
            per_token[(ptr + i) % T].append(e)
        ptr += counts[e]
    ids = np.array(per_token, np.int32)
    assert ids.shape == (T, K) and all(len(set(r)) == K for r in per_token)
    return ids


# slot row counts on both sides of every token box (16 / 32 / 64 rows) and of the splits of a slot
# into two and three chunks (above 64 and 128 rows), plus an empty slot
EDGE_COUNTS = [0, 1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 47]


@pytest.mark.parametrize("wq", ["e4m3", "e2m1"])
def test_grouped_gemms_at_token_box_edges(wq):
    """FP8 / FP4 decode-shaped GEMMs (token-major, one CTA per SM: chunks of at most 64 rows,
    M = 64 MMAs) on a layout whose slots hold 0, 1, 15-17, 31-33, 63-65 and 127-129 rows (and a
    shared expert with every token): the token box of each chunk is the smallest of 16 / 32 / 64
    rows covering it, the MMA reads stale shared memory past the box, and slots above 64 rows
    split into two or three chunks.  Values within tolerance of the oracle, padding rows
    untouched, token tiles = sum over slots of ceil(rows / 64)."""
    T, K = 192, 4
    base = SMALL["e4m3_masked_shared"] if wq == "e4m3" else SMALL["e2m1_masked_shared"]
    cfg = base.replace(name="edges_" + wq, T=T, K=K, E=len(EDGE_COUNTS), M_max=T)
    wl = Workload(cfg)
    wl.ids = routing_with_counts(EDGE_COUNTS, T, K)
    lay = oracle_layout(wl)
    assert list(lay["masked_m"][:len(EDGE_COUNTS)]) == EDGE_COUNTS
    check_grouped_swiglu(wl)
    check_grouped_down(wl)
    L = wl.layer()
    assert moe.moe_gemm_tile_rows(L.p, 3) == 64 and moe.moe_gemm_tile_rows(L.p, 4) == 64
    lay, xg, xgs, w13, w13s, w2, w2s = gemm_inputs(wl)
    L.xg.copy_(to_dev(xg))
    L.xg_s.copy_(to_dev(xgs))
    L.masked_m.copy_(to_dev(lay["masked_m"]))
    L.offsets.copy_(to_dev(lay["offsets"]))
    L.swiglu()
    torch.cuda.synchronize()
    c = L.ws[:moe.MOE_STATS_BYTES].view(torch.int32).cpu().numpy().reshape(2, moe.MOE_STATS_CTAS, 2).sum(axis=1)
    want = sum(-(-m // 64) for m in EDGE_COUNTS) + -(-T // 64)  # the shared slot holds all T rows
    assert c[0, 1] == oracle.token_tiles(lay["masked_m"], 64) == want


@pytest.mark.parametrize("name", [n for n in NAMES if SMALL[n].gemm != "f32"])
def test_gemm_issue_counters(workloads, name):
    """The GEMMs' token tiles (summed over CTAs from the counters in the workspace) equal the
    oracle's sum over slots of ceil(masked_m / BM), BM the GEMM's tile height (64 for FP8 / FP4
    on one CTA, 128 for bf16, 256 on SM pairs): no tile for padding rows or empty slots; every
    unit belongs to one such tile (units = tiles x tile pairs x K splits).  The one-launch FFN
    runs on single CTAs: 64-row tiles for FP8 / FP4, 128 for bf16."""
    wl = workloads[name]
    cfg = wl.cfg
    lay, xg, xgs, w13, w13s, w2, w2s = gemm_inputs(wl)
    L = wl.layer()
    bm = {3: moe.moe_gemm_tile_rows(L.p, 3), 4: moe.moe_gemm_tile_rows(L.p, 4)}
    assert bm[3] in (64, 128, 256) and bm[4] in (64, 128, 256)
    want = oracle.token_tiles(lay["masked_m"], 64 if bm[3] == 256 else bm[3])
    L.xg.copy_(to_dev(xg))
    if xgs is not None:
        L.xg_s.copy_(to_dev(xgs))
    L.masked_m.copy_(to_dev(lay["masked_m"]))
    L.offsets.copy_(to_dev(lay["offsets"]))

    def counters():
        torch.cuda.synchronize()
        c = L.ws[:moe.MOE_STATS_BYTES].view(torch.int32).cpu().numpy().reshape(2, moe.MOE_STATS_CTAS, 2)
        return c.sum(axis=1)  # [phase][units, tiles]

    for step, call in ((3, L.swiglu), (4, L.down)):
        call()
        c = counters()
        want_s = oracle.token_tiles(lay["masked_m"], bm[step])
        assert c[0, 1] == want_s and c[1].sum() == 0
        assert c[0, 0] % max(want_s, 1) == 0 and c[0, 0] >= want_s
    L.ffn()
    c = counters()
    assert c[0, 1] == want and c[1, 1] == want


# ---- a5 combine ---------------------------------------------------------------------

@pytest.mark.parametrize("name", NAMES)
def test_combine(workloads, name):
    wl = workloads[name]
    cfg = wl.cfg
    lay = oracle_layout(wl)
    rows = cfg.rows
    yg = mi.normal(9, 55, (rows, cfg.H), dtype="f32" if cfg.y_dtype == "f32" else "bf16")
    w32 = wl.w.astype(np.float32)
    out_ref, exact = oracle.combine(cfg, yg, lay["row_of"], w32)
    L = wl.layer()
    L.yg.copy_(to_dev(yg))
    L.row_of.copy_(to_dev(lay["row_of"]))
    L.w.copy_(to_dev(w32))
    L.combine()
    torch.cuda.synchronize()
    got = real(to_host(L.out), cfg.out)
    # fp32 sum of the same stored values in k order, then one rounding: within half an
    # output ulp of the exact sum plus the fp32 summation error on sum_k |w_k y_k|
    yv = real(yg, cfg.y_dtype)
    ro = lay["row_of"]
    wk = np.concatenate([w32, np.ones((cfg.T, cfg.S), np.float32)], axis=1).astype(np.float64)
    mag = sum(np.abs(wk[:, k:k + 1]) * np.abs(yv[ro[:, k]]) for k in range(cfg.K + cfg.S))
    half_ulp = 2.0 ** -8 if cfg.out == "bf16" else 2.0 ** -24  # 8 or 24 significant bits
    assert (np.abs(got - exact) <= half_ulp * np.abs(exact) * 1.0001 + 2.0 ** -22 * mag).all()
    assert rel_err(got, real(out_ref, cfg.out)) <= TOL[cfg.out]


# ---- two-level accumulation ("Inference INFRA methodology (5)", section "DeepGEMM") ----

def test_fp8_promotion_deep_k_all_positive():
    """All-positive data and K = 16384: with the 128-K promotion to fp32 the down
    GEMM stays at bf16-output accuracy; the page reports about 0.17% with the
    two-level scheme against about 25% without it on its hardware."""
    cfg = SMALL["e4m3_masked_shared"].replace(name="deepk", T=8, H=256, I=16384, E=1, K=1, shared=0, M_max=8)
    rng = np.random.default_rng(0)
    hq = oracle.e4m3_encode(rng.uniform(0.5, 448.0, (cfg.T * 1, cfg.I)).astype(np.float32))
    hs = np.full((cfg.T, cfg.I // 128), 1.0 / 448.0, np.float32)
    wq = oracle.e4m3_encode(rng.uniform(0.5, 448.0, (1, cfg.H, cfg.I)).astype(np.float32))
    ws = np.full((1, cfg.H // 128, cfg.I // 128), 1.0 / 448.0, np.float32)
    masked_m = np.array([cfg.T], np.int32)
    offsets = np.array([0, cfg.T], np.int32)
    ref = oracle.grouped_down(cfg, hq, hs, wq, ws, masked_m, offsets)
    exact = oracle.dequant(hq, "e4m3", hs, 1) @ oracle.dequant(wq[0], "e4m3", ws[0], 128).T
    p = moe.Problem.make(T=cfg.T, H=cfg.H, I=cfg.I, E=1, K=1, M_max=cfg.T, act="bf16", wt="e4m3", out="bf16")
    yg = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_t = torch.empty(max(moe.moe_workspace_bytes(p), 256), dtype=torch.uint8, device="cuda")
    moe.moe_grouped_down_gemm(p, to_dev(hq), to_dev(hs), to_dev(wq), to_dev(ws), to_dev(masked_m),
                              to_dev(offsets), yg, err, ws_t)
    torch.cuda.synchronize()
    got = real(to_host(yg), "bf16")
    rel = np.abs(got - exact) / np.abs(exact)
    assert rel.max() < 0.004  # bf16 output rounding is 2^-9 = 0.2%
    assert rel_err(got, real(ref, "bf16")) < 0.004


# ---- determinism ---------------------------------------------------------------------

@pytest.mark.parametrize("name", ["bf16_masked", "e4m3_eplb_zipf", "e4m3_contig"])
def test_rerun_bitwise_identical(workloads, name):
    wl = workloads[name]
    L = wl.layer()
    x, lg = to_dev(wl.x), to_dev(wl.logits)
    a = to_host(L.forward(x, lg).clone())
    for fused in (False, True, True):  # the one-launch FFN gives the same bits, run after run
        b = to_host(L.forward(x, lg, fused=fused).clone())
        assert (a == b).all()


def test_grouped_ffn_rejects_bad_arguments():
    wl = Workload(SMALL["e2m1_masked_shared"])
    L = wl.layer()
    f = moe.moe_grouped_ffn
    base = [L.p, L.xg, L.xg_s, L.w13, L.w13_s, L.w2, L.w2_s, L.masked_m, L.offsets, L.hg, L.hg_s, L.yg, L.err, L.ws]
    for i in (2, 4, 6, 10):  # e4m3 activations / e2m1 weights need every scale array
        args = list(base)
        args[i] = None
        with pytest.raises(moe.MoeError):
            f(*args)
    args = list(base)
    args[5] = L.w2.view(-1)[16:]  # packed 4-bit weights must start on a 32-byte boundary
    with pytest.raises(moe.MoeError):
        f(*args)
    args = list(base)
    args[13] = L.ws[:8]  # workspace too small for the per-slot counters
    with pytest.raises(moe.MoeError):
        f(*args)


# ---- DeepSeek-V3 routing: sigmoid scores, correction bias, grouped top-k ------------

@pytest.mark.parametrize("T,E,K,ng,tg,with_bias", [(128, 256, 8, 8, 4, True), (37, 64, 6, 8, 3, False),
                                                    (5, 32, 4, 1, 1, False), (64, 512, 10, 16, 4, True),
                                                    (9, 8, 2, 4, 2, True)])
def test_route_grouped(T, E, K, ng, tg, with_bias):
    logits = mi.normal(4, 88, (T, E), dtype="f32")
    logits[0, :] = 0.25                       # all keys tie
    if T > 3:
        logits[3, ::2] = logits[3, 1]         # many ties
    bias = (0.05 * mi.normal(4, 89, (E,), dtype="f32")).astype(np.float32) if with_bias else None
    ids, w = oracle.route_grouped(logits, K, ng, tg, bias=bias, renormalize=True, scale=2.5)
    p = moe.Problem.make(T=T, H=128, I=128, E=E, K=K, M_max=T, act="bf16", wt="bf16", out="bf16")
    gids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    gw = torch.empty((T, K), dtype=torch.float32, device="cuda")
    moe.moe_route_grouped_topk(p, to_dev(logits), to_dev(bias), ng, tg, gids, gw, renormalize=True, scale=2.5)
    torch.cuda.synchronize()
    assert (to_host(gids) == ids).all()
    np.testing.assert_allclose(to_host(gw), w, rtol=2e-6, atol=1e-7)


def test_route_grouped_rejects_bad_groups():
    p = moe.Problem.make(T=4, H=128, I=128, E=12, K=4, M_max=4, act="bf16", wt="bf16", out="bf16")
    t = torch.empty(64, dtype=torch.float32, device="cuda")
    for ng, tg in ((5, 2), (4, 0), (4, 5), (12, 1)):  # 12 % 5, no group, too many groups, K > 1 * 1
        with pytest.raises(moe.MoeError):
            moe.moe_route_grouped_topk(p, t, None, ng, tg, t, t)


# ---- f EPLB load statistics -------------------------------------------------------

@pytest.mark.parametrize("name", ["e4m3_eplb_zipf", "bf16_masked"])
def test_eplb_record_and_rebalance(workloads, name):
    """Record masked_m of several dispatch passes into a wrapping window, then rebalance."""
    wl = workloads[name]
    cfg = wl.cfg
    W, passes = 3, 5
    win = torch.full((W, cfg.P), SENT_I32, dtype=torch.int32, device="cuda")
    want = np.full((W, cfg.P), SENT_I32, np.int32)
    for ps in range(passes):
        logits = mi.normal(8, 300 + ps, (cfg.T, cfg.E), dtype="f32")
        ids, _ = oracle.route(logits, cfg.K)
        Lp = run_permute(wl, ids)
        moe.moe_eplb_record(Lp.p, Lp.masked_m, ps, W, win)
        want[ps % W] = oracle.layout(cfg, ids, wl.p2l)["masked_m"][:cfg.P]
    torch.cuda.synchronize()
    assert (to_host(win) == want).all()
    load, new = oracle.eplb_rebalance(want, cfg.E, wl.p2l)
    gl = torch.empty(cfg.E, dtype=torch.int64, device="cuda")
    gn = torch.full((cfg.P,), SENT_I32, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    p2l = None if wl.p2l is None else torch.from_numpy(wl.p2l).cuda()
    moe.moe_eplb_rebalance(wl.problem, win, W, p2l, gl, gn, err)
    torch.cuda.synchronize()
    assert int(to_host(err)[0]) == 0
    assert (to_host(gl) == load).all()
    assert (to_host(gn) == new).all()


@pytest.mark.parametrize("E,P,W", [(8, 16, 4), (256, 288, 10), (1024, 1024, 2), (64, 96, 1)])
def test_eplb_rebalance_ties_and_sizes(E, P, W):
    rng = np.random.default_rng(E + P)
    window = rng.integers(0, 4, size=(W, P)).astype(np.int32)   # small counts: many equal loads
    p2l = None if P == E else mi.replica_map(rng.integers(0, 50, size=E), E, P - E)
    load, new = oracle.eplb_rebalance(window, E, p2l)
    p = moe.Problem.make(T=1, H=128, I=128, E=E, K=1, P=P, M_max=1)
    gl = torch.empty(E, dtype=torch.int64, device="cuda")
    gn = torch.empty(P, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_eplb_rebalance(p, to_dev(window), W, None if p2l is None else to_dev(p2l), gl, gn, err)
    torch.cuda.synchronize()
    assert int(to_host(err)[0]) == 0
    assert (to_host(gl) == load).all()
    assert (to_host(gn) == new).all()


def test_eplb_rebalance_flags_and_rejects():
    E, P, W = 8, 12, 2
    p = moe.Problem.make(T=1, H=128, I=128, E=E, K=1, P=P, M_max=1)
    window = torch.ones((W, P), dtype=torch.int32, device="cuda")
    gl = torch.empty(E, dtype=torch.int64, device="cuda")
    gn = torch.empty(P, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([0, 1, 2, 3, 4, 5, 6, 7, 0, 8, 1, -1], dtype=torch.int32, device="cuda")
    moe.moe_eplb_rebalance(p, window, W, bad, gl, gn, err)
    torch.cuda.synchronize()
    assert int(to_host(err)[0]) & moe.MOE_FLAG_BAD_MAP
    with pytest.raises(moe.MoeError):      # no map although P != E
        moe.moe_eplb_rebalance(p, window, W, None, gl, gn, err)
    with pytest.raises(moe.MoeError):      # empty window
        moe.moe_eplb_rebalance(p, window, 0, bad, gl, gn, err)
    p2 = moe.Problem.make(T=1, H=128, I=128, E=4, K=1, P=12, M_max=1)
    with pytest.raises(moe.MoeError):      # more extra slots than experts
        moe.moe_eplb_rebalance(p2, window, W, bad, gl, gn, err)
    with pytest.raises(moe.MoeError):
        moe.moe_eplb_record(p, window, 0, 0, window)


# ---- failure detection: a bounded wait that runs out --------------------------------

def test_bounded_wait_expires_with_a_flag():
    """The wait every kernel uses, on an mbarrier nothing completes: after its limit
    (2e6 cycles, about a millisecond) the kernel reports MOE_FLAG_TIMEOUT and returns, and
    the context keeps working."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_selftest_bounded_wait(2_000_000, err)
    torch.cuda.synchronize()
    assert int(to_host(err)[0]) == moe.MOE_FLAG_TIMEOUT
    x = torch.arange(8, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 28.0
    with pytest.raises(moe.MoeError):
        moe.moe_selftest_bounded_wait(0, err)
