"""The whole layer on the GPU (route -> permute -> gate/up -> down -> combine)
against the token-by-token fp64 oracle.

Reduced workloads: every token.  Full-size workloads (the launch
configuration the benchmark times): routing and layout bit-exact over all
tokens, e4m3 activations bit-exact on sampled rows, layer outputs on sampled
tokens (the oracle computes them one by one)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from cases import SMALL
from gpu_util import TOL, Workload, real, rel_err, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from routed_expert_layer_moe_gb300 import build
    build.build()


def check_layer(wl, tokens=None, fused=False):
    cfg = wl.cfg
    L = wl.layer()
    out = L.forward(to_dev(wl.x), to_dev(wl.logits), fused=fused)
    torch.cuda.synchronize()
    assert int(to_host(L.err)[0]) == 0
    assert (to_host(L.ids) == wl.ids).all()
    lay = oracle.layout(cfg, wl.ids, wl.p2l)
    assert (to_host(L.masked_m) == lay["masked_m"]).all()
    assert (to_host(L.offsets) == lay["offsets"]).all()
    assert (to_host(L.row_of) == lay["row_of"]).all()
    ref, exact = oracle.layer(cfg, wl.x, wl.logits, wl.w13, wl.w13_s, wl.w2, wl.w2_s, tokens=tokens)
    got = real(to_host(out), cfg.out)
    if tokens is not None:
        got = got[tokens]
    e = rel_err(got, exact)
    assert e <= TOL[cfg.gemm], e
    return L, lay


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("name", list(SMALL))
def test_layer_small(name, fused):
    check_layer(Workload(SMALL[name]), fused=fused)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("T", [1, 2, 7])
def test_layer_few_tokens(T, fused):
    check_layer(Workload(SMALL["e4m3_masked_shared"].replace(T=T, M_max=T)), fused=fused)
    check_layer(Workload(SMALL["bf16_masked"].replace(T=T, M_max=T)), fused=fused)
    check_layer(Workload(SMALL["e2m1_masked_shared"].replace(T=T, M_max=T)), fused=fused)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("base,E,K", [("e4m3_masked_shared", 1023, 32), ("bf16_masked", 1024, 8),
                                      ("e2m1_masked_shared", 1023, 16)])
def test_layer_maximum_slots_and_k(base, E, K, fused):
    """The largest problem the ABI takes in slots and experts per token: P + S = 1024 slots
    (1023 routed experts + the shared one, or 1024 routed) and K up to 32, at small H and I;
    every token checked."""
    cfg = SMALL[base].replace(T=24, H=256, I=128, E=E, K=K, M_max=24)
    check_layer(Workload(cfg), fused=fused)


def test_layer_all_tokens_on_few_experts():
    cfg = SMALL["e4m3_masked_shared"]
    x, logits = mi.activations(cfg)
    logits = logits.copy()
    logits[:, :cfg.K] += 50.0  # experts 0..K-1 win for every token; the rest stay empty
    wl = Workload(cfg, logits=logits)
    L, lay = check_layer(wl)
    assert (lay["masked_m"][cfg.K:cfg.P] == 0).all()


@pytest.mark.parametrize("fused", [False, True])
def test_layer_empty_batch(fused):
    cfg = SMALL["bf16_masked"].replace(T=0, M_max=4)
    wl = Workload(SMALL["bf16_masked"])
    wl.cfg = cfg
    from gpu_util import problem_of
    wl.problem = problem_of(cfg)
    wl.ids = np.zeros((0, cfg.K), np.int32)
    L = wl.layer()
    L.forward(torch.empty((0, cfg.H), dtype=torch.bfloat16, device="cuda"),
              torch.empty((0, cfg.E), dtype=torch.float32, device="cuda"), fused=fused)
    torch.cuda.synchronize()
    assert (to_host(L.masked_m) == 0).all() and (to_host(L.offsets) == 0).all()


# ---- full-size workloads, sampled --------------------------------------------------------

FULL = ["tiny", "mixtral_decode", "dsv3_decode", "skew_eplb", "prefill", "dsv4_fp4_decode"]


@pytest.fixture(scope="module")
def dsv3_weights():
    cfg = mi.CONFIGS["dsv3_decode"]
    w13, w13s = mi.expert_weights(cfg, "w13")
    w2, w2s = mi.expert_weights(cfg, "w2")
    return w13, w13s, w2, w2s


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_layer_full_size_sampled(name, request):
    cfg = mi.CONFIGS[name]
    weights = None
    if name in ("dsv3_decode", "skew_eplb"):  # same logical experts (same seed and shapes)
        weights = request.getfixturevalue("dsv3_weights")
    wl = Workload(cfg, weights=weights)
    rng = np.random.default_rng(1)
    n = min(cfg.T, 24)
    tokens = np.unique(np.concatenate([[0, cfg.T - 1], rng.choice(cfg.T, n, replace=False)])).astype(np.int32)
    # the benchmark's launch configuration: gate/up and down in one launch for bf16 experts
    L, lay = check_layer(wl, tokens=tokens, fused=(cfg.gemm == "bf16"))
    if cfg.gemm == "e4m3":
        # dispatch quantisation bit-exact on the sampled tokens' rows
        rows = lay["row_of"][tokens].ravel()
        rows = rows[rows >= 0]
        xf = oracle.bf16_decode(wl.x[tokens]).astype(np.float32)
        q, s = oracle.quant_rows_e4m3(xf)
        gx, gs = to_host(L.xg), to_host(L.xg_s)
        for i, t in enumerate(tokens):
            for r in lay["row_of"][t]:
                assert (gx[r] == q[i]).all() and (gs[r] == s[i]).all()
    del L
    torch.cuda.empty_cache()


def run_layer(wl, fused):
    """The whole pass through the separate calls or through moe_route_permute +
    moe_ffn_combine; every output buffer, with padding rows of the grouped buffers set to a
    sentinel first."""
    L = wl.layer()
    for t in (L.xg, L.hg):
        t.zero_()
    L.yg.fill_(-3.0)
    L.forward(to_dev(wl.x), to_dev(wl.logits), fused=fused)
    torch.cuda.synchronize()
    assert int(to_host(L.err)[0]) == 0
    outs = {n: to_host(getattr(L, n))
            for n in ("ids", "w", "masked_m", "offsets", "row_of", "src_of", "xg", "hg", "yg", "out")}
    for n in ("xg_s", "hg_s"):
        if getattr(L, n) is not None:
            outs[n] = to_host(getattr(L, n))
    return outs, L


@pytest.mark.parametrize("name", list(SMALL) + ["bf16_split_k", "e4m3_t1"])
def test_fused_calls_bit_identical(name):
    """moe_route_permute and moe_ffn_combine give the separate calls' outputs bit for bit: ids,
    weights, layout, the grouped buffers' valid rows (xg, hg, yg and scales) and the layer
    output -- through the one-launch route + dispatch (small batches without a map), its
    two-kernel fallback (replica map), the combine fused into the split-K reduction and the
    combine after an unsplit down GEMM.  The output is also within tolerance of the oracle."""
    # I = 1024: enough K blocks for the down GEMM of a 4-token batch to be split along K
    extra = {"bf16_split_k": SMALL["bf16_masked"].replace(name="bf16_split_k", T=4, I=1024, M_max=4),
             "e4m3_t1": SMALL["e4m3_masked_shared"].replace(name="e4m3_t1", T=1, M_max=1)}
    cfg = extra.get(name) or SMALL[name]
    wl = Workload(cfg)
    sep, _ = run_layer(wl, False)
    fus, L = run_layer(wl, True)
    valid = sep["src_of"] >= 0
    for n in ("ids", "w", "masked_m", "offsets", "row_of", "src_of", "out"):
        assert (fus[n].view(np.uint8) == sep[n].view(np.uint8)).all(), n
    for n in ("xg", "hg", "yg", "xg_s", "hg_s"):
        if n in sep:
            assert (fus[n][valid] == sep[n][valid]).all(), n
    assert (real(fus["yg"][~valid], cfg.y_dtype) == -3.0).all()
    ref, exact = oracle.layer(cfg, wl.x, wl.logits, wl.w13, wl.w13_s, wl.w2, wl.w2_s)
    assert rel_err(real(fus["out"], cfg.out), exact) <= TOL[cfg.gemm]
