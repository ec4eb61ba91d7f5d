"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test checks the oracle against one of: a worked example printed on the
pages, a library routine the step reduces to, a closed form, a conservation
law the pages state, or brute force on tiny inputs.  A plausible slip in the
oracle (a dropped term, a swapped gate/up, a transposed weight, a wrong tie
rule, a wrong rounding) fails at least one of them."""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special
import torch

import moe_inputs as mi
import oracle
from cases import SMALL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- EPLB maps (vLLM EPLB, section 1.2, worked example) --------------------

def test_eplb_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "eplb_worked_example.json")))
    E = g["num_logical_experts"]
    for case in g["cases"]:
        l2p, rc, r = oracle.eplb_invert(case["physical_to_logical_map"], E)
        assert l2p.tolist() == case["logical_to_physical_map"]
        assert rc.tolist() == case["logical_replica_count"]
        assert r == max(case["logical_replica_count"])


def test_pad_waste_worked_example():
    """The pages' padding-waste figures at M_e = 5 rows (golden file), and the tile count they
    rest on: ceil(rows / BM) tiles per slot with rows, none for an empty slot."""
    g = json.load(open(os.path.join(GOLDEN, "deepgemm_pad_waste.json")))
    for c in g["cases"]:
        assert oracle.pad_waste(g["M_e"], c["BM"]) == pytest.approx(c["waste"], rel=1e-12)
    mm = np.array([5, 0, 128, 129, 1, 256], np.int32)
    assert oracle.token_tiles(mm, 128) == 1 + 0 + 1 + 2 + 1 + 2
    assert oracle.token_tiles(mm, 16) == 1 + 0 + 8 + 9 + 1 + 16


def test_eplb_rejects_bad_map():
    with pytest.raises(ValueError):
        oracle.eplb_invert([0, 1, 4], 4)
    with pytest.raises(ValueError):
        oracle.eplb_invert([0, 0, 0], 2, R=2)


# ---- routing ---------------------------------------------------------------

def _ref_route(logits, K):
    """Library reference: stable argsort on -logit, scipy softmax over all E,
    renormalised over the chosen K."""
    ids = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :K]
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    pk = np.take_along_axis(p, ids, axis=1)
    return ids, pk / pk.sum(axis=1, keepdims=True)


@pytest.mark.parametrize("T,E,K", [(16, 8, 2), (33, 256, 8), (20, 512, 10), (5, 4, 4), (7, 6, 1)])
def test_route_matches_library(T, E, K):
    logits = mi.normal(3, 99, (T, E), dtype="f32")
    ids, w = oracle.route(logits, K)
    rid, rw = _ref_route(logits, K)
    assert (ids == rid).all()
    np.testing.assert_allclose(w, rw, rtol=1e-13, atol=1e-15)


def test_route_special_cases():
    rng = np.random.default_rng(0)
    logits = rng.standard_normal((9, 6)).astype(np.float32)
    # K = E: every expert, weights = the full softmax
    ids, w = oracle.route(logits, 6)
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, ids, 1), rtol=1e-13)
    # K = 1: weight 1
    _, w1 = oracle.route(logits, 1)
    assert (w1 == 1.0).all()
    # equal logits: ids 0..K-1 (ties to the lower index), equal weights
    ids, w = oracle.route(np.zeros((3, 8), np.float32), 3)
    assert ids.tolist() == [[0, 1, 2]] * 3
    np.testing.assert_allclose(w, 1.0 / 3.0, rtol=1e-15)
    # partial ties: lower index first among equal logits
    l = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]], np.float32)
    ids, _ = oracle.route(l, 4)
    assert ids.tolist() == [[1, 2, 4, 3]]


def test_route_top2_then_softmax_equivalence():
    """Mixtral computes top-2 first and a softmax over those two logits; the
    softmax-then-renormalise form gives the same weights."""
    logits = mi.normal(5, 7, (50, 8), dtype="f32")
    ids, w = oracle.route(logits, 2)
    top = np.take_along_axis(logits.astype(np.float64), ids, 1)
    np.testing.assert_allclose(w, scipy.special.softmax(top, axis=1), rtol=1e-13)


# ---- codecs -----------------------------------------------------------------

def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert (np.isnan(v) == nan).all() and nan.sum() == 2  # S.1111.111
    assert (v[~nan] == lib[~nan]).all()
    # constants of the OCP E4M3 format
    assert v[0x7E] == 448.0 and v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6 and v[0x38] == 1.0
    assert v[0xFE] == -448.0 and v[0x80] == 0.0


def test_e4m3_encode_rne_satfinite():
    fin = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (fin[:-1] + fin[1:]) / 2.0  # exact ties
    rng = np.random.default_rng(1)
    vals = np.concatenate([fin, mids, -mids, rng.standard_normal(20000) * 50,
                           rng.standard_normal(2000) * 1e-3, [449.0, 463.9, 470.0, 1e6, -1e6, -0.0]])
    vals = vals.astype(np.float32)
    got = oracle.e4m3_encode(vals)
    ref = torch.from_numpy(vals).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (got == ref).all()
    # ties go to the even code
    tie = oracle.e4m3_encode(np.array([(1.0 + 1.125) / 2, (1.125 + 1.25) / 2], np.float32))
    assert tie.tolist() == [0x38, 0x3A]


# OCP Microscaling Formats (MX) v1.0, section 5.3.3 (FP4 E2M1): exponent bias
# 1, one mantissa bit, no Inf/NaN; the eight magnitudes as the spec lists them.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_all_codes():
    v = oracle.e2m1_decode(np.arange(16))
    assert v[:8].tolist() == E2M1_MAGNITUDES
    assert (v[8:] == -np.array(E2M1_MAGNITUDES)).all() and np.signbit(v[8])


def test_e2m1_packed_nibble_order_and_scales():
    """Byte j of a row holds column 2j in its low nibble; block scales index
    [row/128][col/128]."""
    data = np.zeros((128, 128), np.uint8)          # 128 rows x 256 columns
    data[0, 0] = 0x71                               # col 0 = 0.5, col 1 = 6
    data[5, 64] = 0x2F                              # col 128 = -6, col 129 = 1
    s = np.array([[2.0, 0.25]], np.float32)         # one 128-row block, two column blocks
    v = oracle.dequant(data, "e2m1", s, 128)
    assert v.shape == (128, 256)
    assert v[0, 0] == 1.0 and v[0, 1] == 12.0 and v[5, 128] == -1.5 and v[5, 129] == 0.25
    assert np.count_nonzero(v) == 4


def _e2m1_unpack_by_hand(q):
    """Independent unpacking for the checks below: nibble -> sign * magnitude."""
    mag = np.array(E2M1_MAGNITUDES)
    lo, hi = q & 15, q >> 4
    out = np.empty(q.shape[:-1] + (2 * q.shape[-1],))
    out[..., 0::2] = np.where(lo & 8, -1.0, 1.0) * mag[lo & 7]
    out[..., 1::2] = np.where(hi & 8, -1.0, 1.0) * mag[hi & 7]
    return out


def test_single_fp4_expert_steps_against_dense():
    """E = 1, K = 1 with FP4 weights: gate/up and down of the oracle against numpy
    matmuls on weights decoded by hand (scales expanded per 128x128 block)."""
    cfg = SMALL["e2m1_masked_shared"].replace(T=6, H=256, I=128, E=1, K=1, shared=0, M_max=6)
    x, logits = mi.activations(cfg)
    w13, w13s = mi.expert_weights(cfg, "w13")
    w2, w2s = mi.expert_weights(cfg, "w2")
    ex = lambda s_: np.repeat(np.repeat(s_.astype(np.float64), 128, 0), 128, 1)
    W13 = _e2m1_unpack_by_hand(w13[0]) * ex(w13s[0])     # [2I, H]
    W2 = _e2m1_unpack_by_hand(w2[0]) * ex(w2s[0])        # [H, I]
    ids, _ = oracle.route(logits, 1)
    lay = oracle.layout(cfg, ids)
    xg, xgs = oracle.dispatch_values(cfg, x, lay["row_of"])
    hg, hgs = oracle.grouped_swiglu(cfg, xg, xgs, w13, w13s, lay["masked_m"], lay["offsets"])
    xq = oracle.dequant(xg[:6], "e4m3", xgs[:6], 1)
    g, u = xq @ W13[:128].T, xq @ W13[128:].T
    h = _silu(g) * u
    hq = oracle.dequant(hg[:6], "e4m3", hgs[:6], 1)
    assert np.abs(hq - h).max() <= np.abs(h).max() / 16      # e4m3 keeps 4 significant bits
    assert np.abs(hq - h).max() > 0
    yg = oracle.grouped_down(cfg, hg, hgs, w2, w2s, lay["masked_m"], lay["offsets"])
    y = hq @ W2.T
    yb = oracle.dequant(yg[:6], "bf16")
    assert np.abs(yb - y).max() <= 2.0 ** -8 * np.abs(y).max()


def test_bf16_encode_rne():
    rng = np.random.default_rng(2)
    base = rng.standard_normal(50000).astype(np.float32)
    bits = base.view(np.uint32)
    ties = ((bits & 0xFFFF0000) | 0x8000).view(np.float32)  # exactly half an ulp
    vals = np.concatenate([base, ties, np.float32([1e-40, 3.4e38, 0.0, -0.0])])
    got = oracle.bf16_encode(vals.astype(np.float64))
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (got == ref).all()


def test_quant_rows_reduces_to_library_calls():
    """The 1x128 rule is fp32 division by amax/448 and an RNE satfinite cast."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 512)).astype(np.float32)
    x[2, 128:256] = 0.0
    q, s = oracle.quant_rows_e4m3(x)
    xt = torch.from_numpy(x).view(6, 4, 128)
    amax = xt.abs().amax(-1)
    sref = torch.where(amax == 0, torch.ones_like(amax), amax / torch.tensor(448.0, dtype=torch.float32))
    qref = (xt / sref[..., None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    assert (s == sref.numpy()).all()
    assert (q == qref.reshape(6, 512).numpy()).all()
    # the largest element of a group maps to +-448 exactly
    g = x[0, :128]
    i = np.argmax(np.abs(g))
    assert q[0, i] in (0x7E, 0xFE)
    assert s[2, 1] == 1.0 and (q[2, 128:256] == 0).all()


# ---- layout -----------------------------------------------------------------

def _brute_layout(cfg, ids, p2l):
    """Definition on tiny inputs: slot by replica round-robin, rows of a slot
    listed by ascending token index."""
    T, K = ids.shape
    P, S = cfg.P, cfg.S
    if p2l is None:
        slot = lambda t, e: e
    else:
        reps = {e: [s for s in range(P) if p2l[s] == e] for e in range(cfg.E)}
        slot = lambda t, e: reps[e][t % len(reps[e])]
    members = {s: [] for s in range(P + S)}
    for t in range(T):
        for k in range(K):
            members[slot(t, ids[t, k])].append((t, k))
        if S:
            members[P].append((t, K))
    counts = [len(members[s]) for s in range(P + S)]
    offsets = [0] + list(itertools.accumulate(counts))
    row_of = np.zeros((T, K + S), np.int64)
    for s in range(P + S):
        for rank, (t, k) in enumerate(sorted(members[s])):
            row_of[t, k] = s * cfg.M_max + rank if cfg.layout == "masked" else offsets[s] + rank
    return np.array(counts), np.array(offsets), row_of


@pytest.mark.parametrize("layout", ["masked", "contig"])
@pytest.mark.parametrize("shared", [0, 1])
@pytest.mark.parametrize("use_map", [False, True])
def test_layout_brute_force(layout, shared, use_map):
    rng = np.random.default_rng(4)
    for trial in range(40):
        E = int(rng.integers(1, 5))
        K = int(rng.integers(1, E + 1))
        T = int(rng.integers(1, 7))
        extra = int(rng.integers(0, 3)) if use_map else 0
        cfg = SMALL["tiny"].replace(T=T, E=E, K=K, shared=shared, layout=layout, M_max=T if layout == "masked" else 0,
                                    redundant=extra)
        ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
        p2l = None
        if use_map:
            p2l = np.concatenate([np.arange(E), rng.integers(0, E, extra)]).astype(np.int32)
            rng.shuffle(p2l)
        got = oracle.layout(cfg, ids, p2l)
        assert got["status"] == 0
        counts, offsets, row_of = _brute_layout(cfg, ids, p2l)
        assert (got["masked_m"] == counts).all()
        assert (got["offsets"] == offsets).all()
        assert (got["row_of"] == row_of).all()
        # src_of inverts row_of on every written row
        for t in range(T):
            for r in got["row_of"][t]:
                assert got["src_of"][r] == t


def test_counts_conserved_and_replicas_sum():
    """MoonEP 'Why dynamic routing is hard': per-expert counts sum to the
    number of routed records (R=1 here: T*K); replica counts sum to the
    logical count; the shared slot holds every token."""
    cfg = SMALL["e4m3_eplb_zipf"]
    x, logits = mi.activations(cfg)
    ids, _ = oracle.route(logits, cfg.K)
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    p2l = mi.replica_map(counts, cfg.E, cfg.redundant)
    lay = oracle.layout(cfg, ids, p2l)
    mm = lay["masked_m"]
    assert mm[:cfg.P].sum() == cfg.T * cfg.K
    assert mm[cfg.P] == cfg.T
    per_logical = np.bincount(p2l, weights=mm[:cfg.P], minlength=cfg.E)
    assert (per_logical == counts).all()
    # replica of record (t, k) is the (t mod replica_count)-th slot of its expert
    l2p, rc, _ = oracle.eplb_invert(p2l, cfg.E)
    for t in range(cfg.T):
        for k in range(cfg.K):
            e = ids[t, k]
            assert lay["slot_of"][t, k] == l2p[e, t % rc[e]]


def test_layout_overflow_and_bad_ids():
    cfg = SMALL["tiny"].replace(T=4, E=2, K=1, M_max=2)
    ids = np.zeros((4, 1), np.int32)
    assert oracle.layout(cfg, ids)["status"] == -2      # 4 rows into M_max = 2
    assert oracle.layout(cfg, ids + 5)["status"] == -1  # expert id out of range
    cfg2 = cfg.replace(K=2, M_max=4)
    assert oracle.layout(cfg2, np.zeros((4, 2), np.int32))["status"] == -3  # same expert twice


# ---- expert FFN ---------------------------------------------------------------

def _silu(z):
    return z / (1.0 + np.exp(-z))


@pytest.mark.parametrize("H,I", [(64, 128), (96, 40)])
def test_single_expert_is_dense_swiglu(H, I):
    """E = 1, K = 1: the layer is one dense SwiGLU FFN, y = W2 (silu(W1 x) * W3 x),
    evaluated here with numpy matmuls on the math (untransposed) weights."""
    cfg = SMALL["tiny"].replace(T=5, H=H, I=I, E=1, K=1, M_max=5)
    x, logits = mi.activations(cfg)
    w13, _ = mi.expert_weights(cfg, "w13")
    w2, _ = mi.expert_weights(cfg, "w2")
    out, exact = oracle.layer(cfg, x, logits, w13, None, w2, None)
    W1 = w13[0, :I, :].astype(np.float64).T   # [H, I]
    W3 = w13[0, I:, :].astype(np.float64).T   # [H, I]
    W2 = w2[0].astype(np.float64).T           # [I, H]
    xf = x.astype(np.float64)
    h = (_silu(xf @ W1) * (xf @ W3)).astype(np.float32).astype(np.float64)
    y = (h @ W2).astype(np.float32).astype(np.float64)
    np.testing.assert_allclose(exact, y, rtol=1e-12, atol=1e-14)


def test_closed_forms():
    """Zero gate weights give silu(0) = 0 and a zero output; an identity-like
    W2 (H = I, ones on the diagonal) returns h itself."""
    cfg = SMALL["tiny"].replace(T=3, H=128, I=128, E=1, K=1, M_max=3)
    x, logits = mi.activations(cfg)
    w13, _ = mi.expert_weights(cfg, "w13")
    w2 = np.eye(128, dtype=np.float32)[None]
    z = w13.copy()
    z[0, :128] = 0.0
    _, ex0 = oracle.layer(cfg, x, logits, z, None, w2, None)
    assert (ex0 == 0).all()
    _, ex1 = oracle.layer(cfg, x, logits, w13, None, w2, None)
    xf = x.astype(np.float64)
    h = _silu(xf @ w13[0, :128].astype(np.float64).T) * (xf @ w13[0, 128:].astype(np.float64).T)
    np.testing.assert_allclose(ex1, h.astype(np.float32), rtol=1e-12)


def test_weighted_combine_and_shared_expert():
    """Two experts plus a shared one on one token, checked by hand: out = w0 y0 + w1 y1 + y_shared."""
    cfg = SMALL["tiny"].replace(T=1, H=128, I=128, E=3, K=2, shared=1, M_max=1)
    x, logits = mi.activations(cfg)
    w13, _ = mi.expert_weights(cfg, "w13")
    w2, _ = mi.expert_weights(cfg, "w2")
    _, exact = oracle.layer(cfg, x, logits, w13, None, w2, None)
    ids, w = oracle.route(logits, 2)
    xf = x[0].astype(np.float64)

    def ffn(e):
        g = w13[e, :128].astype(np.float64) @ xf
        u = w13[e, 128:].astype(np.float64) @ xf
        h = (_silu(g) * u).astype(np.float32).astype(np.float64)
        return (w2[e].astype(np.float64) @ h).astype(np.float32).astype(np.float64)

    ref = w[0, 0] * ffn(ids[0, 0]) + w[0, 1] * ffn(ids[0, 1]) + ffn(3)
    np.testing.assert_allclose(exact[0], ref, rtol=1e-12)


@pytest.mark.parametrize("name", list(SMALL))
def test_steps_compose_to_layer(name):
    """The per-call oracles (dispatch, gate/up, down, combine) chained over the
    grouped layout reproduce the token-by-token layer, replicas included."""
    cfg = SMALL[name]
    x, logits = mi.activations(cfg)
    w13, w13s = mi.expert_weights(cfg, "w13")
    w2, w2s = mi.expert_weights(cfg, "w2")
    ids, w = oracle.route(logits, cfg.K)
    p2l = None
    if cfg.redundant:
        p2l = mi.replica_map(np.bincount(ids.ravel(), minlength=cfg.E), cfg.E, cfg.redundant)
    lay = oracle.layout(cfg, ids, p2l)
    assert lay["status"] == 0
    order = mi.slot_experts(cfg, p2l)
    sw13, sw2 = w13[order], w2[order]
    sw13s = None if w13s is None else w13s[order]
    sw2s = None if w2s is None else w2s[order]
    xg, xgs = oracle.dispatch_values(cfg, x, lay["row_of"])
    hg, hgs = oracle.grouped_swiglu(cfg, xg, xgs, sw13, sw13s, lay["masked_m"], lay["offsets"])
    yg = oracle.grouped_down(cfg, hg, hgs, sw2, sw2s, lay["masked_m"], lay["offsets"])
    out, exact = oracle.combine(cfg, yg, lay["row_of"], w.astype(np.float32))
    lout, lexact = oracle.layer(cfg, x, logits, w13, w13s, w2, w2s)
    scale = np.abs(lexact).max()
    assert np.abs(exact - lexact).max() <= 1e-6 * scale


def test_replica_invariance():
    """A replica map changes where tokens run, not the layer's output."""
    cfg = SMALL["e4m3_eplb_zipf"]
    x, logits = mi.activations(cfg)
    w13, w13s = mi.expert_weights(cfg, "w13")
    w2, w2s = mi.expert_weights(cfg, "w2")
    ids, w = oracle.route(logits, cfg.K)
    outs = []
    for p2l in (None, mi.replica_map(np.bincount(ids.ravel(), minlength=cfg.E), cfg.E, cfg.redundant)):
        c = cfg if p2l is not None else cfg.replace(redundant=0)
        lay = oracle.layout(c, ids, p2l)
        order = mi.slot_experts(c, p2l)
        xg, xgs = oracle.dispatch_values(c, x, lay["row_of"])
        hg, hgs = oracle.grouped_swiglu(c, xg, xgs, w13[order], w13s[order], lay["masked_m"], lay["offsets"])
        yg = oracle.grouped_down(c, hg, hgs, w2[order], w2s[order], lay["masked_m"], lay["offsets"])
        outs.append(oracle.combine(c, yg, lay["row_of"], w.astype(np.float32))[1])
    assert (outs[0] == outs[1]).all()


# ---- coverage (INFRA-5, section "Batch") ----------------------------------------

def test_coverage_formula_monte_carlo():
    """Under uniform routing a batch of B tokens touches about E * C(B) experts,
    C(B) = 1 - (1 - k/E)^B."""
    T, E, K = 128, 256, 8
    touched = []
    for seed in range(12):
        logits = mi.normal(seed, mi.STREAM_LOGITS, (T, E), dtype="f32")
        ids, _ = oracle.route(logits, K)
        touched.append(len(np.unique(ids)))
    C = 1.0 - (1.0 - K / E) ** T
    assert abs(np.mean(touched) - E * C) < 1.5


# ---- sigmoid + bias grouped routing ("MoE inference and expert parallelism", Table 3-1) ----

def _sig(x):
    return scipy.special.expit(np.asarray(x, np.float64))


def test_grouped_route_worked_example():
    """E = 8 in 4 groups of 2, keep 2 groups, K = 2.  Group maxima (logits) are 5, 1, 4, 3,
    so groups {0,1} and {4,5} survive and experts 6, 7 (logit 3) are excluded although
    their logits beat expert 0's and 5's."""
    l = np.array([[0.0, 5.0, 1.0, 1.0, 4.0, 0.0, 3.0, 3.0]], np.float32)
    ids, w = oracle.route_grouped(l, 2, n_group=4, topk_group=2)
    assert ids.tolist() == [[1, 4]]
    s = _sig([5.0, 4.0])
    np.testing.assert_allclose(w[0], s / s.sum(), rtol=1e-14)
    # a bias of +1 on expert 7 lifts its group and wins the selection; the weight stays unbiased
    bias = np.array([0, 0, 0, 0, 0, 0, 0, 1.0], np.float32)
    ids, w = oracle.route_grouped(l, 2, n_group=4, topk_group=2, bias=bias)
    assert ids.tolist() == [[7, 1]]
    s = _sig([3.0, 5.0])
    np.testing.assert_allclose(w[0], s / s.sum(), rtol=1e-14)
    # without renormalisation, with a scaling factor
    ids, w = oracle.route_grouped(l, 2, n_group=4, topk_group=2, renormalize=False, scale=2.5)
    np.testing.assert_allclose(w[0], 2.5 * _sig([5.0, 4.0]), rtol=1e-14)


def test_grouped_route_one_group_is_sorted_topk():
    """One group and no bias: sigmoid is increasing, so the choice is the stable sort of the logits."""
    logits = mi.normal(2, 41, (30, 64), dtype="f32")
    ids, w = oracle.route_grouped(logits, 6, n_group=1, topk_group=1)
    ref = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :6]
    assert (ids == ref).all()
    s = np.take_along_axis(_sig(logits), ref, 1)
    np.testing.assert_allclose(w, s / s.sum(1, keepdims=True), rtol=1e-13)


def test_grouped_route_brute_force_sorting():
    """Tiny inputs against the definition written with sorts instead of repeated arg-max."""
    rng = np.random.default_rng(5)
    for _ in range(200):
        ng = int(rng.choice([1, 2, 4]))
        gs = int(rng.integers(1, 4))
        E = ng * gs
        tg = int(rng.integers(1, ng + 1))
        K = int(rng.integers(1, tg * gs + 1))
        l = np.round(rng.standard_normal((1, E)) * 2, 1).astype(np.float32)  # rounding creates ties
        bias = (np.round(rng.standard_normal(E), 1).astype(np.float32) if rng.random() < 0.5 else None)
        ids, _ = oracle.route_grouped(l, K, ng, tg, bias=bias)
        key = _sig(l[0]) + (0 if bias is None else bias.astype(np.float64))
        gmax = [max(key[g * gs:(g + 1) * gs]) for g in range(ng)]
        groups = sorted(range(ng), key=lambda g: (-gmax[g], g))[:tg]
        cand = [e for e in range(E) if e // gs in groups]
        ref = sorted(cand, key=lambda e: (-key[e], e))[:K]
        assert ids[0].tolist() == ref


# ---- EPLB load statistics (vLLM EPLB, section 1.2) ---------------------------------------

def test_eplb_rebalance_worked_map():
    """The page's map [0,1,2,3,0,1]: slots P0/P4 hold E0 and P1/P5 hold E1, so a
    window's physical loads fold onto the logical experts through the map."""
    win = np.array([[10, 4, 3, 2, 6, 1], [5, 1, 7, 0, 2, 0]], np.int32)
    load, new = oracle.eplb_rebalance(win, 4, p2l=[0, 1, 2, 3, 0, 1])
    assert load.tolist() == [10 + 6 + 5 + 2, 4 + 1 + 1 + 0, 3 + 7, 2 + 0]
    assert new.tolist() == [0, 1, 2, 3, 0, 2]  # the two extra slots go to the two hottest


def test_eplb_rebalance_counts_match_routing():
    """Recording masked_m of a pass and folding it through the map gives back the
    per-expert routing counts (the replica split does not lose or add tokens)."""
    cfg = SMALL["e4m3_eplb_zipf"]
    x, logits = mi.activations(cfg)
    ids, _ = oracle.route(logits, cfg.K)
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    p2l = mi.replica_map(counts, cfg.E, cfg.redundant)
    lay = oracle.layout(cfg, ids, p2l)
    win = lay["masked_m"][None, :cfg.P].astype(np.int32)
    load, new = oracle.eplb_rebalance(win, cfg.E, p2l)
    assert (load == counts).all()
    hottest = sorted(range(cfg.E), key=lambda e: (-counts[e], e))[:cfg.redundant]
    assert new[cfg.E:].tolist() == hottest and new[:cfg.E].tolist() == list(range(cfg.E))
    # the rebalanced map reproduces the replica rule used to build the workload
    assert (new == p2l).all()
