"""The seeded input generator: determinism, slicing, distributions, recipes."""
import numpy as np

import moe_inputs as mi
import oracle
from cases import SMALL


def test_deterministic_and_sliceable():
    a = mi.normal(0, 4, (1000,))
    b = mi.normal(0, 4, (1000,))
    assert (a == b).all()
    # counter based: any window is the same as the slice of the whole
    c = mi.normal(0, 4, (301,), offset=333)
    assert (c == a[333:634]).all()
    assert not (mi.normal(1, 4, (1000,)) == a).any()


def test_normal_moments():
    x = mi.normal(0, 1, (400000,))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    u = mi.uniform(0, 2, (200000,), 0.5, 2.0)
    assert u.min() >= 0.5 and u.max() < 2.0 and abs(u.mean() - 1.25) < 0.01


def test_expert_slices_match_whole():
    cfg = SMALL["e4m3_masked_shared"]
    q, s = mi.expert_weights(cfg, "w13")
    q2, s2 = mi.expert_weights(cfg, "w13", e0=5, ne=3)
    assert (q2 == q[5:8]).all() and (s2 == s[5:8]).all()
    b = SMALL["bf16_masked"]
    w, _ = mi.expert_weights(b, "w2")
    w2, _ = mi.expert_weights(b, "w2", e0=7, ne=1)
    assert (w2 == w[7:8]).all()


def test_e4m3_weight_recipe():
    """Per 128x128 block: s = u * max|w| / 448 with u in [0.5, 2]; so the largest
    code magnitude of a block is 448/u (saturated at 448), and the dequantised
    block has standard deviation near w_std."""
    cfg = SMALL["e4m3_masked_shared"]
    q, s = mi.expert_weights(cfg, "w2")
    v = oracle.e4m3_decode(q).reshape(q.shape[0], cfg.H // 128, 128, cfg.I // 128, 128)
    amax_code = np.abs(v).max(axis=(2, 4))
    u = 448.0 / amax_code
    sat = amax_code >= 448.0
    assert (u[~sat] >= 0.5 * (1 - 1 / 16) - 1e-9).all() and (u[~sat] <= 2.0 * (1 + 1 / 16) + 1e-9).all()
    assert sat.mean() < 0.5
    deq = oracle.dequant(q, "e4m3", s, 128)
    assert abs(deq.std() - cfg.w_std) < 0.1 * cfg.w_std


def test_e2m1_weight_recipe():
    """FP4 weights: per 128x128 block s = u * max|w| / 6 with u in [0.5, 2], so the
    block's largest code magnitude is e2m1(6/u): 6 when u <= 1.2 (saturated or
    rounded up), else 3 or 4; the codes are packed two per byte; the dequantised
    weights keep the drawn standard deviation within FP4's coarse grid."""
    cfg = SMALL["e2m1_masked_shared"]
    q, s = mi.expert_weights(cfg, "w13")
    assert q.shape == (cfg.n_exp, 2 * cfg.I, cfg.H // 2) and s.shape == (cfg.n_exp, 2 * cfg.I // 128, cfg.H // 128)
    v = oracle.dequant(q, "e2m1", np.ones_like(s), 128)
    blocks = np.abs(v).reshape(cfg.n_exp, 2 * cfg.I // 128, 128, cfg.H // 128, 128).max(axis=(2, 4))
    assert set(np.unique(blocks)) <= {3.0, 4.0, 6.0}
    deq = oracle.dequant(q, "e2m1", s, 128)
    assert abs(deq.std() - cfg.w_std) < 0.25 * cfg.w_std
    # same draws as the e4m3 weights of the same shapes: the two dequantisations agree to FP4 precision
    q8, s8 = mi.expert_weights(cfg.replace(wq=""), "w13")
    d8 = oracle.dequant(q8, "e4m3", s8, 128)
    assert np.corrcoef(deq.ravel(), d8.ravel())[0, 1] > 0.97


def test_router_recipes():
    cfg = SMALL["e4m3_eplb_zipf"]
    _, logits = mi.activations(cfg)
    # Zipf bias: expert 0 is chosen far more often than the last one
    ids, _ = oracle.route(logits, cfg.K)
    cnt = np.bincount(ids.ravel(), minlength=cfg.E)
    assert cnt[0] > cnt[-1] + cfg.T // 4
    t = SMALL["tiny"]
    x, lg = mi.activations(t)
    assert x.dtype == np.float32 and lg.shape == (t.T, t.E)
    p2l = mi.replica_map(np.array([5, 9, 9, 1]), 4, 2)
    assert p2l.tolist() == [0, 1, 2, 3, 1, 2]
