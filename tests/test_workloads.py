"""The seeded input recipe: shapes, determinism and the drawn-logit statistics
the recipe is built to produce.  CPU only."""
import numpy as np

import oracle
import spx_workloads as W


def test_shapes_and_dtypes():
    s = W.CONFIGS["deepseek_v2_lite"]
    ex = W.gen_w4_expert(W.scaled(s, I=256), 0, 3)
    assert ex["qw_gate"].shape == (s.H // 8, 256) and ex["qw_gate"].dtype == np.int32
    assert ex["s_gate"].shape == (s.H // 128, 256) and ex["s_gate"].dtype == np.uint16
    assert ex["qw_down"].shape == (256 // 8, s.H) and ex["s_down"].shape == (2, s.H)
    f = W.gen_f16_expert(W.scaled(s, I=128), 0, 1)
    assert f["w_gate"].shape == (128, s.H) and f["w_down"].shape == (s.H, 128)
    assert W.gen_x(s, 17).shape == (17, s.H)
    assert W.gen_logits(s, 17).shape == (17, s.E)


def test_deterministic_and_independent_streams():
    s = W.CONFIGS["tiny"]
    a = W.gen_w4_expert(s, 0, 2)
    b = W.gen_w4_expert(s, 0, 2)
    c = W.gen_w4_expert(s, 0, 3)
    assert all(np.array_equal(a[k], b[k]) for k in a)
    assert not np.array_equal(a["qw_gate"], c["qw_gate"])
    assert not np.array_equal(W.gen_x(s, 4, step=0), W.gen_x(s, 4, step=1))


def test_value_ranges():
    s = W.scaled(W.CONFIGS["tiny"], H=512, I=1024)
    ex = W.gen_w4_expert(s, 0, 0)
    sc = ex["s_gate"].view(np.float16).astype(np.float64)
    assert sc.min() >= 0.005 - 1e-5 and sc.max() <= 0.02 + 1e-5
    codes = (ex["qw_gate"].view(np.uint32)[:, :, None] >> (4 * np.arange(8, dtype=np.uint32))) & 15
    hist = np.bincount(codes.reshape(-1), minlength=16)
    assert hist.min() > 0.9 * hist.mean() and hist.max() < 1.1 * hist.mean()
    w = W.gen_f16_expert(s, 0, 0)["w_gate"].view(np.float16).astype(np.float64)
    assert abs(w.std() - 0.02) < 0.001
    x = W.gen_x(s, 64).view(np.float16).astype(np.float64)
    assert abs(x.std() - 1.0) < 0.02


def test_zipf_top1_share_and_hot_share():
    # Gumbel-top-k of ln p + G samples k experts without replacement prop. to p
    s = W.CONFIGS["deepseek_v2_lite"]
    lg = W.gen_logits(s, 20000, layer=0, step=99)
    ids, _ = oracle.route_topk(lg.astype(np.float64), s.k, False)
    first = np.bincount(ids[:, 0], minlength=s.E) / len(ids)
    r = np.arange(1, s.E + 1) ** -1.1
    assert abs(first.max() - r[0] / r.sum()) < 0.01   # ~25%
    p = W.CONFIGS["phi35_moe"]
    lg = W.gen_logits(p, 20000, layer=0, step=99)
    ids, _ = oracle.route_topk(lg.astype(np.float64), p.k, True)
    share = np.sort(np.bincount(ids.reshape(-1), minlength=p.E))[::-1][:4].sum() / ids.size
    assert abs(share - 0.5) < 0.01


def test_verify_logits_reuse_draft_steps():
    s = W.CONFIGS["deepseek_v2_lite_x26"]
    v = W.verify_logits(s, 5)
    assert v.shape == (s.K + 1, s.E)
    for i in range(1, s.K + 1):
        assert np.array_equal(v[i - 1], W.draft_logits(s, 5, i)[0])
