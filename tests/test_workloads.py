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


def test_other_draft_format_generators():
    """Zero points and GGUF experts: shapes, determinism, independent streams
    and the scale ranges the recipe states (read back through the format's
    byte layout, not through the oracle)."""
    s = W.scaled(W.CONFIGS["tiny"], H=512, I=256)
    z = W.gen_w4_zeros(s, 0, 1)
    assert z["qz_gate"].shape == (s.H // 128, s.I // 8) and z["qz_down"].shape == (s.I // 128, s.H // 8)
    nib = (z["qz_gate"].view(np.uint32)[..., None] >> (4 * np.arange(8, dtype=np.uint32))) & 15
    assert set(np.unique(nib)) == set(range(16))
    q8 = W.gen_q8_expert(s, 0, 1)
    assert q8["q8_gate"].shape == (s.I, s.H // 32, 34) and q8["q8_down"].shape == (s.H, s.I // 32, 34)
    d = q8["q8_gate"][..., :2].copy().view(np.float16).astype(np.float64)
    assert d.min() >= 0.0003 - 1e-6 and d.max() <= 0.00125 + 1e-6
    q2 = W.gen_q2k_expert(s, 0, 1)
    assert q2["q2k_gate"].shape == (s.I, s.H // 256, 84) and q2["q8_down"].shape == (s.H, s.I // 32, 34)
    d2 = q2["q2k_up"][..., 80:82].copy().view(np.float16).astype(np.float64)
    m2 = q2["q2k_up"][..., 82:84].copy().view(np.float16).astype(np.float64)
    assert d2.min() >= 0.001 - 1e-6 and d2.max() <= 0.003 + 1e-6 and m2.max() <= 0.004 + 1e-6
    q4 = W.gen_q4k_expert(s, 0, 1)
    assert q4["q4k_gate"].shape == (s.I, s.H // 256, 144)
    d4 = q4["q4k_gate"][..., 0:2].copy().view(np.float16).astype(np.float64)
    assert d4.min() >= 0.00015 - 1e-7 and d4.max() <= 0.0004 + 1e-6
    for gen in (W.gen_w4_zeros, W.gen_q8_expert, W.gen_q2k_expert, W.gen_q4k_expert):
        a, b, c = gen(s, 0, 2), gen(s, 0, 2), gen(s, 0, 3)
        assert all(np.array_equal(a[k], b[k]) for k in a)
        assert not all(np.array_equal(a[k], c[k]) for k in a)
