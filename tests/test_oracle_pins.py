"""Pins for the CPU oracle: each check ties an oracle step to something other
than the oracle itself (a library routine, brute force, a closed form, an
invariant, or a hand-derived fixture from the format's definition).
Runs on CPU only."""
import itertools
import json
import os

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
import spx_workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ fp16
def test_half_decode_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros survive
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0])


def test_half_encode_rne_vs_numpy():
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(200000) * np.exp(rng.uniform(-20, 12, 200000)),
        # exact ties between neighbouring halves, normal and subnormal ranges
        (np.arange(1, 4000, dtype=np.float64) + 0.5) * 2.0 ** -24,
        (np.arange(1024, 3048, dtype=np.float64) + 0.5) * 2.0 ** -10,
        np.array([65504.0, 65519.999, 65520.0, 1e9, -65520.0, 2.0 ** -25, 2.0 ** -26,
                  3 * 2.0 ** -26, 0.0, -0.0, 6.1e-5, 2.0 ** -14 - 2.0 ** -26]),
    ])
    ours = oracle.double_to_half(v)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# -------------------------------------------------------- router product
def _f16(a):
    return np.asarray(a, np.float64).astype(np.float16).view(np.uint16)


def test_router_logits_one_hot_router_rows_select_x():
    """A router row that is 1.0 at position h and 0 elsewhere gives the
    logit x[t][h] exactly; positions cover both ends of H, so a loop over a
    wrong range of h, or over the wrong operand, fails."""
    rng = np.random.default_rng(11)
    T, H, E = 5, 640, 9
    x = _f16(rng.standard_normal((T, H)))
    pos = np.array([0, H - 1, 1, H - 2, 127, 128, 300, 511, 513])
    wr = np.zeros((E, H), np.uint16)
    wr[np.arange(E), pos] = _f16(1.0)
    got = oracle.router_logits(x, wr)
    want = x.view(np.float16).astype(np.float64)[:, pos]
    assert np.array_equal(got, want)


def test_router_logits_one_hot_tokens_select_router_columns():
    """The transposed case: token t that is 1.0 at position h_t picks
    column h_t of every router row, logits[t][e] = wr[e][h_t]."""
    rng = np.random.default_rng(12)
    T, H, E = 6, 384, 64
    wr = _f16(rng.standard_normal((E, H)) * 0.02)
    pos = np.array([0, H - 1, 5, 200, 257, 128])
    x = np.zeros((T, H), np.uint16)
    x[np.arange(T), pos] = _f16(1.0)
    got = oracle.router_logits(x, wr)
    assert np.array_equal(got, wr.view(np.float16).astype(np.float64)[:, pos].T)


def test_router_logits_vs_numpy_matmul_and_closed_form():
    """Random fp16 operands: fp64 products of fp16 values are exact, so the
    oracle's ascending-h sum agrees with numpy's fp64 product to a few ulp of
    the sum of |terms|; a router of constant rows c gives c * sum_h x[t][h]."""
    rng = np.random.default_rng(13)
    for T, H, E in [(1, 2048, 64), (9, 2048, 60), (4, 256, 8), (17, 4096, 16)]:
        x = _f16(rng.standard_normal((T, H)))
        wr = _f16(rng.standard_normal((E, H)) * 0.02)
        xd, wd = x.view(np.float16).astype(np.float64), wr.view(np.float16).astype(np.float64)
        got = oracle.router_logits(x, wr)
        ref = xd @ wd.T
        bound = 4 * H * np.finfo(np.float64).eps * (np.abs(xd) @ np.abs(wd).T)
        assert np.all(np.abs(got - ref) <= bound)
        c = 0.25
        const = oracle.router_logits(x, np.full((3, H), _f16(c), np.uint16))
        assert np.allclose(const, c * xd.sum(1, keepdims=True), rtol=0, atol=4 * H * 2.2e-16 * np.abs(xd).sum())


# ------------------------------------------------------------- routing
def _brute_topk(v, k):
    order = sorted(range(len(v)), key=lambda e: (-float(np.float32(v[e])), e))
    return order[:k]


def test_topk_all_permutations_tiny():
    for perm in itertools.permutations([0.5, -1.0, 2.0, 0.25]):
        lg = np.array([perm], np.float64)
        for k in range(1, 5):
            ids, _ = oracle.route_topk(lg, k, False)
            assert list(ids[0]) == _brute_topk(perm, k)


def test_topk_ties_lower_index_first_and_signed_zero():
    lg = np.array([[1.0, 3.0, 3.0, -0.0, 0.0, 3.0, 0.0, -1.0]])
    ids, _ = oracle.route_topk(lg, 6, False)
    assert list(ids[0]) == [1, 2, 5, 0, 3, 4]


def test_topk_random_vs_stable_argsort():
    rng = np.random.default_rng(3)
    for E, k in [(64, 6), (60, 4), (16, 2), (256, 8), (8, 8)]:
        lg = rng.standard_normal((33, E)).astype(np.float32)
        lg[:, ::7] = lg[:, :1]  # plant ties
        ids, _ = oracle.route_topk(lg.astype(np.float64), k, False)
        ref = np.argsort(-lg, axis=1, kind="stable")[:, :k]
        assert np.array_equal(ids, ref)


def test_topk_decides_in_fp32():
    # two logits that differ in fp64 but round to the same fp32 value tie
    a = 1.0
    b = 1.0 + 2.0 ** -30
    ids, _ = oracle.route_topk(np.array([[a, b]]), 1, False)
    assert ids[0, 0] == 0


def test_softmax_and_weights_vs_scipy():
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((9, 60)).astype(np.float32).astype(np.float64)
    ids, w, p = oracle.route_topk(lg, 4, False, want_probs=True)
    ref = softmax(lg, axis=1)
    assert np.allclose(p, ref, rtol=1e-13, atol=0)
    assert np.allclose(p.sum(1), 1.0, atol=1e-14)
    assert np.allclose(w, np.take_along_axis(ref, ids, 1), rtol=1e-13)
    ids2, w2 = oracle.route_topk(lg, 4, True)
    assert np.array_equal(ids, ids2)
    assert np.allclose(w2.sum(1), 1.0, atol=1e-14)
    sel = np.take_along_axis(ref, ids, 1)
    assert np.allclose(w2, sel / sel.sum(1, keepdims=True), rtol=1e-13)


def test_renorm_with_k_equal_E_is_softmax():
    rng = np.random.default_rng(6)
    lg = rng.standard_normal((4, 8)).astype(np.float32).astype(np.float64)
    ids, w, p = oracle.route_topk(lg, 8, True, want_probs=True)
    assert np.allclose(w, np.take_along_axis(p, ids, 1), rtol=1e-14)


# --------------------------------------------------------- ELB / gather
def test_elb_counter_sum_and_depth1_golden():
    g = json.load(open(os.path.join(GOLD, "elb_depth1.json")))
    E, k = g["E"], g["k"]
    rng = np.random.default_rng(11)
    L = 3
    elb = np.zeros((L, E), np.uint32)
    expect = np.zeros(L, np.int64)
    for layer in range(L):
        for _ in range(5):
            T = int(rng.integers(1, 18))
            ids, _ = oracle.route_topk(rng.standard_normal((T, E)), k, False)
            oracle.elb_accumulate(elb, layer, ids)
            expect[layer] += T * k
    # sum of increments per layer = (calls) * T * k
    assert np.array_equal(elb.sum(1).astype(np.int64), expect)
    # depth-1 draft step: exactly k distinct experts per layer (the pages' 6.0)
    elb1 = np.zeros((1, E), np.uint32)
    ids, _ = oracle.route_topk(rng.standard_normal((1, E)), k, False)
    oracle.elb_accumulate(elb1, 0, ids)
    assert float(np.count_nonzero(elb1[0])) == g["distinct_experts_per_layer"]
    assert elb1.sum() == k


def test_elb_matches_bincount():
    rng = np.random.default_rng(12)
    E, k, L = 64, 6, 4
    elb = np.zeros((L, E), np.uint32)
    ref = np.zeros((L, E), np.int64)
    for _ in range(20):
        layer = int(rng.integers(0, L))
        T = int(rng.integers(1, 18))
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        oracle.elb_accumulate(elb, layer, ids)
        ref[layer] += np.bincount(ids.reshape(-1), minlength=E)
    assert np.array_equal(elb.astype(np.int64), ref)


@pytest.mark.parametrize("T,k,E", [(1, 6, 64), (17, 6, 64), (9, 4, 60), (17, 2, 16), (4, 2, 8), (3, 8, 8)])
def test_gather_vs_stable_argsort(T, k, E):
    rng = np.random.default_rng(T * 100 + k)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    g = oracle.gather_by_expert(ids, E)
    flat = ids.reshape(-1)
    assert np.array_equal(g["counts"], np.bincount(flat, minlength=E))
    assert g["offsets"][0] == 0 and g["offsets"][E] == T * k
    assert np.array_equal(np.diff(g["offsets"]), g["counts"])
    assert np.array_equal(g["sorted_slots"], np.argsort(flat, kind="stable"))
    act = np.nonzero(g["counts"])[0]
    assert g["n_active"] == len(act)
    assert np.array_equal(g["active"][:len(act)], act)
    # scatter(gather(v)) is the identity
    v = rng.standard_normal(T * k)
    gathered = v[g["sorted_slots"]]
    back = np.empty_like(v)
    back[g["sorted_slots"]] = gathered
    assert np.array_equal(back, v)
    # each expert segment holds only that expert, in ascending slot order
    for e in act:
        seg = g["sorted_slots"][g["offsets"][e]:g["offsets"][e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


def test_gather_all_tokens_on_one_expert():
    ids = np.array([[3], [3], [3], [3]], np.int32)
    g = oracle.gather_by_expert(ids, 8)
    assert g["n_active"] == 1 and g["active"][0] == 3
    assert list(g["sorted_slots"]) == [0, 1, 2, 3]


# ------------------------------------------------------------ dequant
def test_dequant_hand_packed_golden():
    gold = json.load(open(os.path.join(GOLD, "gptq_nibbles.json")))
    for case in gold["cases"]:
        q = np.array([[case["word"]]], np.int32)
        s = np.array([[case["scale"]]], np.float16).view(np.uint16)
        # one word covers rows 0..7; one group row of scales covers 128 rows
        qq = np.zeros((16, 1), np.int32)
        qq[0, 0] = q[0, 0]
        out = oracle.w4_dequant(qq, s)
        assert list(out[:8, 0]) == case["values"]


def test_dequant_every_nibble_position_and_code():
    K, N = 256, 16
    codes = (np.arange(K)[:, None] * 7 + np.arange(N)[None, :] * 3) % 16
    q = np.zeros((K // 8, N), np.uint32)
    for kk in range(K):
        q[kk // 8] |= (codes[kk].astype(np.uint32) << np.uint32(4 * (kk % 8)))
    sc = (np.arange(2 * N, dtype=np.float64).reshape(2, N) + 1) / 64.0
    s = sc.astype(np.float16)
    out = oracle.w4_dequant(q.view(np.int32), s.view(np.uint16))
    ref = (codes - 8) * np.repeat(s.astype(np.float64), 128, axis=0)
    assert np.array_equal(out, ref)
    assert set(np.unique(codes)) == set(range(16))


def _pack_zeros(z):
    """[G][N] zero points -> [G][N/8] int32, column n at bits 4*(n%8), low nibble first."""
    G, N = z.shape
    qz = np.zeros((G, N // 8), np.uint32)
    for n in range(N):
        qz[:, n // 8] |= z[:, n].astype(np.uint32) << np.uint32(4 * (n % 8))
    return qz.view(np.int32)


def test_dequant_zero_points_closed_form():
    """Asymmetric INT4: W = (code - zero) * scale for every nibble position of
    the code word, every zero nibble position and every code / zero value."""
    K, N = 256, 16
    codes = (np.arange(K)[:, None] * 5 + np.arange(N)[None, :] * 3) % 16
    q = np.zeros((K // 8, N), np.uint32)
    for kk in range(K):
        q[kk // 8] |= (codes[kk].astype(np.uint32) << np.uint32(4 * (kk % 8)))
    zeros = (np.arange(2)[:, None] * 9 + np.arange(N)[None, :] * 7) % 16   # [K/128][N]
    sc = ((np.arange(2 * N, dtype=np.float64).reshape(2, N) + 3) / 32.0).astype(np.float16)
    out = oracle.w4_dequant(q.view(np.int32), sc.view(np.uint16), _pack_zeros(zeros))
    ref = (codes - np.repeat(zeros, 128, axis=0)) * np.repeat(sc.astype(np.float64), 128, axis=0)
    assert np.array_equal(out, ref)
    assert set(np.unique(zeros)) == set(range(16)) and set(np.unique(codes)) == set(range(16))
    # all zero points 8 is the symmetric format
    eight = _pack_zeros(np.full((2, N), 8))
    assert np.array_equal(oracle.w4_dequant(q.view(np.int32), sc.view(np.uint16), eight),
                          oracle.w4_dequant(q.view(np.int32), sc.view(np.uint16)))


def test_identity_expert_with_zero_points():
    """Identity expert built on per-column zero points: code z+1 on the
    diagonal, code z elsewhere, so W = I whatever the zero point."""
    n = 256
    z = (np.arange(n) * 5 % 15)[None, :].repeat(n // 128, 0)        # zero point per column, 0..14
    codes = np.repeat(z, 128, axis=0).copy()
    codes[np.arange(n), np.arange(n)] += 1
    q = np.zeros((n // 8, n), np.uint32)
    for kk in range(n):
        q[kk // 8] |= (codes[kk].astype(np.uint32) << np.uint32(4 * (kk % 8)))
    s = np.ones((n // 128, n), np.float16).view(np.uint16)
    qz = _pack_zeros(z)
    ex = dict(qw_gate=q.view(np.int32), s_gate=s, qz_gate=qz, qw_up=q.view(np.int32), s_up=s, qz_up=qz,
              qw_down=q.view(np.int32), s_down=s, qz_down=qz)
    x = (np.random.default_rng(5).standard_normal(n) * 2).astype(np.float16)
    xd = x.astype(np.float64)
    y = oracle.swiglu_w4(x.view(np.uint16), ex)
    assert np.allclose(y, xd * expit(xd) * xd, rtol=1e-14, atol=1e-300)


# ------------------------------------------------------- GGUF Q8_0 draft
def _q8_blocks(codes, d):
    """[N][K] int codes and [N][K/32] fp16 scales -> [N][K/32][34] uint8 Q8_0 blocks."""
    N, K = codes.shape
    out = np.zeros((N, K // 32, 34), np.uint8)
    dv = np.asarray(d, np.float16).view(np.uint16)
    out[:, :, 0] = dv & 0xFF
    out[:, :, 1] = dv >> 8
    out[:, :, 2:] = codes.astype(np.int8).view(np.uint8).reshape(N, K // 32, 32)
    return out


def test_q8_dequant_hand_derived_golden():
    gold = json.load(open(os.path.join(GOLD, "gguf_q8_0.json")))
    cases = gold["cases"]
    w = np.zeros((1, len(cases), 34), np.uint8)
    for b, case in enumerate(cases):
        w[0, b, :2] = case["d_bytes"]
        w[0, b, 2:2 + len(case["code_bytes"])] = case["code_bytes"]
        assert float(np.array(case["d_bytes"], np.uint8).view(np.float16)[0]) == case["d"]
    out = oracle.q8_dequant(w)
    for b, case in enumerate(cases):
        assert list(out[0, 32 * b:32 * b + 8]) == case["values"]
        assert not np.any(out[0, 32 * b + 8:32 * b + 32])


def test_q8_dequant_every_code_and_position():
    """W[n][k] = d[n][k/32] * code[n][k] for every int8 code at every position."""
    N, K = 8, 256
    codes = ((np.arange(N)[:, None] * 37 + np.arange(K)[None, :] * 11) % 256) - 128
    d = ((np.arange(N * K // 32).reshape(N, K // 32) % 13) - 6.5) / 16.0
    out = oracle.q8_dequant(_q8_blocks(codes, d))
    ref = codes * np.repeat(np.asarray(d, np.float16).astype(np.float64), 32, axis=1)
    assert np.array_equal(out, ref)
    assert set(np.unique(codes)) == set(range(-128, 128))


def test_q8_expert_equals_the_same_weights_in_int4():
    """A GPTQ INT4 expert re-expressed exactly in Q8_0 (code q - 8, the group
    scale on each of the group's four blocks) gives the same MLP output, term
    for term: the Q8_0 indexing is pinned to the INT4 one."""
    shape = W.scaled(W.CONFIGS["tiny"], H=256, I=384)
    ex = W.gen_w4_expert(shape, 0, 1)
    q8 = {}
    for name, K in (("gate", shape.H), ("up", shape.H), ("down", shape.I)):
        Wk = oracle.w4_dequant(ex["qw_" + name], ex["s_" + name])          # [K][N]
        s = ex["s_" + name].view(np.float16).astype(np.float64)            # [K/128][N]
        d = np.repeat(s, 4, axis=0).T                                      # [N][K/32]
        codes = np.rint(Wk.T / np.repeat(d, 32, axis=1)).astype(np.int64)  # q - 8, exact
        assert np.array_equal(codes * np.repeat(d, 32, axis=1), Wk.T)
        q8["q8_" + name] = _q8_blocks(codes, d.astype(np.float16))
    for step in range(3):
        x = W.gen_x(shape, 1, step=step)[0]
        y4, h4 = oracle.swiglu_w4(x, ex, want_h=True)
        y8, h8 = oracle.swiglu_q8(x, q8, want_h=True)
        assert np.array_equal(h4, h8) and np.array_equal(y4, y8)


def test_q8_identity_expert_closed_form():
    n = 256
    codes = np.eye(n, dtype=np.int64)
    eye = _q8_blocks(codes, np.ones((n, n // 32)))
    ex = dict(q8_gate=eye, q8_up=eye, q8_down=eye)
    x = (np.random.default_rng(6).standard_normal(n) * 2).astype(np.float16)
    xd = x.astype(np.float64)
    assert np.allclose(oracle.swiglu_q8(x.view(np.uint16), ex), xd * expit(xd) * xd, rtol=1e-14, atol=1e-300)


def test_q8_mlp_matches_dequantised_matmul():
    shape = W.scaled(W.CONFIGS["tiny"], H=256, I=384)
    ex = W.gen_q8_expert(shape, 0, 0)
    x = W.gen_x(shape, 1)[0]
    Wg, Wu, Wd = (oracle.q8_dequant(ex[k]) for k in ("q8_gate", "q8_up", "q8_down"))  # [out][in]
    xd = x.view(np.float16).astype(np.float64)
    g, u = Wg @ xd, Wu @ xd
    ref = Wd @ (g * expit(g) * u)
    assert np.allclose(oracle.swiglu_q8(x, ex), ref, rtol=1e-10, atol=1e-10)


# ------------------------------------------------------- GGUF Q2_K draft
def _q2k_blocks(q, sc, mn, d, dmin):
    """Codes q [N][K] (0..3), sub-block scales and mins [N][K/16] (0..15), fp16
    d and dmin [N][K/256] -> [N][K/256][84] uint8 Q2_K super-blocks (code of
    value w at bits 2*((w%128)//32) of byte 16 + 32*(w//128) + w%32)."""
    N, K = q.shape
    out = np.zeros((N, K // 256, 84), np.uint8)
    out[:, :, :16] = (np.asarray(sc) | (np.asarray(mn) << 4)).reshape(N, K // 256, 16)
    qb = q.reshape(N, K // 256, 256)
    for w in range(256):
        out[:, :, 16 + 32 * (w // 128) + w % 32] |= (qb[:, :, w] << (2 * ((w % 128) // 32))).astype(np.uint8)
    for off, v in ((80, d), (82, dmin)):
        bits = np.asarray(v, np.float16).view(np.uint16)
        out[:, :, off] = bits & 0xFF
        out[:, :, off + 1] = bits >> 8
    return out


def test_q2k_dequant_hand_derived_golden():
    gold = json.load(open(os.path.join(GOLD, "gguf_q2_k.json")))
    blk = np.zeros((1, 1, 84), np.uint8)
    blk[0, 0, :16] = gold["sub_block_bytes"]
    for i, v in gold["code_bytes"].items():
        blk[0, 0, 16 + int(i)] = v
    blk[0, 0, 80:82] = gold["d_bytes"]
    blk[0, 0, 82:84] = gold["dmin_bytes"]
    assert float(np.array(gold["d_bytes"], np.uint8).view(np.float16)[0]) == gold["d"]
    assert float(np.array(gold["dmin_bytes"], np.uint8).view(np.float16)[0]) == gold["dmin"]
    out = oracle.q2k_dequant(blk)[0]
    for w, v in gold["checks"]:
        assert out[w] == v, w


def test_q2k_dequant_every_position_closed_form():
    """d*sc*q - dmin*m at every value position of two super-blocks per row,
    every code, every scale and min nibble."""
    rng = np.random.default_rng(11)
    N, K = 6, 512
    q = rng.integers(0, 4, size=(N, K))
    sc = rng.integers(0, 16, size=(N, K // 16))
    mn = rng.integers(0, 16, size=(N, K // 16))
    d = rng.uniform(0.01, 0.1, size=(N, K // 256)).astype(np.float16)
    dmin = rng.uniform(0.01, 0.1, size=(N, K // 256)).astype(np.float16)
    out = oracle.q2k_dequant(_q2k_blocks(q, sc, mn, d, dmin))
    rep16 = lambda a: np.repeat(a, 16, axis=1)  # noqa: E731
    rep256 = lambda a: np.repeat(np.asarray(a, np.float64), 256, axis=1)  # noqa: E731
    ref = rep256(d) * rep16(sc) * q - rep256(dmin) * rep16(mn)
    assert np.array_equal(out, ref)
    assert set(np.unique(q)) == set(range(4)) and set(np.unique(sc)) == set(range(16))


def test_q2k_expert_equals_its_fp16_copy():
    """Q2_K gate/up and Q8_0 down with power-of-two scales, so every weight is
    exact in fp16: the expert equals the FP16 oracle on those weights term
    for term (both sum in the same order)."""
    rng = np.random.default_rng(12)
    H, I = 512, 256
    ex = {}
    for name in ("gate", "up"):
        q = rng.integers(0, 4, size=(I, H))
        sc = rng.integers(0, 16, size=(I, H // 16))
        mn = rng.integers(0, 16, size=(I, H // 16))
        d = np.full((I, H // 256), 2.0 ** -9)
        dmin = np.full((I, H // 256), 2.0 ** -8)
        ex["q2k_" + name] = _q2k_blocks(q, sc, mn, d, dmin)
    codes = rng.integers(-128, 128, size=(H, I))
    ex["q8_down"] = _q8_blocks(codes, np.full((H, I // 32), 2.0 ** -12))
    f16 = dict(w_gate=oracle.q2k_dequant(ex["q2k_gate"]).astype(np.float16).view(np.uint16),
               w_up=oracle.q2k_dequant(ex["q2k_up"]).astype(np.float16).view(np.uint16),
               w_down=oracle.q8_dequant(ex["q8_down"]).astype(np.float16).view(np.uint16))
    assert np.array_equal(f16["w_gate"].view(np.float16).astype(np.float64), oracle.q2k_dequant(ex["q2k_gate"]))
    shape = W.scaled(W.CONFIGS["tiny"], H=H, I=I)
    for step in range(2):
        x = W.gen_x(shape, 1, step=step)[0]
        y2, h2 = oracle.swiglu_q2k(x, ex, want_h=True)
        y16, h16 = oracle.swiglu_f16(x, f16, want_h=True)
        assert np.array_equal(h2, h16) and np.array_equal(y2, y16)


def test_q2k_identity_expert_closed_form():
    n = 256
    q = np.eye(n, dtype=np.int64)
    one = np.ones((n, n // 16), np.int64)
    gu = _q2k_blocks(q, one, 0 * one, np.ones((n, 1)), np.ones((n, 1)))
    ex = dict(q2k_gate=gu, q2k_up=gu, q8_down=_q8_blocks(np.eye(n, dtype=np.int64), np.ones((n, n // 32))))
    x = (np.random.default_rng(13).standard_normal(n) * 2).astype(np.float16)
    xd = x.astype(np.float64)
    assert np.allclose(oracle.swiglu_q2k(x.view(np.uint16), ex), xd * expit(xd) * xd, rtol=1e-14, atol=1e-300)


# ------------------------------------------------------- GGUF Q4_K draft
def _q4k_scale_bytes(sc, mn):
    """8 six-bit scales and mins -> the 12 bytes of a Q4_K super-block."""
    b = np.zeros(12, np.int64)
    for s in range(4):
        b[s] = (sc[s] & 63) | ((sc[s + 4] >> 4) << 6)
        b[s + 4] = (mn[s] & 63) | ((mn[s + 4] >> 4) << 6)
        b[s + 8] = (sc[s + 4] & 15) | ((mn[s + 4] & 15) << 4)
    return b.astype(np.uint8)


def _q4k_blocks(q, sc, mn, d, dmin):
    """Codes q [N][K] (0..15), sub-block scales and mins [N][K/32] (0..63), fp16
    d and dmin [N][K/256] -> [N][K/256][144] uint8 Q4_K super-blocks."""
    N, K = q.shape
    out = np.zeros((N, K // 256, 144), np.uint8)
    for n in range(N):
        for b in range(K // 256):
            out[n, b, 4:16] = _q4k_scale_bytes(sc[n, 8 * b:8 * b + 8], mn[n, 8 * b:8 * b + 8])
    qb = q.reshape(N, K // 256, 256)
    for w in range(256):
        sh = 0 if w % 64 < 32 else 4
        out[:, :, 16 + 32 * (w // 64) + w % 32] |= (qb[:, :, w] << sh).astype(np.uint8)
    for off, v in ((0, d), (2, dmin)):
        bits = np.asarray(v, np.float16).view(np.uint16)
        out[:, :, off] = bits & 0xFF
        out[:, :, off + 1] = bits >> 8
    return out


def test_q4k_dequant_hand_derived_golden():
    gold = json.load(open(os.path.join(GOLD, "gguf_q4_k.json")))
    blk = np.zeros((1, 1, 144), np.uint8)
    blk[0, 0, 0:2] = gold["d_bytes"]
    blk[0, 0, 2:4] = gold["dmin_bytes"]
    blk[0, 0, 4:16] = gold["scale_bytes"]
    for i, v in gold["code_bytes"].items():
        blk[0, 0, 16 + int(i)] = v
    assert list(_q4k_scale_bytes(np.array(gold["scales"]), np.array(gold["mins"]))) == gold["scale_bytes"]
    out = oracle.q4k_dequant(blk)[0]
    for w, v in gold["checks"]:
        assert out[w] == v, w


def test_q4k_dequant_every_position_closed_form():
    """d*scale*q - dmin*min at every value position, every code, scales and
    mins over the full 6-bit range in every sub-block slot."""
    rng = np.random.default_rng(21)
    N, K = 6, 512
    q = rng.integers(0, 16, size=(N, K))
    sc = rng.integers(0, 64, size=(N, K // 32))
    mn = rng.integers(0, 64, size=(N, K // 32))
    d = rng.uniform(0.01, 0.1, size=(N, K // 256)).astype(np.float16)
    dmin = rng.uniform(0.01, 0.1, size=(N, K // 256)).astype(np.float16)
    out = oracle.q4k_dequant(_q4k_blocks(q, sc, mn, d, dmin))
    rep32 = lambda a: np.repeat(a, 32, axis=1)  # noqa: E731
    rep256 = lambda a: np.repeat(np.asarray(a, np.float64), 256, axis=1)  # noqa: E731
    ref = rep256(d) * rep32(sc) * q - rep256(dmin) * rep32(mn)
    assert np.array_equal(out, ref)
    assert set(np.unique(q)) == set(range(16)) and sc.max() == 63 and mn.min() == 0


def test_q4k_expert_equals_its_fp16_copy():
    """Q4_K gate/up and Q8_0 down with power-of-two scales (every weight exact
    in fp16) equal the FP16 oracle on those weights term for term."""
    rng = np.random.default_rng(22)
    H, I = 512, 256
    ex = {}
    for name in ("gate", "up"):
        q = rng.integers(0, 16, size=(I, H))
        sc = rng.integers(0, 64, size=(I, H // 32))
        mn = rng.integers(0, 64, size=(I, H // 32))
        ex["q4k_" + name] = _q4k_blocks(q, sc, mn, np.full((I, H // 256), 2.0 ** -12), np.full((I, H // 256), 2.0 ** -8))
    ex["q8_down"] = _q8_blocks(rng.integers(-128, 128, size=(H, I)), np.full((H, I // 32), 2.0 ** -12))
    f16 = dict(w_gate=oracle.q4k_dequant(ex["q4k_gate"]).astype(np.float16).view(np.uint16),
               w_up=oracle.q4k_dequant(ex["q4k_up"]).astype(np.float16).view(np.uint16),
               w_down=oracle.q8_dequant(ex["q8_down"]).astype(np.float16).view(np.uint16))
    assert np.array_equal(f16["w_up"].view(np.float16).astype(np.float64), oracle.q4k_dequant(ex["q4k_up"]))
    shape = W.scaled(W.CONFIGS["tiny"], H=H, I=I)
    for step in range(2):
        x = W.gen_x(shape, 1, step=step)[0]
        y4, h4 = oracle.swiglu_q4k(x, ex, want_h=True)
        y16, h16 = oracle.swiglu_f16(x, f16, want_h=True)
        assert np.array_equal(h4, h16) and np.array_equal(y4, y16)


# ---------------------------------------------------------------- MLP
def _identity_w4(n):
    q = np.full((n // 8, n), 0x88888888, np.uint32)
    for i in range(n):
        word = q[i // 8, i]
        sh = np.uint32(4 * (i % 8))
        q[i // 8, i] = (word & ~(np.uint32(15) << sh)) | (np.uint32(9) << sh)
    s = np.ones((n // 128, n), np.float16).view(np.uint16)
    return q.view(np.int32), s


def test_identity_expert_closed_form():
    n = 256
    q, s = _identity_w4(n)
    ex = dict(qw_gate=q, s_gate=s, qw_up=q, s_up=s, qw_down=q, s_down=s)
    x = (np.random.default_rng(1).standard_normal(n) * 2).astype(np.float16)
    xd = x.astype(np.float64)
    ref = xd * expit(xd) * xd  # silu(x) * x through identity gate/up/down
    y = oracle.swiglu_w4(x.view(np.uint16), ex)
    assert np.allclose(y, ref, rtol=1e-14, atol=1e-300)
    eye = np.eye(n).astype(np.float16).view(np.uint16)
    y16 = oracle.swiglu_f16(x.view(np.uint16), dict(w_gate=eye, w_up=eye, w_down=eye))
    assert np.allclose(y16, ref, rtol=1e-14, atol=1e-300)


def test_f16_mlp_is_textbook_swiglu_via_matmul():
    rng = np.random.default_rng(2)
    H, I = 128, 96
    wg = (rng.standard_normal((I, H)) * 0.1).astype(np.float16)
    wu = (rng.standard_normal((I, H)) * 0.1).astype(np.float16)
    wd = (rng.standard_normal((H, I)) * 0.1).astype(np.float16)
    x = rng.standard_normal(H).astype(np.float16)
    g = wg.astype(np.float64) @ x.astype(np.float64)
    u = wu.astype(np.float64) @ x.astype(np.float64)
    ref = wd.astype(np.float64) @ (g * expit(g) * u)
    y = oracle.swiglu_f16(x.view(np.uint16), dict(w_gate=wg.view(np.uint16), w_up=wu.view(np.uint16),
                                                  w_down=wd.view(np.uint16)))
    assert np.allclose(y, ref, rtol=1e-10, atol=1e-12)


def test_w4_mlp_matches_dequantised_matmul():
    shape = W.scaled(W.CONFIGS["tiny"], H=256, I=384)
    ex = W.gen_w4_expert(shape, 0, 0)
    x = W.gen_x(shape, 1)[0]
    Wg = oracle.w4_dequant(ex["qw_gate"], ex["s_gate"])   # [H, I]
    Wu = oracle.w4_dequant(ex["qw_up"], ex["s_up"])
    Wd = oracle.w4_dequant(ex["qw_down"], ex["s_down"])   # [I, H]
    xd = x.view(np.float16).astype(np.float64)
    g, u = xd @ Wg, xd @ Wu
    ref = (g * expit(g) * u) @ Wd
    y = oracle.swiglu_w4(x, ex)
    assert np.allclose(y, ref, rtol=1e-10, atol=1e-10)


def test_shared_gate_vs_expit():
    rng = np.random.default_rng(4)
    x = rng.standard_normal(256).astype(np.float16)
    w = (rng.standard_normal(256) * 0.05).astype(np.float16)
    ref = expit(float(x.astype(np.float64) @ w.astype(np.float64)))
    assert abs(oracle.shared_gate(x.view(np.uint16), w.view(np.uint16)) - ref) < 1e-15


# ------------------------------------------------------------- combine
def test_combine_closed_form_and_rounding():
    rng = np.random.default_rng(8)
    T, k, H = 3, 2, 16
    w = rng.random((T, k))
    y = rng.standard_normal((T, k, H))
    sh = rng.standard_normal((T, H))
    gam = rng.random(T)
    out, outh = oracle.combine(w, y, gam, sh)
    ref = w[:, 0, None] * y[:, 0] + w[:, 1, None] * y[:, 1] + gam[:, None] * sh
    assert np.allclose(out, ref, rtol=1e-15, atol=1e-15)
    assert np.array_equal(outh, out.astype(np.float16).view(np.uint16))
    out2, _ = oracle.combine(w, y)
    assert np.allclose(out2, ref - gam[:, None] * sh, rtol=1e-14, atol=1e-14)


# --------------------------------------------------------------- layer
def _tiny_layer(mode, relabel=None):
    shape = W.CONFIGS["tiny"]
    x = W.gen_x(shape, shape.T_draft)
    wr = W.gen_router(shape)
    perm = np.arange(shape.E) if relabel is None else relabel
    wr_p = np.empty_like(wr)
    wr_p[perm] = wr           # expert e is stored under label perm[e]
    inv = np.argsort(perm)

    def expert(lbl):
        ex = W.gen_w4_expert(shape, 0, int(inv[lbl]))
        return ex if mode == "draft" else oracle.f16_copy_of_w4(ex)
    return oracle.moe_layer(mode, x, shape.k, shape.renorm, expert, shape.E, w_router=wr_p)


def test_layer_invariant_under_expert_relabelling():
    # expert-wise reordering is "mathematically identical": relabelling experts
    # changes the gather order but not the output
    base = _tiny_layer("draft")
    perm = np.random.default_rng(9).permutation(W.CONFIGS["tiny"].E)
    other = _tiny_layer("draft", perm)
    assert np.array_equal(base["out_half"], other["out_half"])
    assert np.array_equal(perm[base["ids"]], other["ids"])


def test_single_expert_layer_is_plain_swiglu():
    shape = W.scaled(W.CONFIGS["tiny"], E=1, k=1, I=256)
    ex = W.gen_w4_expert(shape, 0, 0)
    x = W.gen_x(shape, 3)
    res = oracle.moe_layer("draft", x, 1, True, lambda e: ex, 1, logits=np.zeros((3, 1), np.float32))
    Wg = oracle.w4_dequant(ex["qw_gate"], ex["s_gate"])
    Wu = oracle.w4_dequant(ex["qw_up"], ex["s_up"])
    Wd = oracle.w4_dequant(ex["qw_down"], ex["s_down"])
    xd = x.view(np.float16).astype(np.float64)
    g, u = xd @ Wg, xd @ Wu
    ref = (g * expit(g) * u) @ Wd
    assert np.allclose(res["out"], ref, rtol=1e-10, atol=1e-10)
    assert np.all(res["w"] == 1.0)


def test_tiny_draft_and_verify_agree_within_weight_rounding():
    d = _tiny_layer("draft")
    v = _tiny_layer("verify")
    assert np.array_equal(d["ids"], v["ids"])
    ref = d["out"]
    err = np.abs(v["out"] - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max()
    assert err.sum() / np.abs(ref).sum() <= 1e-3


def test_gated_shared_expert_in_layer():
    shape = W.scaled(W.CONFIGS["qwen15_moe"], H=256, I=128, E=8, k=2, I_s=256)
    x = W.gen_x(shape, 2)
    sh = W.gen_shared(shape)
    lg = np.zeros((2, 8), np.float32)
    lg[:, 0] = 5.0
    lg[:, 1] = 4.0

    def expert(e):
        return W.gen_w4_expert(shape, 0, e)
    res = oracle.moe_layer("draft", x, 2, False, expert, 8, logits=lg, shared=sh)
    for t in range(2):
        gam = expit(float(x[t].view(np.float16).astype(np.float64) @ sh["w_sgate"].view(np.float16).astype(np.float64)))
        ys = [oracle.swiglu_w4(x[t], expert(e)) for e in (0, 1)]
        ref = res["w"][t, 0] * ys[0] + res["w"][t, 1] * ys[1] + gam * oracle.swiglu_f16(x[t], sh)
        assert np.allclose(res["out"][t], ref, rtol=1e-12, atol=1e-12)
