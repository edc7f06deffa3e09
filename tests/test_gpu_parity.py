"""GPU parity: every C-ABI call of libspx against the CPU oracle on the same
seeded inputs.  Routing ids, counters and gathers must be bit-exact; fp32 /
fp16 outputs within the tolerance in gpu_helpers (max err <= 1e-2 max|ref|,
mean relative error <= 1e-3)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import spx_workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from quantized_expert_gb300 import build, spx
    build.build()
    spx.load()
    yield


def _spx():
    from quantized_expert_gb300 import spx
    return spx


def _gh():
    import gpu_helpers
    return gpu_helpers


# ------------------------------------------------------------------ routing
@pytest.mark.parametrize("E,k,T,renorm", [(64, 6, 17, False), (64, 6, 1, False), (60, 4, 9, False),
                                          (16, 2, 17, True), (8, 2, 4, True), (8, 8, 3, True), (256, 8, 64, False),
                                          (1, 1, 5, True)])
def test_route_topk_given_logits(E, k, T, renorm):
    spx, gh = _spx(), _gh()
    rng = np.random.default_rng(E * 100 + T)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[:, ::5] = lg[:, :1]           # exact ties across experts
    lg[0, :] = 0.0                    # an all-tie row
    lg[min(1, T - 1), ::2] = -0.0     # signed zeros tie with +0.0
    ids_ref, w_ref = oracle.route_topk(lg.astype(np.float64), k, renorm)
    d_lg = gh.dev(lg)
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    ws = spx.new_workspace(T, 128)
    spx.spx_route_topk(None, None, d_lg, T, 128, E, k, renorm, ids, w, ws)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("name", ["tiny", "qwen15_moe"])
def test_route_router_product(name):
    spx, gh = _spx(), _gh()
    s = W.CONFIGS[name]
    wr = W.gen_router(s)
    for T in sorted({s.T_draft, s.T_verify}):
        x = W.gen_x(s, T)
        lg_ref = oracle.router_logits(x, wr)
        ids_ref, w_ref = oracle.route_topk(lg_ref, s.k, s.renorm)
        lg = torch.empty(T, s.E, dtype=torch.float32, device="cuda")
        ids = torch.empty(T, s.k, dtype=torch.int32, device="cuda")
        w = torch.empty(T, s.k, dtype=torch.float32, device="cuda")
        ws = spx.new_workspace(T, s.H)
        for rep in range(2):  # the completion ticket must reset itself
            spx.spx_route_topk(gh.dev_f16(x), gh.dev_f16(wr), lg, T, s.H, s.E, s.k, s.renorm, ids, w, ws)
            torch.cuda.synchronize()
            lg_g = lg.cpu().numpy().astype(np.float64)
            assert np.allclose(lg_g, lg_ref, rtol=1e-5, atol=1e-5 * np.abs(lg_ref).max())
            srt = np.sort(lg_ref.astype(np.float32), axis=1)[:, ::-1]
            margin = (srt[:, s.k - 1] - srt[:, s.k]).min()
            assert margin > 1e-4, "seeded inputs have a near-tie at the top-k boundary"
            assert np.array_equal(ids.cpu().numpy(), ids_ref)
            assert np.allclose(w.cpu().numpy(), w_ref, rtol=1e-5)


def test_elb_and_gather_bit_exact():
    spx, gh = _spx(), _gh()
    rng = np.random.default_rng(21)
    L, E, k = 26, 64, 6
    elb = torch.zeros(L, E, dtype=torch.int32, device="cuda")
    elb_ref = np.zeros((L, E), np.uint32)
    for it in range(40):
        layer = int(rng.integers(0, L))
        T = int(rng.integers(1, 65))
        kk = int(rng.integers(1, 9))
        Ee = int(rng.integers(kk, 257))
        ids_np = np.stack([rng.choice(Ee, kk, replace=False) for _ in range(T)]).astype(np.int32)
        g_ref = oracle.gather_by_expert(ids_np, Ee)
        ids = gh.dev(ids_np)
        counts = torch.empty(Ee, dtype=torch.int32, device="cuda")
        offsets = torch.empty(Ee + 1, dtype=torch.int32, device="cuda")
        ss = torch.empty(T * kk, dtype=torch.int32, device="cuda")
        act = torch.empty(Ee, dtype=torch.int32, device="cuda")
        na = torch.empty(1, dtype=torch.int32, device="cuda")
        spx.spx_gather_by_expert(ids, Ee, counts, offsets, ss, act, na)
        if Ee == E:
            spx.spx_elb_accumulate(elb, layer, ids)
            oracle.elb_accumulate(elb_ref, layer, ids_np)
        torch.cuda.synchronize()
        assert np.array_equal(counts.cpu().numpy(), g_ref["counts"])
        assert np.array_equal(offsets.cpu().numpy(), g_ref["offsets"])
        assert np.array_equal(ss.cpu().numpy(), g_ref["sorted_slots"])
        assert int(na.item()) == g_ref["n_active"]
        assert np.array_equal(act.cpu().numpy()[:g_ref["n_active"]], g_ref["active"][:g_ref["n_active"]])
        assert np.all(act.cpu().numpy()[g_ref["n_active"]:] == -1)
    assert np.array_equal(elb.cpu().numpy().astype(np.uint32), elb_ref)
    # read (device and pinned host destinations) and reset
    host = torch.empty(L, E, dtype=torch.int32).pin_memory()
    spx.spx_elb_read(elb, host)
    torch.cuda.synchronize()
    assert np.array_equal(host.numpy().astype(np.uint32), elb_ref)
    spx.spx_elb_reset(elb)
    torch.cuda.synchronize()
    assert int(elb.abs().sum().item()) == 0


# ------------------------------------------------------------ expert calls
def _routing_dev(ids_np, E):
    gh = _gh()
    g = oracle.gather_by_expert(ids_np, E)
    return g, dict(offsets=gh.dev(g["offsets"]), sorted_slots=gh.dev(g["sorted_slots"]),
                   active=gh.dev(g["active"].astype(np.int32)), n_active=gh.dev(np.array([g["n_active"]], np.int32)))


def _small(name, **kw):
    return W.scaled(W.CONFIGS[name], **kw)


SMALL_CASES = [
    # (shape, T, slice_cols): several tiles, ragged token tiles, both slice widths
    (_small("tiny"), 4, 32),
    (_small("tiny"), 4, 16),
    (_small("deepseek_v2_lite", I=256, E=16), 1, 32),
    (_small("deepseek_v2_lite", I=256, E=16), 17, 32),
    (_small("deepseek_v2_lite", I=256, E=16), 8, 16),    # 8 tokens, 16-column slices: the expert launch's 1-tile instance
    (_small("qwen15_moe", I=384, E=12, I_s=512), 9, 16),
    (_small("phi35_moe", H=1024, I=512), 17, 16),
    (_small("phi35_moe", H=1024, I=512, k=2), 33, 16),   # > 24 tokens: 64-token kernel
    (_small("deepseek_v2_lite", H=256, I=128, E=8, k=8), 64, 16),  # k = E, maximum T
    (_small("deepseek_v2_lite", I=256, E=16), 5, 16),    # the draft launch's largest call
]


@pytest.mark.parametrize("case", range(len(SMALL_CASES)))
def test_draft_and_verify_unit_calls(case):
    spx, gh = _spx(), _gh()
    s, T, S = SMALL_CASES[case]
    x = W.gen_x(s, T, step=case)
    rng = np.random.default_rng(case)
    lg = rng.standard_normal((T, s.E)).astype(np.float64)
    ids, w = oracle.route_topk(lg, s.k, s.renorm)
    lay = gh.Layer(s, needed=sorted(set(ids.reshape(-1).tolist())), slice_cols=S)
    g, r = _routing_dev(ids, s.E)
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    dx = gh.dev_f16(x)
    for mode in ("draft", "verify"):
        mlp = oracle.swiglu_w4 if mode == "draft" else oracle.swiglu_f16
        host = lay.w4_host if mode == "draft" else lay.f16_host
        y_ref = np.stack([mlp(x[int(sl) // s.k], host[int(ids.reshape(-1)[sl])]) for sl in g["sorted_slots"]])
        y = torch.empty(T * s.k, s.H, dtype=torch.float32, device="cuda")
        for rep in range(2):  # queue counters and scratch must reset themselves
            if mode == "draft":
                spx.spx_moe_draft_w4a16(dx, lay.w4, s.k, r["offsets"], r["sorted_slots"], r["active"],
                                        r["n_active"], y, ws)
            else:
                spx.spx_moe_verify_fp16(dx, lay.f16, s.k, r["offsets"], r["sorted_slots"], r["active"],
                                        r["n_active"], y, ws)
            torch.cuda.synchronize()
            gh.check_close(y.cpu().numpy(), y_ref, f"{mode} case {case} rep {rep}")
        assert spx.spx_workspace_status(ws) == 0


def test_verify_unit_call_one_group():
    """Wide activations (T = 20, H = 4096) leave room for one consumer group
    only: FP16 slices then reduce through the shared-memory buffer."""
    spx, gh = _spx(), _gh()
    s = _small("phi35_moe", H=4096, I=256, E=4, k=2)
    T = 20
    x = W.gen_x(s, T, step=20)
    lg = np.random.default_rng(20).standard_normal((T, s.E))
    ids, w = oracle.route_topk(lg, s.k, s.renorm)
    lay = gh.Layer(s, needed=sorted(set(ids.reshape(-1).tolist())), draft=False)
    g, r = _routing_dev(ids, s.E)
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k)
    y_ref = np.stack([oracle.swiglu_f16(x[int(sl) // s.k], lay.f16_host[int(ids.reshape(-1)[sl])])
                      for sl in g["sorted_slots"]])
    y = torch.empty(T * s.k, s.H, dtype=torch.float32, device="cuda")
    for rep in range(2):
        spx.spx_moe_verify_fp16(gh.dev_f16(x), lay.f16, s.k, r["offsets"], r["sorted_slots"], r["active"],
                                r["n_active"], y, ws)
        torch.cuda.synchronize()
        gh.check_close(y.cpu().numpy(), y_ref, f"one group rep {rep}")
    assert spx.spx_workspace_status(ws) == 0


def test_draft_wide_slices_reject_many_tokens():
    """INT4 slices of 32 columns serve at most 24 tokens per expert; more is an
    explicit SPX_ERR_UNSUPPORTED (pack with slice_cols=16 for such batches)."""
    spx, gh = _spx(), _gh()
    from quantized_expert_gb300.spx import SpxError
    s = _small("phi35_moe", H=256, I=256, E=4, k=2)
    T = 25
    ids = np.array([[0, 1]] * T, np.int32)
    lay = gh.Layer(s, needed=[0, 1], verify=False, slice_cols=32)
    g, r = _routing_dev(ids, s.E)
    y = torch.empty(T * s.k, s.H, device="cuda")
    with pytest.raises(SpxError) as ei:
        spx.spx_moe_draft_w4a16(gh.dev_f16(W.gen_x(s, T)), lay.w4, s.k, r["offsets"], r["sorted_slots"],
                                r["active"], r["n_active"], y, spx.new_workspace(T, s.H, s.I, s.E, s.k))
    assert ei.value.status == spx.SPX_ERR_UNSUPPORTED


@pytest.mark.parametrize("gated", [False, True])
def test_combine_with_shared(gated):
    spx, gh = _spx(), _gh()
    s = _small("qwen15_moe", I=256, E=8, I_s=512, shared_gate=gated)
    T = 9
    x = W.gen_x(s, T)
    sh = W.gen_shared(s)
    rng = np.random.default_rng(3)
    ids, w = oracle.route_topk(rng.standard_normal((T, s.E)), s.k, False)
    g = oracle.gather_by_expert(ids, s.E)
    y_slot = rng.standard_normal((T * s.k, s.H))
    gamma = np.array([oracle.shared_gate(x[t], sh["w_sgate"]) for t in range(T)]) if gated else None
    shv = np.stack([oracle.swiglu_f16(x[t], sh) for t in range(T)])
    _, ref = oracle.combine(w, y_slot.reshape(T, s.k, s.H), gamma, shv)
    packed = spx.pack_shared(gh.dev_f16(sh["w_gate"]), gh.dev_f16(sh["w_up"]), gh.dev_f16(sh["w_down"]),
                             gh.dev_f16(sh["w_sgate"]) if gated else None)
    ysorted = gh.dev(y_slot[g["sorted_slots"]].astype(np.float32))
    out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    ws = spx.new_workspace(T, s.H)
    for rep in range(2):
        spx.spx_combine(ysorted, gh.dev(g["sorted_slots"]), gh.dev(w.astype(np.float32)), gh.dev_f16(x), packed,
                        T, s.H, s.k, out, ws)
        torch.cuda.synchronize()
        gh.check_close(gh.f16_out(out), ref.view(np.float16).astype(np.float64), f"combine rep {rep}")
    # without a shared expert the combine is the weighted sum alone
    _, ref2 = oracle.combine(w, y_slot.reshape(T, s.k, s.H))
    spx.spx_combine(ysorted, gh.dev(g["sorted_slots"]), gh.dev(w.astype(np.float32)), gh.dev_f16(x), None,
                    T, s.H, s.k, out, ws)
    torch.cuda.synchronize()
    gh.check_close(gh.f16_out(out), ref2.view(np.float16).astype(np.float64), "combine no shared")


# --------------------------------------------------------------- composite
def _run_layer(lay, mode, x, logits, elb=None):
    spx, gh = _spx(), _gh()
    s = lay.shape
    T = x.shape[0]
    routing = spx.Routing.empty(T, s.E, s.k)
    out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    d_lg = gh.dev(np.asarray(logits, np.float32)) if logits is not None else torch.empty(
        T, s.E, dtype=torch.float32, device="cuda")
    args, keep = spx.layer_args(0 if mode == "draft" else 1, gh.dev_f16(x), s.E, s.k, s.renorm, d_lg, routing, out,
                                ws, w4=lay.w4, f16=lay.f16, shared=lay.shared, w_router=lay.w_router, elb=elb,
                                layer=lay.layer, gguf=lay.gguf)
    outs = []
    for rep in range(2):
        spx.spx_moe_layer(args, None)
        torch.cuda.synchronize()
        outs.append(gh.f16_out(out))
    assert spx.spx_workspace_status(ws) == 0
    return outs, routing, d_lg


@pytest.mark.parametrize("name", ["tiny", "deepseek_v2_lite", "qwen15_moe", "phi35_moe"])
@pytest.mark.parametrize("mode", ["draft", "verify"])
def test_layer_full_size(name, mode):
    """The five configurations' layer shapes at full size, through spx_moe_layer."""
    gh = _gh()
    s = W.CONFIGS[name]
    T = s.T_draft if mode == "draft" else s.T_verify
    if name == "tiny":
        T = 4
    x = W.gen_x(s, T, which=int(mode == "verify"))
    logits = None if s.logits == "router" else W.gen_logits(s, T, which=int(mode == "verify"))
    need = gh.needed_experts(s, [logits], [x])
    lay = gh.Layer(s, needed=need, draft=(mode == "draft"), verify=(mode == "verify"))
    ref = lay.oracle_layer(mode, x, logits=logits)
    outs, routing, d_lg = _run_layer(lay, mode, x, logits)
    assert np.array_equal(routing.topk_ids.cpu().numpy(), ref["ids"])
    g = ref["gather"]
    assert np.array_equal(routing.offsets.cpu().numpy(), g["offsets"])
    assert np.array_equal(routing.sorted_slots.cpu().numpy(), g["sorted_slots"])
    for rep, o in enumerate(outs):
        gh.check_close(o, ref["out_half"].view(np.float16).astype(np.float64), f"{name} {mode} rep {rep}")


@pytest.mark.parametrize("E,k", [(256, 8), (64, 40), (33, 33), (16, 1)])
def test_draft_layer_routing_extremes(E, k):
    """One-token draft layers at the routing's edges: 256 experts (the wide
    selection instance), more than 32 selections (the general table builder),
    every expert selected, a single selection; routing outputs bit-exact
    (ids, offsets, sorted slots), output within tolerance of the oracle."""
    gh = _gh()
    s = _small("deepseek_v2_lite", H=256, I=128, E=E, k=k, I_s=256)
    T = 1
    x = W.gen_x(s, T, step=170 + E + k)
    logits = W.gen_logits(s, T, step=170 + E + k)
    lay = gh.Layer(s, needed=gh.needed_experts(s, [logits], [x]), verify=False, slice_cols=16)
    ref = lay.oracle_layer("draft", x, logits=logits)
    outs, routing, _ = _run_layer(lay, "draft", x, logits)
    assert np.array_equal(routing.topk_ids.cpu().numpy(), ref["ids"])
    g = ref["gather"]
    assert np.array_equal(routing.offsets.cpu().numpy(), g["offsets"])
    assert np.array_equal(routing.sorted_slots.cpu().numpy(), g["sorted_slots"])
    for rep, o in enumerate(outs):
        gh.check_close(o, ref["out_half"].view(np.float16).astype(np.float64), f"E={E} k={k} rep {rep}")


@pytest.mark.parametrize("T", [1, 9, 17])
def test_verify_layer_odd_slice_count(T):
    """Verify layer whose shared expert is an odd number of 16-column slices
    (I_s = 272): the launch streams FP16 slices in pairs, so the shared
    expert's last slice stands alone (routed widths are multiples of 128)."""
    gh = _gh()
    s = _small("qwen15_moe", H=512, I=384, E=6, k=2, I_s=272, shared_gate=True)
    x = W.gen_x(s, T, step=T, which=1)
    need = gh.needed_experts(s, None, [x])
    lay = gh.Layer(s, needed=need, draft=False)
    ref = lay.oracle_layer("verify", x)
    outs, routing, _ = _run_layer(lay, "verify", x, None)
    assert np.array_equal(routing.topk_ids.cpu().numpy(), ref["ids"])
    for rep, o in enumerate(outs):
        gh.check_close(o, ref["out_half"].view(np.float16).astype(np.float64), f"odd slices T={T} rep {rep}")


@pytest.mark.parametrize("T", [2, 8])
def test_draft_layer_gated_shared_many_tokens(T):
    """Draft layer through the split-K draft launch with T tokens, a gated
    shared expert and a router product (Qwen-shaped, reduced sizes)."""
    gh = _gh()
    s = _small("qwen15_moe", I=384, E=12, I_s=768)
    x = W.gen_x(s, T, step=T)
    need = gh.needed_experts(s, None, [x])
    lay = gh.Layer(s, needed=need, verify=False)
    ref = lay.oracle_layer("draft", x)
    outs, routing, _ = _run_layer(lay, "draft", x, None)
    assert np.array_equal(routing.topk_ids.cpu().numpy(), ref["ids"])
    for rep, o in enumerate(outs):
        gh.check_close(o, ref["out_half"].view(np.float16).astype(np.float64), f"draft T={T} rep {rep}")


def test_tiny_draft_matches_verify_on_gpu():
    """Tiny layer: verify weights are FP16 copies of the dequantised draft
    weights, so the two paths agree within the weights' fp16 rounding."""
    gh = _gh()
    s = W.CONFIGS["tiny"]
    x = W.gen_x(s, 4)
    lay = gh.Layer(s)
    d, _, _ = _run_layer(lay, "draft", x, None)
    v, _, _ = _run_layer(lay, "verify", x, None)
    gh.check_close(v[0], d[0], "tiny draft vs verify")


def test_layer_elb_counts_draft_steps():
    spx, gh = _spx(), _gh()
    s = _small("deepseek_v2_lite", I=128)
    L = 3
    elb = torch.zeros(L, s.E, dtype=torch.int32, device="cuda")
    elb_ref = np.zeros((L, s.E), np.uint32)
    lays = [gh.Layer(s, layer=l, needed=None, verify=False) for l in range(L)]
    for step in range(1, 5):
        for l in range(L):
            x = W.gen_x(s, 1, layer=l, step=step)
            lg = W.draft_logits(s, l, step)
            ref = lays[l].oracle_layer("draft", x, logits=lg, elb=elb_ref)
            routing = spx.Routing.empty(1, s.E, s.k)
            out = torch.empty(1, s.H, dtype=torch.float16, device="cuda")
            ws = spx.new_workspace(1, s.H, s.I, s.E, s.k, s.I_s)
            args, keep = spx.layer_args(0, gh.dev_f16(x), s.E, s.k, s.renorm, gh.dev(lg), routing, out, ws,
                                        w4=lays[l].w4, shared=lays[l].shared, elb=elb, layer=l)
            spx.spx_moe_layer(args)
            torch.cuda.synchronize()
            gh.check_close(gh.f16_out(out), ref["out_half"].view(np.float16).astype(np.float64), f"elb step {step}")
    assert np.array_equal(elb.cpu().numpy().astype(np.uint32), elb_ref)
    assert np.all(elb.cpu().numpy().sum(1) == 4 * s.k)


def test_invalid_arguments_rejected():
    spx, gh = _spx(), _gh()
    from quantized_expert_gb300.spx import SpxError
    ws = spx.new_workspace(4, 256)
    lg = torch.zeros(4, 8, device="cuda")
    ids = torch.empty(4, 9, dtype=torch.int32, device="cuda")
    w = torch.empty(4, 9, device="cuda")
    with pytest.raises(SpxError) as ei:
        spx.spx_route_topk(None, None, lg, 4, 256, 8, 9, 0, ids, w, ws)   # k > E
    assert ei.value.status == spx.SPX_ERR_INVALID_ARG
    with pytest.raises(SpxError) as ei:
        spx.spx_route_topk(None, None, lg, 65, 256, 8, 2, 0, ids, w, ws)  # T > 64
    assert ei.value.status == spx.SPX_ERR_UNSUPPORTED
    small_ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    x = torch.zeros(4, 256, dtype=torch.float16, device="cuda")
    y = torch.zeros(8, 256, device="cuda")
    z = torch.zeros(9, dtype=torch.int32, device="cuda")
    p = spx.PackedF16(torch.zeros(16, dtype=torch.uint8, device="cuda"), 8, 256, 512)
    with pytest.raises(SpxError) as ei:
        spx.spx_moe_verify_fp16(x, p, 2, z, z, z, z, y, small_ws)
    assert ei.value.status == spx.SPX_ERR_WORKSPACE
    p_bad = spx.PackedF16(torch.zeros(16, dtype=torch.uint8, device="cuda"), 8, 200, 512)  # H % 128 != 0
    with pytest.raises(SpxError) as ei:
        spx.spx_moe_verify_fp16(torch.zeros(4, 200, dtype=torch.float16, device="cuda"), p_bad, 2, z, z, z, z, y, ws)
    assert ei.value.status == spx.SPX_ERR_UNSUPPORTED


def test_chained_layer_calls_back_to_back():
    """Layer calls back to back on one stream, each taking the previous call's
    output as its activations and sharing its workspace (a launch may start
    before the one it follows has finished, so it must not read activations,
    routing or workspace before then).  Draft calls at T = 1 (draft launch)
    and T = 9 (routing + expert launch), verify calls at T = 9; each call is
    checked against the oracle on the input it was given, and the draft calls'
    Expert Lookahead Buffer counts against the oracle's routing."""
    spx, gh = _spx(), _gh()
    s = _small("qwen15_moe", H=512, I=256, E=8, I_s=256)  # router product: routing follows x
    lay = gh.Layer(s)
    L = 2
    elb = torch.zeros(L, s.E, dtype=torch.int32, device="cuda")
    chains = [("draft", 1, 2), ("verify", 9, 2), ("draft", 9, 2), ("draft", 1, 2)]  # outputs shrink ~10x a layer
    calls, keep = [], []
    for mode, T, n in chains:
        ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
        x = gh.dev_f16(W.gen_x(s, T, step=10 + T, which=int(mode == "verify")))
        for j in range(n):
            out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
            r = spx.Routing.empty(T, s.E, s.k)
            lg = torch.empty(T, s.E, dtype=torch.float32, device="cuda")
            args, kp = spx.layer_args(0 if mode == "draft" else 1, x, s.E, s.k, s.renorm, lg, r, out, ws,
                                      w4=lay.w4, f16=lay.f16, shared=lay.shared, w_router=lay.w_router,
                                      elb=elb if mode == "draft" else None, layer=j)
            spx.spx_moe_layer(args)  # no synchronisation between the calls
            calls.append((mode, T, j, x, out, r))
            keep.append((args, kp, lg, ws))
            x = out
    torch.cuda.synchronize()
    elb_ref = np.zeros((L, s.E), np.uint32)
    for mode, T, j, x, out, r in calls:
        xin = x.cpu().numpy().view(np.uint16)
        ref = lay.oracle_layer(mode, xin)
        assert np.array_equal(r.topk_ids.cpu().numpy(), ref["ids"]), (mode, T, j)
        gh.check_close(gh.f16_out(out), ref["out_half"].view(np.float16).astype(np.float64), f"chain {mode} T={T} #{j}")
        if mode == "draft":
            oracle.elb_accumulate(elb_ref, j, ref["ids"])
    assert np.array_equal(elb.cpu().numpy().astype(np.uint32), elb_ref)


def _cache_case(mode, T):
    s = _small("deepseek_v2_lite", I=256, E=16, I_s=512)
    x = W.gen_x(s, T, step=30 + T, which=int(mode == "verify"))
    logits = W.gen_logits(s, T, step=30 + T, which=int(mode == "verify"))
    need = _gh().needed_experts(s, [logits], [x])
    lay = _gh().Layer(s, needed=need)
    return s, x, logits, lay


@pytest.mark.parametrize("mode,T", [("verify", 17), ("draft", 1), ("draft", 9)])
def test_cache_aware_order_and_ready_flags(mode, T):
    """Cache-aware calls (resident experts queued first, a ready flag per
    expert, all set): the same routing outputs and layer output as the oracle
    (the order changes no result); draft calls take the routing + expert
    launch path."""
    spx, gh = _spx(), _gh()
    s, x, logits, lay = _cache_case(mode, T)
    ref = lay.oracle_layer(mode, x, logits=logits)
    rng = np.random.default_rng(T)
    resident = torch.from_numpy((rng.random(s.E) < 0.5).astype(np.uint8)).cuda()
    ready = torch.ones(s.E, dtype=torch.int32, device="cuda")
    r = spx.Routing.empty(T, s.E, s.k)
    out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    args, keep = spx.layer_args(0 if mode == "draft" else 1, gh.dev_f16(x), s.E, s.k, s.renorm, gh.dev(logits), r,
                                out, ws, w4=lay.w4, f16=lay.f16, shared=lay.shared, resident=resident, ready=ready)
    for rep in range(2):
        spx.spx_moe_layer(args)
        torch.cuda.synchronize()
        assert np.array_equal(r.topk_ids.cpu().numpy(), ref["ids"])
        assert np.array_equal(r.sorted_slots.cpu().numpy(), ref["gather"]["sorted_slots"])
        gh.check_close(gh.f16_out(out), ref["out_half"].view(np.float16).astype(np.float64), f"cache {mode} {rep}")
    assert spx.spx_workspace_status(ws) == 0


def test_cache_aware_ready_flags_set_late():
    """Ready flags that land while the call runs (a host-to-device copy on
    another stream, issued after the call, no kernel involved): the expert
    launch waits for them and the result matches the oracle."""
    import time
    spx, gh = _spx(), _gh()
    s, x, logits, lay = _cache_case("verify", 17)
    ref = lay.oracle_layer("verify", x, logits=logits)
    ready = torch.zeros(s.E, dtype=torch.int32, device="cuda")
    ones = torch.ones(s.E, dtype=torch.int32).pin_memory()
    r = spx.Routing.empty(17, s.E, s.k)
    out = torch.empty(17, s.H, dtype=torch.float16, device="cuda")
    ws = spx.new_workspace(17, s.H, s.I, s.E, s.k, s.I_s)
    args, keep = spx.layer_args(1, gh.dev_f16(x), s.E, s.k, s.renorm, gh.dev(logits), r, out, ws, f16=lay.f16,
                                shared=lay.shared, ready=ready)
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    spx.spx_moe_layer(args)
    time.sleep(0.005)
    with torch.cuda.stream(side):
        ready.copy_(ones, non_blocking=True)
    torch.cuda.synchronize()
    assert spx.spx_workspace_status(ws) == 0
    gh.check_close(gh.f16_out(out), ref["out_half"].view(np.float16).astype(np.float64), "ready set late")


def test_cache_aware_ready_flag_never_set_times_out():
    """An active expert whose ready flag nothing sets: the expert launch gives
    up after the call's wait bound with SPX_ERR_TIMEOUT in the status word, the
    context stays usable, and a call on a re-zeroed workspace succeeds."""
    spx, gh = _spx(), _gh()
    s, x, logits, lay = _cache_case("verify", 17)
    ref = lay.oracle_layer("verify", x, logits=logits)
    missing = int(ref["ids"][0, 0])
    ready = torch.ones(s.E, dtype=torch.int32, device="cuda")
    ready[missing] = 0
    r = spx.Routing.empty(17, s.E, s.k)
    out = torch.empty(17, s.H, dtype=torch.float16, device="cuda")
    ws = spx.new_workspace(17, s.H, s.I, s.E, s.k, s.I_s)
    dx, dl = gh.dev_f16(x), gh.dev(logits)
    args, keep = spx.layer_args(1, dx, s.E, s.k, s.renorm, dl, r, out, ws, f16=lay.f16, shared=lay.shared,
                                ready=ready, wait_budget_ns=20_000_000)
    spx.spx_moe_layer(args)
    torch.cuda.synchronize()
    assert spx.spx_workspace_status(ws) == spx.SPX_ERR_TIMEOUT
    assert np.array_equal(r.topk_ids.cpu().numpy(), ref["ids"])  # routing ran before the wait
    spx.spx_workspace_init(ws)
    args2, keep2 = spx.layer_args(1, dx, s.E, s.k, s.renorm, dl, r, out, ws, f16=lay.f16, shared=lay.shared)
    spx.spx_moe_layer(args2)
    torch.cuda.synchronize()
    assert spx.spx_workspace_status(ws) == 0
    gh.check_close(gh.f16_out(out), ref["out_half"].view(np.float16).astype(np.float64), "after a timeout")


@pytest.mark.parametrize("T", [4, 5, 8])
def test_batched_draft_full_size(T):
    """Several requests' draft tokens in one draft call (DeepSeek-V2-Lite
    shape, T = 4, 5 and 8 tokens; up to 5 one draft launch, 8 through the
    routing launch and the expert launch), each expert the tokens share read
    once; routing outputs bit-exact and the layer output within tolerance."""
    gh = _gh()
    s = W.CONFIGS["deepseek_v2_lite"]
    x = W.gen_x(s, T, step=40 + T)
    logits = W.gen_logits(s, T, step=40 + T)
    need = gh.needed_experts(s, [logits], [x])
    lay = gh.Layer(s, needed=need, verify=False)
    ref = lay.oracle_layer("draft", x, logits=logits)
    outs, routing, _ = _run_layer(lay, "draft", x, logits)
    assert np.array_equal(routing.topk_ids.cpu().numpy(), ref["ids"])
    g = ref["gather"]
    assert np.array_equal(routing.offsets.cpu().numpy(), g["offsets"])
    assert np.array_equal(routing.sorted_slots.cpu().numpy(), g["sorted_slots"])
    for rep, o in enumerate(outs):
        gh.check_close(o, ref["out_half"].view(np.float16).astype(np.float64), f"batched draft T={T} rep {rep}")


# ------------------------------------------- asymmetric INT4 (zero points)
@pytest.mark.parametrize("T,S", [(1, 32), (1, 16), (4, 32), (5, 16), (8, 16), (9, 16), (17, 16), (17, 32)])
def test_draft_layer_zero_points_full_size(T, S):
    """Per-group zero points (the AWQ form, W = (code - zero) * scale, zeros
    uniform over 0..15) on every draft expert, DeepSeek-V2-Lite shape, through
    spx_moe_layer: routing bit-exact, output within tolerance of the oracle.
    Up to 5 tokens the draft launch serves the call, from 6 on the routing
    launch and the expert launch."""
    gh = _gh()
    s = W.CONFIGS["deepseek_v2_lite"]
    x = W.gen_x(s, T, step=60 + T)
    logits = W.gen_logits(s, T, step=60 + T)
    need = gh.needed_experts(s, [logits], [x])
    lay = gh.Layer(s, needed=need, verify=False, slice_cols=S, zeros=True)
    ref = lay.oracle_layer("draft", x, logits=logits)
    outs, routing, _ = _run_layer(lay, "draft", x, logits)
    assert np.array_equal(routing.topk_ids.cpu().numpy(), ref["ids"])
    for rep, o in enumerate(outs):
        gh.check_close(o, ref["out_half"].view(np.float16).astype(np.float64), f"zero points T={T} S={S} rep {rep}")


@pytest.mark.parametrize("case", [0, 1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_draft_unit_call_zero_points(case):
    """spx_moe_draft_w4a16 with zero points on the small cases (several tiles,
    ragged token tiles and groups, both slice widths; up to 5 tokens on the
    draft launch, then the expert launch with 1, 2, 3, 5 or 8 token tiles)."""
    spx, gh = _spx(), _gh()
    s, T, S = SMALL_CASES[case]
    x = W.gen_x(s, T, step=70 + case)
    lg = np.random.default_rng(70 + case).standard_normal((T, s.E))
    ids, w = oracle.route_topk(lg, s.k, s.renorm)
    lay = gh.Layer(s, needed=sorted(set(ids.reshape(-1).tolist())), verify=False, slice_cols=S, zeros=True)
    g, r = _routing_dev(ids, s.E)
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    y_ref = np.stack([oracle.swiglu_w4(x[int(sl) // s.k], lay.w4_host[int(ids.reshape(-1)[sl])])
                      for sl in g["sorted_slots"]])
    y = torch.empty(T * s.k, s.H, dtype=torch.float32, device="cuda")
    for rep in range(2):
        spx.spx_moe_draft_w4a16(gh.dev_f16(x), lay.w4, s.k, r["offsets"], r["sorted_slots"], r["active"],
                                r["n_active"], y, ws)
        torch.cuda.synchronize()
        gh.check_close(y.cpu().numpy(), y_ref, f"zero points case {case} rep {rep}")
    assert spx.spx_workspace_status(ws) == 0


@pytest.mark.parametrize("case", [2, 3, 5])
def test_zero_points_of_eight_match_the_symmetric_path(case):
    """Zero points all 8 reduce the asymmetric form to the symmetric one: the
    corrections add exactly zero.  On the draft launch (1 token) every item's
    partial sums are bit-identical to the zero-point-free launch's and the
    outputs differ at most by the order of the fp32 atomic additions; on the
    expert launch (17 and 9 tokens) a chunk also carries its groups' zero
    points, so chunks hold fewer groups and the fp32 partial sums are grouped
    differently as well."""
    spx, gh = _spx(), _gh()
    s, T, S = SMALL_CASES[case]
    x = W.gen_x(s, T, step=80)
    ids, _ = oracle.route_topk(np.random.default_rng(80).standard_normal((T, s.E)), s.k, s.renorm)
    lay = gh.Layer(s, needed=sorted(set(ids.reshape(-1).tolist())), verify=False, slice_cols=S)
    eights = np.int32(np.uint32(0x88888888).view(np.int32))
    E, H, I = s.E, s.H, s.I
    w4z = spx.spx_w4_zeros_repack(lay.w4, gh.dev(np.full((E, H // 128, I // 8), eights, np.int32)),
                                  gh.dev(np.full((E, H // 128, I // 8), eights, np.int32)),
                                  gh.dev(np.full((E, I // 128, H // 8), eights, np.int32)))
    g, r = _routing_dev(ids, s.E)
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    ys = []
    for w4 in (lay.w4, w4z):
        y = torch.empty(T * s.k, s.H, dtype=torch.float32, device="cuda")
        spx.spx_moe_draft_w4a16(gh.dev_f16(x), w4, s.k, r["offsets"], r["sorted_slots"], r["active"],
                                r["n_active"], y, ws)
        torch.cuda.synchronize()
        ys.append(y.cpu().numpy())
    # expert launch: a reassociation of fp32 sums over H = 2048 products
    # (measured 8.5e-6 of the largest output at 32-column slices)
    d = float(np.abs(ys[0] - ys[1]).max()) / float(np.abs(ys[0]).max())
    assert d <= (1e-6 if T <= 5 else 3e-5), d


@pytest.mark.parametrize("T", [1, 9])
def test_cache_aware_draft_with_zero_points(T):
    """A cache-aware draft layer call with zero points (resident experts first,
    ready flags all set) takes the routing + expert launch path at any token
    count and matches the oracle."""
    spx, gh = _spx(), _gh()
    s = _small("deepseek_v2_lite", I=256, E=16, I_s=512)
    x = W.gen_x(s, T, step=90 + T)
    logits = W.gen_logits(s, T, step=90 + T)
    lay = gh.Layer(s, needed=gh.needed_experts(s, [logits], [x]), verify=False, slice_cols=16, zeros=True)
    ref = lay.oracle_layer("draft", x, logits=logits)
    resident = torch.from_numpy((np.random.default_rng(T).random(s.E) < 0.5).astype(np.uint8)).cuda()
    ready = torch.ones(s.E, dtype=torch.int32, device="cuda")
    r = spx.Routing.empty(T, s.E, s.k)
    out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    args, keep = spx.layer_args(0, gh.dev_f16(x), s.E, s.k, s.renorm, gh.dev(logits), r, out, ws, w4=lay.w4,
                                shared=lay.shared, resident=resident, ready=ready)
    for rep in range(2):
        spx.spx_moe_layer(args)
        torch.cuda.synchronize()
        assert np.array_equal(r.topk_ids.cpu().numpy(), ref["ids"])
        gh.check_close(gh.f16_out(out), ref["out_half"].view(np.float16).astype(np.float64), f"cache zp T={T} {rep}")
    assert spx.spx_workspace_status(ws) == 0


def test_zero_points_wide_slices_reject_many_tokens():
    """32-column INT4 slices take at most 24 tokens per call on the expert
    launch, with zero points as without."""
    spx, gh = _spx(), _gh()
    from quantized_expert_gb300.spx import SpxError
    s = _small("deepseek_v2_lite", I=256, E=16)
    T = 25
    lay = gh.Layer(s, needed=list(range(s.E)), verify=False, slice_cols=32, zeros=True)
    ids, _ = oracle.route_topk(np.random.default_rng(90).standard_normal((T, s.E)), s.k, s.renorm)
    g, r = _routing_dev(ids, s.E)
    y = torch.empty(T * s.k, s.H, device="cuda")
    with pytest.raises(SpxError) as ei:
        spx.spx_moe_draft_w4a16(gh.dev_f16(W.gen_x(s, T)), lay.w4, s.k, r["offsets"], r["sorted_slots"],
                                r["active"], r["n_active"], y, spx.new_workspace(T, s.H, s.I, s.E, s.k))
    assert ei.value.status == spx.SPX_ERR_UNSUPPORTED


# ------------------------------------------------------------- GGUF drafts
@pytest.mark.parametrize("kind", ["q8_0", "q2_k", "q4_k"])
@pytest.mark.parametrize("name,T", [("deepseek_v2_lite", 1), ("deepseek_v2_lite", 5), ("qwen15_moe", 1),
                                    ("phi35_moe", 1)])
def test_gguf_draft_layer_full_size(name, T, kind):
    """GGUF draft experts at full size through spx_moe_layer: Q8_0 (fp16
    scale per 32 weights, int8 codes), or Q2_K / Q4_K gate/up (super-blocks
    of 256 with 4- / 6-bit sub-block scales and mins, 2- / 4-bit codes) with a
    Q8_0 down projection: routing bit-exact, output within tolerance of the
    oracle."""
    gh = _gh()
    s = W.CONFIGS[name]
    x = W.gen_x(s, T, step=100 + T)
    logits = None if s.logits == "router" else W.gen_logits(s, T, step=100 + T)
    need = gh.needed_experts(s, [logits], [x])
    lay = gh.Layer(s, needed=need, verify=False, gguf=kind)
    ref = lay.oracle_layer("draft", x, logits=logits)
    outs, routing, _ = _run_layer(lay, "draft", x, logits)
    assert np.array_equal(routing.topk_ids.cpu().numpy(), ref["ids"])
    g = ref["gather"]
    assert np.array_equal(routing.sorted_slots.cpu().numpy(), g["sorted_slots"])
    for rep, o in enumerate(outs):
        gh.check_close(o, ref["out_half"].view(np.float16).astype(np.float64), f"{kind} {name} T={T} rep {rep}")


GGUF_ENGINE_KINDS = ["q8_0", "q2_k", "q4_k"]  # served by the expert launch too (above 5 tokens, cache-aware)


@pytest.mark.parametrize("kind,case", [(kd, c) for kd in ["q8_0", "q2_k", "q4_k"] for c in [1, 2, 9]] +
                         [(kd, c) for kd in GGUF_ENGINE_KINDS for c in [3, 4, 5, 6, 7, 8]])
def test_gguf_draft_unit_call(case, kind):
    """spx_moe_draft_gguf on the small cases with 16-column slices: per-slot
    expert outputs against the oracle (up to 5 tokens on the draft launch,
    then the expert launch with 1, 2, 3, 5 or 8 token tiles)."""
    spx, gh = _spx(), _gh()
    s, T, S = SMALL_CASES[case]
    x = W.gen_x(s, T, step=110 + case)
    lg = np.random.default_rng(110 + case).standard_normal((T, s.E))
    ids, w = oracle.route_topk(lg, s.k, s.renorm)
    lay = gh.Layer(s, needed=sorted(set(ids.reshape(-1).tolist())), verify=False, gguf=kind)
    g, r = _routing_dev(ids, s.E)
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    y_ref = np.stack([oracle.swiglu_draft(x[int(sl) // s.k], lay.w4_host[int(ids.reshape(-1)[sl])])
                      for sl in g["sorted_slots"]])
    y = torch.empty(T * s.k, s.H, dtype=torch.float32, device="cuda")
    for rep in range(2):
        spx.spx_moe_draft_gguf(gh.dev_f16(x), lay.gguf, s.k, r["offsets"], r["sorted_slots"], r["active"],
                               r["n_active"], y, ws)
        torch.cuda.synchronize()
        gh.check_close(y.cpu().numpy(), y_ref, f"{kind} case {case} rep {rep}")
    assert spx.spx_workspace_status(ws) == 0


@pytest.mark.parametrize("kind", ["q8_0", "q2_k", "q4_k"])
def test_gguf_draft_ragged_ranges(kind):
    """Ragged item ranges: H = 1536 is 6 super-blocks (Q2_K items of 4 + 2,
    Q4_K items of 3 + 3) or 12 Q8_0 groups (3 + 3 + 3 + 3); I = 384 is one
    Q8_0 down range of 3 groups and 24 slices; T = 3 tokens over 8 experts."""
    spx, gh = _spx(), _gh()
    s = _small("phi35_moe", H=1536, I=384, E=8, k=2)
    T = 3
    x = W.gen_x(s, T, step=130)
    lg = np.random.default_rng(130).standard_normal((T, s.E))
    ids, w = oracle.route_topk(lg, s.k, s.renorm)
    lay = gh.Layer(s, needed=sorted(set(ids.reshape(-1).tolist())), verify=False, gguf=kind)
    g, r = _routing_dev(ids, s.E)
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    y_ref = np.stack([oracle.swiglu_draft(x[int(sl) // s.k], lay.w4_host[int(ids.reshape(-1)[sl])])
                      for sl in g["sorted_slots"]])
    y = torch.empty(T * s.k, s.H, dtype=torch.float32, device="cuda")
    spx.spx_moe_draft_gguf(gh.dev_f16(x), lay.gguf, s.k, r["offsets"], r["sorted_slots"], r["active"],
                           r["n_active"], y, ws)
    torch.cuda.synchronize()
    gh.check_close(y.cpu().numpy(), y_ref, f"{kind} ragged")
    assert spx.spx_workspace_status(ws) == 0


@pytest.mark.parametrize("kind", GGUF_ENGINE_KINDS)
@pytest.mark.parametrize("T", [9, 17])
def test_gguf_layer_on_the_expert_launch_full_size(kind, T):
    """GGUF draft layers above 5 tokens (DeepSeek-V2-Lite shape) take the
    routing launch and the expert launch: routing bit-exact, output within
    tolerance of the oracle."""
    gh = _gh()
    s = W.CONFIGS["deepseek_v2_lite"]
    x = W.gen_x(s, T, step=140 + T)
    logits = W.gen_logits(s, T, step=140 + T)
    lay = gh.Layer(s, needed=gh.needed_experts(s, [logits], [x]), verify=False, gguf=kind)
    ref = lay.oracle_layer("draft", x, logits=logits)
    outs, routing, _ = _run_layer(lay, "draft", x, logits)
    assert np.array_equal(routing.topk_ids.cpu().numpy(), ref["ids"])
    for rep, o in enumerate(outs):
        gh.check_close(o, ref["out_half"].view(np.float16).astype(np.float64), f"{kind} T={T} rep {rep}")


@pytest.mark.parametrize("kind", GGUF_ENGINE_KINDS)
@pytest.mark.parametrize("T", [1, 9])
def test_cache_aware_draft_with_gguf(kind, T):
    """A cache-aware draft layer call with GGUF experts (resident experts
    first, ready flags all set) matches the oracle."""
    spx, gh = _spx(), _gh()
    s = _small("deepseek_v2_lite", I=256, E=16, I_s=512)
    x = W.gen_x(s, T, step=150 + T)
    logits = W.gen_logits(s, T, step=150 + T)
    lay = gh.Layer(s, needed=gh.needed_experts(s, [logits], [x]), verify=False, gguf=kind)
    ref = lay.oracle_layer("draft", x, logits=logits)
    resident = torch.from_numpy((np.random.default_rng(T).random(s.E) < 0.5).astype(np.uint8)).cuda()
    ready = torch.ones(s.E, dtype=torch.int32, device="cuda")
    r = spx.Routing.empty(T, s.E, s.k)
    out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    args, keep = spx.layer_args(0, gh.dev_f16(x), s.E, s.k, s.renorm, gh.dev(logits), r, out, ws, gguf=lay.gguf,
                                shared=lay.shared, resident=resident, ready=ready)
    for rep in range(2):
        spx.spx_moe_layer(args)
        torch.cuda.synchronize()
        assert np.array_equal(r.topk_ids.cpu().numpy(), ref["ids"])
        gh.check_close(gh.f16_out(out), ref["out_half"].view(np.float16).astype(np.float64), f"cache {kind} {T} {rep}")
    assert spx.spx_workspace_status(ws) == 0


def test_gguf_invalid_calls():
    """INT4 and GGUF experts in one call, or an unknown GGUF format, are
    invalid arguments; Q2_K and Q4_K need H a multiple of 256."""
    spx, gh = _spx(), _gh()
    from quantized_expert_gb300.spx import SpxError
    s = _small("deepseek_v2_lite", I=256, E=16)
    lay = gh.Layer(s, needed=list(range(s.E)), verify=False, gguf="q2_k")
    T = 1
    routing = spx.Routing.empty(T, s.E, s.k)
    out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    lg = gh.dev(np.random.default_rng(121).standard_normal((T, s.E)).astype(np.float32))
    x = gh.dev_f16(W.gen_x(s, T))
    w4 = gh.Layer(s, needed=[0], verify=False, slice_cols=16).w4
    args, keep = spx.layer_args(0, x, s.E, s.k, s.renorm, lg, routing, out, ws, w4=w4, gguf=lay.gguf)
    with pytest.raises(SpxError) as ei:
        spx.spx_moe_layer(args, None)
    assert ei.value.status == spx.SPX_ERR_INVALID_ARG
    bad = spx.PackedGguf(lay.gguf.buf, lay.gguf.E, lay.gguf.H, lay.gguf.I, 7)
    args, keep = spx.layer_args(0, x, s.E, s.k, s.renorm, lg, routing, out, ws, gguf=bad)
    with pytest.raises(SpxError) as ei:
        spx.spx_moe_layer(args, None)
    assert ei.value.status == spx.SPX_ERR_INVALID_ARG
    assert spx.load().spx_gguf_packed_bytes(4, 384, 256, spx.SPX_GGUF_Q2_K) == 0   # H not a multiple of 256
    assert spx.load().spx_gguf_packed_bytes(4, 384, 256, spx.SPX_GGUF_Q4_K) == 0
    assert spx.load().spx_gguf_packed_bytes(4, 384, 256, spx.SPX_GGUF_Q8_0) > 0
