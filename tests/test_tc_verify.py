"""Verify layers on the tensor-memory launches (tcgen05 products, accumulators
in tensor memory, TMA tensor copies): routing bit-exact, output within the
layer tolerance of the oracle, at small sizes that span several units and
ragged token tiles, and at the full Phi-3.5-MoE, DeepSeek-V2-Lite and
Qwen1.5-MoE sizes.  [P1 Key Contributions 4: expert-wise verification turns
each expert's GEMVs into one dense product over its tokens]"""
import numpy as np
import pytest
import torch

import spx_workloads as W

pytestmark = pytest.mark.gpu


def _spx():
    from quantized_expert_gb300 import spx
    return spx


def _gh():
    import gpu_helpers
    return gpu_helpers


def _run(lay, x, logits, launch, tc_ws=True):
    spx, gh = _spx(), _gh()
    s = lay.shape
    T = x.shape[0]
    routing = spx.Routing.empty(T, s.E, s.k)
    out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s, tc=tc_ws)
    d_lg = gh.dev(np.asarray(logits, np.float32)) if logits is not None else torch.empty(
        T, s.E, dtype=torch.float32, device="cuda")
    args, keep = spx.layer_args(1, gh.dev_f16(x), s.E, s.k, s.renorm, d_lg, routing, out, ws, f16=lay.f16,
                                shared=lay.shared, w_router=lay.w_router, layer=lay.layer, verify_launch=launch)
    outs = []
    for _ in range(2):  # the second call checks that the first left the accumulator zeroed
        spx.spx_moe_layer(args, None)
        torch.cuda.synchronize()
        outs.append(gh.f16_out(out))
    assert spx.spx_workspace_status(ws) == 0
    return outs, routing


def _check(s, T, step, launch=2):
    gh = _gh()
    x = W.gen_x(s, T, step=step)
    logits = None if s.logits == "router" else W.gen_logits(s, T, step=step)
    need = gh.needed_experts(s, [logits], [x])
    lay = gh.Layer(s, needed=need, draft=False, verify=True)
    ref = lay.oracle_layer("verify", x, logits=logits)
    outs, routing = _run(lay, x, logits, launch)
    assert np.array_equal(routing.topk_ids.cpu().numpy(), ref["ids"])
    for rep, o in enumerate(outs):
        gh.check_close(o, ref["out_half"].view(np.float16).astype(np.float64), f"{s.name} T={T} rep {rep}")


@pytest.mark.parametrize("T", [1, 5, 17, 33, 64])
def test_tc_verify_small(T):
    """DeepSeek-shaped layer with I = 256 (4 gate/up units per expert), 16
    experts and a shared expert of 512: token counts from one to the maximum,
    ragged 16-token tiles (5, 17, 33), every expert slot."""
    _check(W.scaled(W.CONFIGS["deepseek_v2_lite"], I=256, E=16, I_s=512), T, step=200 + T)


def test_tc_verify_small_shared_gate_and_router():
    """Qwen-shaped (router product on the device, sigmoid shared-expert gate),
    small, 40 tokens."""
    _check(W.scaled(W.CONFIGS["qwen15_moe"], I=384, E=12, I_s=640), 40, step=240)


@pytest.mark.parametrize("E,k,T,I_s", [(256, 8, 64, 192), (8, 8, 33, 0), (16, 4, 9, 320)])
def test_tc_verify_slot_extremes(E, k, T, I_s):
    """Slot-table extremes of the tensor-memory launches: 257 slots (256
    experts, top-8 of 64 tokens), every expert selected (k = E), and shared
    experts whose k range is not a multiple of the routed one (uneven down
    pieces), at the automatic token threshold."""
    _check(W.scaled(W.CONFIGS["deepseek_v2_lite"], H=256, I=128, E=E, k=k, I_s=I_s), T, step=280 + T)


def test_tc_verify_no_shared_expert():
    """Phi-shaped (no shared expert, renormalised top-2), small, 33 tokens."""
    _check(W.scaled(W.CONFIGS["phi35_moe"], H=1024, I=512), 33, step=250)


@pytest.mark.parametrize("name,T", [("phi35_moe", 33), ("phi35_moe", 17), ("deepseek_v2_lite", 33),
                                    ("qwen15_moe", 33), ("deepseek_v2_lite", 17), ("qwen15_moe", 9),
                                    ("deepseek_v2_lite", 5), ("deepseek_v2_lite", 64), ("phi35_moe", 64)])
def test_tc_verify_full_size(name, T):
    """Full-size layers on the tensor-memory launches: from 9 tokens through
    the automatic choice (Phi-3.5-MoE at 33 tokens has no expert-launch
    geometry; 64 tokens is the maximum call), at 5 forced."""
    _check(W.CONFIGS[name], T, step=260 + T, launch=0 if T >= 9 else 2)


def test_tc_verify_invalid_calls():
    """Forced tensor-memory calls without the tile packs, with a cache-aware
    option, or with too small a workspace are rejected on the host; a
    misaligned pack is an invalid argument."""
    spx, gh = _spx(), _gh()
    s = W.scaled(W.CONFIGS["deepseek_v2_lite"], I=256, E=16, I_s=512)
    T = 5  # below the automatic choice: spx_workspace_size leaves the tensor-memory scratch out
    x = W.gen_x(s, T, step=270)
    lay = gh.Layer(s, needed=list(range(s.E)), draft=False, verify=True)
    routing = spx.Routing.empty(T, s.E, s.k)
    out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    ws_small = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s, tc=True)
    lg = gh.dev(W.gen_logits(s, T, step=270))
    lib = spx.load()

    def call(f16, ws_, launch=2, ready=None, shared=lay.shared):
        a, keep = spx.layer_args(1, gh.dev_f16(x), s.E, s.k, s.renorm, lg, routing, out, ws_, f16=f16,
                                 shared=shared, verify_launch=launch, ready=ready)
        return lib.spx_moe_layer(spx.C.byref(a), None)

    no_canon = spx.PackedF16(lay.f16.buf, s.E, s.H, s.I)
    assert call(no_canon, ws) == spx.SPX_ERR_UNSUPPORTED
    odd = spx.PackedF16(lay.f16.buf, s.E, s.H, s.I, lay.f16.tc[8:])  # not 16-byte aligned
    assert call(odd, ws) == spx.SPX_ERR_INVALID_ARG
    sh_no_canon = spx.PackedShared(lay.shared.buf, None, s.H, s.I_s)
    assert call(lay.f16, ws, shared=sh_no_canon) == spx.SPX_ERR_UNSUPPORTED
    ready = torch.ones(s.E, dtype=torch.int32, device="cuda")
    assert call(lay.f16, ws, ready=ready) == spx.SPX_ERR_UNSUPPORTED
    assert call(lay.f16, ws_small) == spx.SPX_ERR_WORKSPACE
    assert call(lay.f16, ws, launch=3) == spx.SPX_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert spx.spx_workspace_status(ws) == 0


def test_tile_pack_layout_matches_the_header():
    """spx_f16_tc_repack writes the layout include/spx.h documents: per expert,
    gate/up tiles (unit u, k-chunk kc) then down tiles (block hb, k-chunk kc),
    128 rows x 64 fp16 each; gate/up tile row 32q + i is gate column
    64u + 16q + i (i < 16) or up column 64u + 16q + i - 16.  Checked element by
    element against the layout built with numpy from the canonical tensors."""
    spx = _spx()
    E, H, I = 2, 256, 192
    rng = np.random.default_rng(5)
    wg, wu = rng.standard_normal((E, I, H)).astype(np.float16), rng.standard_normal((E, I, H)).astype(np.float16)
    wd = rng.standard_normal((E, H, I)).astype(np.float16)
    dev = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    buf = spx.spx_f16_tc_repack(dev(wg), dev(wu), dev(wd))
    torch.cuda.synchronize()
    got = buf.cpu().numpy().view(np.float16)
    tiles = []
    for e in range(E):
        for u in range(I // 64):
            for kc in range(H // 64):
                t = np.empty((128, 64), np.float16)
                for q in range(4):
                    cols = 64 * u + 16 * q + np.arange(16)
                    t[32 * q:32 * q + 16] = wg[e, cols, 64 * kc:64 * kc + 64]
                    t[32 * q + 16:32 * q + 32] = wu[e, cols, 64 * kc:64 * kc + 64]
                tiles.append(t)
        for hb in range(H // 128):
            for kc in range(I // 64):
                tiles.append(wd[e, 128 * hb:128 * hb + 128, 64 * kc:64 * kc + 64])
    want = np.stack(tiles).reshape(-1)
    assert got.shape == want.shape
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
