"""The full draft-then-verify cycle on the 26-layer DeepSeek-V2-Lite-shaped
stack (K = 16 draft steps at T = 1 through every layer, then one T = 17 verify
pass), through spx_moe_layer at full size.

Checked against the CPU oracle on every layer: top-k IDs of every call, the
gather arrays of the verify pass, and the Expert Lookahead Buffer counters
accumulated on the device over the 16 draft steps, with the distinct experts
per layer that follow from them (all bit-exact).  Layer outputs are checked
within the fp16 tolerance on a seeded subset of layers, whose weights are the
oracle's; the other layers carry device-generated random weights, since their
routing does not depend on the weights (logits are given).

Reading of the cycle (the pages leave the data flow between layers open):
each (layer, step) gets its own seeded N(0,1) input; verify token i < K routes
on the logits of draft step i + 1, token K on a fresh draw."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import spx_workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu

CHECK_LAYERS = (3, 17)  # outputs checked against the oracle on these layers


def _device_weights(s, layer, spx):
    """Random canonical weights generated on the device (not the oracle's)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(7_000_003 + 131 * layer)
    E, H, I = s.E, s.H, s.I

    def codes(*shape):
        return torch.randint(-2 ** 31, 2 ** 31, shape, dtype=torch.int32, device="cuda", generator=g)

    def scales(*shape):
        return (torch.rand(shape, device="cuda", generator=g) * 0.015 + 0.005).half()

    def normal(*shape):
        return (torch.randn(shape, device="cuda", generator=g) * 0.02).half()

    w4 = spx.spx_w4_repack(codes(E, H // 8, I), scales(E, H // 128, I), codes(E, H // 8, I),
                           scales(E, H // 128, I), codes(E, I // 8, H), scales(E, I // 128, H), slice_cols=32)
    f16 = spx.spx_f16_repack(normal(E, I, H), normal(E, I, H), normal(E, H, I))
    sh = spx.pack_shared(normal(s.I_s, H), normal(s.I_s, H), normal(H, s.I_s), None)
    return w4, f16, sh


def test_cycle_26_layers_elb_and_routing():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import gpu_helpers as gh
    from quantized_expert_gb300 import build, spx
    build.build()
    spx.load()
    s = W.CONFIGS["deepseek_v2_lite_x26"]
    L, K, E, k = s.layers, s.K, s.E, s.k
    Tv = s.T_verify

    # oracle routing of every call (cheap): draft ids per (step, layer), verify ids per layer
    draft_ids = {(st, l): oracle.route_topk(W.draft_logits(s, l, st).astype(np.float64), k, s.renorm)[0]
                 for st in range(1, K + 1) for l in range(L)}
    verify_ids = {l: oracle.route_topk(W.verify_logits(s, l).astype(np.float64), k, s.renorm)[0] for l in range(L)}

    lays = {}
    for l in range(L):
        if l in CHECK_LAYERS:
            need = set(verify_ids[l].reshape(-1).tolist())
            for st in range(1, K + 1):
                need |= set(draft_ids[(st, l)].reshape(-1).tolist())
            lay = gh.Layer(s, layer=l, needed=sorted(need))
            lays[l] = (lay.w4, lay.f16, lay.shared, lay)
        else:
            lays[l] = _device_weights(s, l, spx) + (None,)

    elb = torch.zeros(L, E, dtype=torch.int32, device="cuda")
    elb_ref = np.zeros((L, E), np.uint32)
    ws_d = spx.new_workspace(1, s.H, s.I, E, k, s.I_s)
    ws_v = spx.new_workspace(Tv, s.H, s.I, E, k, s.I_s)
    r_d, r_v = spx.Routing.empty(1, E, k), spx.Routing.empty(Tv, E, k)
    out_d = torch.empty(1, s.H, dtype=torch.float16, device="cuda")
    out_v = torch.empty(Tv, s.H, dtype=torch.float16, device="cuda")

    elb_host = {l: np.zeros(E, np.uint32) for l in CHECK_LAYERS}  # oracle-side ELB of the checked layers
    for st in range(1, K + 1):
        for l in range(L):
            w4, f16, sh, lay = lays[l]
            x = W.gen_x(s, 1, layer=l, step=st)
            lg = W.draft_logits(s, l, st)
            args, keep = spx.layer_args(0, gh.dev_f16(x), E, k, s.renorm, gh.dev(lg), r_d, out_d, ws_d, w4=w4,
                                        shared=sh, elb=elb, layer=l)
            spx.spx_moe_layer(args)
            hdr = ws_d[:256].view(torch.int32).cpu().numpy()  # status word and the site of a wait that gave up
            assert hdr[2] == 0, (f"draft step {st} layer {l}: status {hdr[2]}, wait site {hdr[5]}, ring state "
                                 f"{hdr[6:18]}, stage seqs {hdr[18:34]}")
            ids = draft_ids[(st, l)]
            oracle.elb_accumulate(elb_ref, l, ids)
            if lay is not None:
                torch.cuda.synchronize()
                ref = lay.oracle_layer("draft", x, logits=lg)
                gh.check_close(gh.f16_out(out_d), ref["out_half"].view(np.float16).astype(np.float64),
                               f"cycle draft step {st} layer {l}")
            if st == K or lay is not None:
                torch.cuda.synchronize()
                assert np.array_equal(r_d.topk_ids.cpu().numpy(), ids), (st, l)
    torch.cuda.synchronize()
    got = elb.cpu().numpy().astype(np.uint32)
    assert np.array_equal(got, elb_ref)
    assert np.all(got.sum(1) == K * k)
    distinct = (got > 0).sum(1)
    assert np.array_equal(distinct, (elb_ref > 0).sum(1))
    assert distinct.min() >= k and distinct.max() <= min(E, K * k)

    for l in range(L):
        w4, f16, sh, lay = lays[l]
        x = W.gen_x(s, Tv, layer=l, step=K + 1, which=1)
        lg = W.verify_logits(s, l)
        args, keep = spx.layer_args(1, gh.dev_f16(x), E, k, s.renorm, gh.dev(lg), r_v, out_v, ws_v, f16=f16,
                                    shared=sh)
        spx.spx_moe_layer(args)
        torch.cuda.synchronize()
        ids = verify_ids[l]
        g = oracle.gather_by_expert(ids, E)
        assert np.array_equal(r_v.topk_ids.cpu().numpy(), ids), l
        assert np.array_equal(r_v.offsets.cpu().numpy(), g["offsets"]), l
        assert np.array_equal(r_v.sorted_slots.cpu().numpy(), g["sorted_slots"]), l
        if lay is not None:
            ref = lay.oracle_layer("verify", x, logits=lg)
            gh.check_close(gh.f16_out(out_v), ref["out_half"].view(np.float16).astype(np.float64),
                           f"cycle verify layer {l}")
    assert spx.spx_workspace_status(ws_d) == 0 and spx.spx_workspace_status(ws_v) == 0
