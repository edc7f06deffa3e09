"""Verify layers whose routed experts arrive through the prefetch plan: the
routed FP16 experts start offloaded (their packed bytes in page-locked host
memory, the device copies zeroed, every ready flag clear); the draft phase's
lookahead counters are planned chunk by chunk (spx_plan_prefetch) and the
copies are enqueued on a side stream (spx_prefetch_issue); after the final
cleanup each verify layer is launched with its ready flags, and the experts
the drafts did not foresee are loaded behind the launch, which waits for
them.  Routing bit-exact and outputs within tolerance of the oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import spx_workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


def _spx():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from quantized_expert_gb300 import build, spx
    build.build()
    spx.load()
    return spx


def test_verify_layers_with_experts_from_the_prefetch_plan():
    spx = _spx()
    import gpu_helpers as gh
    s = W.scaled(W.CONFIGS["deepseek_v2_lite"], I=256, E=16)
    L, K, E, k, Tv = 3, s.K, s.E, s.k, s.T_verify
    lays = [gh.Layer(s, layer=l, needed=None, draft=False, verify=True) for l in range(L)]
    eb = spx.load().spx_f16_packed_bytes(1, s.H, s.I)
    assert lays[0].f16.buf.numel() == E * eb
    host = [lay.f16.buf.cpu().pin_memory() for lay in lays]
    dev = [torch.zeros_like(lay.f16.buf) for lay in lays]  # offloaded: nothing on the device yet
    for lay, d in zip(lays, dev):
        lay.f16 = spx.PackedF16(d, E, s.H, s.I)
    ready = torch.zeros(L, E, dtype=torch.int32, device="cuda")
    resident = torch.zeros(L, E, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()

    # the draft phase's counters, step by step from the cycle's draft logits
    import oracle
    picks = [[oracle.route_topk(W.draft_logits(s, l, st).astype(np.float64), k, False)[0][0]
              for l in range(L)] for st in range(1, K + 1)]
    cfg = spx.PlanCfg(L, E, K, E, 1, 200.0, 90.0)
    elb = np.zeros((L, E), np.uint32)
    cached = np.zeros((L, E), np.uint8)
    done, phases = 0, []
    while True:
        phase, acts, chunk = spx.spx_plan_prefetch(cfg, elb, done, cached)
        phases.append((done, phase, len(acts), chunk))
        spx.spx_prefetch_issue(acts, host, dev, eb, ready, resident, stream=side)
        if phase == spx.SPX_PLAN_FINAL_CLEANUP:
            break
        for st in range(done, done + chunk):
            for l in range(L):
                elb[l, picks[st][l]] += 1
        done += chunk
    assert phases[0][1] == spx.SPX_PLAN_COLD_START and sum(p[3] for p in phases) == K

    for l, lay in enumerate(lays):
        x = W.gen_x(s, Tv, layer=l, step=K + 1, which=1)
        lg = W.verify_logits(s, l)
        ref = lay.oracle_layer("verify", x, logits=lg)
        r = spx.Routing.empty(Tv, E, k)
        out = torch.empty(Tv, s.H, dtype=torch.float16, device="cuda")
        ws = spx.new_workspace(Tv, s.H, s.I, E, k, s.I_s)
        args, keep = spx.layer_args(1, gh.dev_f16(x), E, k, s.renorm, gh.dev(lg), r, out, ws, f16=lay.f16,
                                    shared=lay.shared, resident=resident[l], ready=ready[l])
        spx.spx_moe_layer(args)  # waits (bounded) on the flags of experts still in flight
        # misses: experts the verify routes to that the drafts never selected, loaded behind the launch
        miss = sorted(set(ref["ids"].reshape(-1).tolist()) - set(np.flatnonzero(cached[l]).tolist()))
        acts = np.array([[l, e, spx.SPX_PLAN_LOAD] for e in miss], np.int32).reshape(-1, 3)
        cached[l, miss] = 1
        spx.spx_prefetch_issue(acts, host, dev, eb, ready, resident, stream=side)
        torch.cuda.synchronize()
        assert spx.spx_workspace_status(ws) == 0
        assert np.array_equal(r.topk_ids.cpu().numpy(), ref["ids"])
        gh.check_close(gh.f16_out(out), ref["out_half"].view(np.float16).astype(np.float64),
                       f"verify layer {l} with prefetched experts")
    # every expert the lookahead or the verify needed is on the device, byte for byte
    for l in range(L):
        for e in np.flatnonzero(cached[l]):
            assert torch.equal(dev[l][e * eb:(e + 1) * eb].cpu(), host[l][e * eb:(e + 1) * eb])
        assert np.array_equal(ready[l].cpu().numpy() != 0, cached[l] != 0)
