"""spx_moe_layer_noalloc: the layer call for callers that cannot allocate
device memory (allocator or pool callbacks, runtimes that forbid device
allocation after start-up), which runs with the library's fixed scratch array
instead of a caller workspace.  Checked through the C ABI against
spx_moe_layer with a caller workspace, on two calls in a row (the fixed array
keeps the previous call's contents, so the second call checks the clearing).

This file is collected last on purpose; it must also pass on its own in a
fresh process."""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import spx_workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from quantized_expert_gb300 import build, spx
    build.build()
    return spx.load()


@pytest.mark.parametrize("mode", ["draft", "verify"])
def test_noalloc_layer_matches_workspace_layer(lib, mode):
    import gpu_helpers as gh
    from quantized_expert_gb300 import spx
    s = W.scaled(W.CONFIGS["deepseek_v2_lite"], I=256, E=16)
    T = s.T_draft if mode == "draft" else s.T_verify
    lay = gh.Layer(s, needed=None, draft=(mode == "draft"), verify=(mode == "verify"))
    x = gh.dev_f16(W.gen_x(s, T, which=int(mode == "verify")))
    lg = gh.dev(W.gen_logits(s, T, which=int(mode == "verify")))
    m = 0 if mode == "draft" else 1
    stream = torch.cuda.current_stream().cuda_stream

    r_ref = spx.Routing.empty(T, s.E, s.k)
    out_ref = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    a_ref, keep_ref = spx.layer_args(m, x, s.E, s.k, s.renorm, lg, r_ref, out_ref, ws, w4=lay.w4, f16=lay.f16,
                                     shared=lay.shared)
    assert lib.spx_moe_layer(C.byref(a_ref), stream) == 0
    torch.cuda.synchronize()
    ref = out_ref.cpu().numpy().astype(np.float64)

    r_na = spx.Routing.empty(T, s.E, s.k)
    out_na = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    a_na, keep_na = spx.layer_args(m, x, s.E, s.k, s.renorm, lg, r_na, out_na, ws, w4=lay.w4, f16=lay.f16,
                                   shared=lay.shared)
    a_na.ws, a_na.ws_bytes = None, 0  # ignored by the fixed-scratch call
    for rep in range(2):
        out_na.zero_()
        assert lib.spx_moe_layer_noalloc(C.byref(a_na), stream) == 0, lib.spx_last_cuda_error()
        torch.cuda.synchronize()
        assert np.array_equal(r_na.topk_ids.cpu().numpy(), r_ref.topk_ids.cpu().numpy())
        assert np.array_equal(r_na.sorted_slots.cpu().numpy(), r_ref.sorted_slots.cpu().numpy())
        gh.check_close(out_na.cpu().numpy().astype(np.float64), ref, f"noalloc {mode} call {rep}")


def test_noalloc_rejects_shapes_beyond_the_fixed_scratch(lib):
    from quantized_expert_gb300 import spx
    a = spx.LayerArgs()
    a.mode, a.T, a.H, a.E, a.k = 1, 64, 8192, 8, 2   # needs > 1 MiB of scratch
    assert lib.spx_moe_layer_noalloc(C.byref(a), None) == spx.SPX_ERR_WORKSPACE
    assert lib.spx_moe_layer_noalloc(None, None) == spx.SPX_ERR_INVALID_ARG
