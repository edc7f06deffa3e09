"""spx_moe_layer_noalloc: the layer call for callers that cannot allocate
device memory (allocator or pool callbacks, runtimes that forbid device
allocation after start-up), which runs with the library's fixed scratch array
instead of a caller workspace, once spx_noalloc_init has loaded the library
onto the device.  Checked through the C ABI against spx_moe_layer with a
caller workspace, on two calls in a row, after a call that gave up on a
bounded wait and left the fixed array dirty (so the clearing is exercised),
with that call's timeout read back through spx_noalloc_status.

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
    lib = spx.load()
    assert lib.spx_noalloc_init() == 0, lib.spx_last_cuda_error()
    assert lib.spx_noalloc_init() == 0  # once per device; later calls return at once
    return lib


def _status(lib, stream):
    st = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    assert lib.spx_noalloc_status(C.c_void_p(st.data_ptr()), stream) == 0
    torch.cuda.synchronize()
    return int(st.item())


def _case(mode):
    import gpu_helpers as gh
    s = W.scaled(W.CONFIGS["deepseek_v2_lite"], I=256, E=16)
    T = s.T_draft if mode == "draft" else s.T_verify
    lay = gh.Layer(s, needed=None, draft=(mode == "draft"), verify=(mode == "verify"))
    x = gh.dev_f16(W.gen_x(s, T, which=int(mode == "verify")))
    lg = gh.dev(W.gen_logits(s, T, which=int(mode == "verify")))
    return s, T, lay, x, lg


@pytest.mark.parametrize("mode", ["draft", "verify"])
def test_noalloc_layer_matches_workspace_layer(lib, mode):
    import gpu_helpers as gh
    from quantized_expert_gb300 import spx
    s, T, lay, x, lg = _case(mode)
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

    # Leave the fixed array dirty: a cache-aware call whose first routed expert
    # never becomes ready gives up after 20 ms with its counters half used.
    ready = torch.ones(s.E, dtype=torch.int32, device="cuda")
    ready[int(r_ref.topk_ids[0, 0].item())] = 0
    r_bad = spx.Routing.empty(T, s.E, s.k)
    out_bad = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    a_bad, keep_bad = spx.layer_args(m, x, s.E, s.k, s.renorm, lg, r_bad, out_bad, ws, w4=lay.w4, f16=lay.f16,
                                     shared=lay.shared, ready=ready, wait_budget_ns=20_000_000)
    assert lib.spx_moe_layer_noalloc(C.byref(a_bad), stream) == 0, lib.spx_last_cuda_error()
    assert _status(lib, stream) == spx.SPX_ERR_TIMEOUT

    r_na = spx.Routing.empty(T, s.E, s.k)
    out_na = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    a_na, keep_na = spx.layer_args(m, x, s.E, s.k, s.renorm, lg, r_na, out_na, ws, w4=lay.w4, f16=lay.f16,
                                   shared=lay.shared)
    a_na.ws, a_na.ws_bytes = None, 0  # ignored by the fixed-scratch call
    for rep in range(2):
        out_na.zero_()
        assert lib.spx_moe_layer_noalloc(C.byref(a_na), stream) == 0, lib.spx_last_cuda_error()
        assert _status(lib, stream) == 0
        assert np.array_equal(r_na.topk_ids.cpu().numpy(), r_ref.topk_ids.cpu().numpy())
        assert np.array_equal(r_na.sorted_slots.cpu().numpy(), r_ref.sorted_slots.cpu().numpy())
        gh.check_close(out_na.cpu().numpy().astype(np.float64), ref, f"noalloc {mode} call {rep}")


def test_noalloc_rejects_before_enqueueing(lib):
    from quantized_expert_gb300 import spx
    a = spx.LayerArgs()
    a.mode, a.T, a.H, a.E, a.k = 1, 64, 8192, 8, 2   # needs > 1 MiB of scratch
    assert lib.spx_moe_layer_noalloc(C.byref(a), None) == spx.SPX_ERR_WORKSPACE
    assert lib.spx_moe_layer_noalloc(None, None) == spx.SPX_ERR_INVALID_ARG
    # a shape that fits but arguments that do not: rejected, nothing cleared
    a.T, a.H = 1, 256
    assert lib.spx_moe_layer_noalloc(C.byref(a), None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_noalloc_status(None, None) == spx.SPX_ERR_INVALID_ARG
