"""The C ABI without a GPU: libspx.so builds (nvcc cross-compiles sm_103a),
loads, exports every entry point include/spx.h declares, and its host-only
functions (sizes, status strings, argument validation before any launch)
behave as documented."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from quantized_expert_gb300 import build, spx
    build.build()
    return spx.load()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"SPX_API\s+[\w\s\*]+?\b(spx_\w+)\s*\(", txt))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    from quantized_expert_gb300 import spx
    names = declared_symbols()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n
        assert n in spx.exported_symbols(), f"binding lacks {n}"


def test_sizes_and_strings(lib):
    from quantized_expert_gb300 import spx
    assert spx.spx_version() == 106
    assert spx.status_string(0) == "ok"
    assert "timed out" in spx.status_string(-5)
    # INT4 unit = 49*H*S/32 bytes; down scales copied once per expert
    assert lib.spx_w4_packed_bytes(64, 2048, 1408, 32) == (64 * 44 * (49 * 2048 * 32 // 32) + 64 * 11 * 2048 * 2
                                                           + 64 * 64 * 11 * (64 + 4 * 512))
    assert lib.spx_shared_packed_bytes(2048, 2816) == 2816 // 16 * 6 * 2048 * 16 + 64 * 176 * 1024
    assert lib.spx_w4_packed_bytes(64, 2048, 1408, 24) == 0
    assert lib.spx_f16_packed_bytes(64, 2048, 1408) == 64 * 1408 * 2048 * 2 * 3
    assert lib.spx_workspace_size(17, 2048, 1408, 64, 6, 2816) >= 256 + 17 * 2048 * 4
    # the draft launch (up to 5 tokens) adds its split-K scratch
    assert lib.spx_workspace_size(1, 2048, 1408, 64, 6, 2816) > lib.spx_workspace_size(1, 2048, 0, 64, 6, 0)
    assert lib.spx_workspace_size(65, 2048, 1408, 64, 6, 0) == 0
    # tile pack of the tensor-memory verify launches: the canonical matrices' size, 16 KB tiles
    assert lib.spx_f16_tc_packed_bytes(64, 2048, 1408) == 64 * 3 * 1408 * 2048 * 2
    assert lib.spx_f16_tc_packed_bytes(16, 4096, 6400) == 16 * 3 * 6400 * 4096 * 2
    assert lib.spx_f16_tc_packed_bytes(1, 2048, 1400) == 0 and lib.spx_f16_tc_packed_bytes(1, 2112, 1408) == 0
    # their scratch: calls of 9+ tokens get it by default, a forced T=5 call asks for it
    ws5, ws5tc = lib.spx_workspace_size(5, 2048, 1408, 64, 6, 2816), lib.spx_workspace_size_tc(5, 2048, 1408, 64, 6,
                                                                                               2816)
    assert ws5tc > ws5 and ws5tc >= (30 + 1) * 16 * (2048 + 2816) * 2
    for T in (9, 17, 33, 64):
        assert lib.spx_workspace_size(T, 2048, 1408, 64, 6, 2816) == lib.spx_workspace_size_tc(T, 2048, 1408, 64, 6,
                                                                                               2816)
    assert lib.spx_workspace_size_tc(17, 2048, 1400, 64, 6, 0) == 0


def test_validation_before_any_launch(lib):
    from quantized_expert_gb300 import spx
    # null pointers and bad shapes are rejected on the host; no CUDA call is made
    assert lib.spx_route_topk(None, None, None, 1, 128, 8, 2, 0, None, None, None, 0, None) == spx.SPX_ERR_INVALID_ARG
    fake = C.c_void_p(256)
    assert lib.spx_route_topk(None, None, fake, 4, 128, 8, 9, 0, fake, fake, fake, 4096, None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_route_topk(None, None, fake, 65, 128, 8, 2, 0, fake, fake, fake, 4096, None) == spx.SPX_ERR_UNSUPPORTED
    assert lib.spx_elb_accumulate(None, 1, 8, 0, fake, 1, 2, None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_elb_accumulate(fake, 2, 8, 2, fake, 1, 2, None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_gather_by_expert(fake, 1, 300, 300, fake, fake, fake, fake, fake, None) == spx.SPX_ERR_UNSUPPORTED
    w = spx.W4Experts(256, 8, 256, 512, 32)
    assert lib.spx_moe_draft_w4a16(fake, 4, C.byref(w), 2, fake, fake, fake, fake, fake, None, 0, None) == \
        spx.SPX_ERR_WORKSPACE
    w.H = 200
    assert lib.spx_moe_draft_w4a16(fake, 4, C.byref(w), 2, fake, fake, fake, fake, fake, None, 0, None) == \
        spx.SPX_ERR_UNSUPPORTED
    assert lib.spx_moe_layer(None, None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_w4_repack(None, None, None, None, None, None, 1, 256, 256, 32, None, None) == spx.SPX_ERR_INVALID_ARG


def test_header_is_plain_c():
    """The public header compiles as C99 with no CUDA include path."""
    import subprocess
    import tempfile
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.c")
        with open(src, "w") as f:
            f.write('#include "spx.h"\nint main(void){ spx_layer_args a; (void)a; return SPX_OK; }\n')
        subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-c", src, "-I", os.path.join(ROOT, "include"),
                               "-o", os.path.join(d, "t.o")])


@pytest.mark.parametrize("cname,pyname", [("spx_layer_args", "LayerArgs"), ("spx_w4_experts", "W4Experts"),
                                           ("spx_f16_experts", "F16Experts"), ("spx_shared", "Shared"),
                                           ("spx_gguf_experts", "GgufExperts")])
def test_struct_layouts_match_the_header(tmp_path, cname, pyname):
    """The binding's argument structs mirror the C structs: a program compiled
    against include/spx.h reports each one's size and field offsets."""
    import ctypes as C
    import os
    import subprocess
    from quantized_expert_gb300 import spx
    cls = getattr(spx, pyname)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "layout.c"
    fields = [f for f, _ in cls._fields_]
    body = "\n".join(f'    printf("%zu\\n", offsetof({cname}, {f}));' for f in fields)
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "spx.h"\nint main(void) {\n'
                   f'    printf("%zu\\n", sizeof({cname}));\n' + body + "\n    return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(root, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert got[0] == C.sizeof(cls)
    for f, off in zip(fields, got[1:]):
        assert getattr(cls, f).offset == off, f


def test_draft_format_sizes_and_validation(lib):
    """Host-side sizes and argument checks of the zero-point and GGUF entry
    points (no CUDA call is made on these paths)."""
    from quantized_expert_gb300 import spx
    E, H, I = 64, 2048, 1408
    # zero points: fp16 per (group of 128 rows, column) of gate, up and down
    assert lib.spx_w4_zeros_bytes(E, H, I, 32) == 2 * (2 * E * (H // 128) * I + E * (I // 128) * H)
    assert lib.spx_w4_zeros_bytes(E, H, I, 24) == 0
    # GGUF: Q8_0 gate/up/down 34 B per 32 weights; Q2_K gate/up 84 B per 256 weights + Q8_0 down;
    # then, for the expert launch, the down codes once more in unit order (1 B per weight) and
    # the down scales [E][I/32][H] fp16
    q8 = E * H * I * 34 // 32

    def udn(h):
        return E * I * h + E * (I // 32) * h * 2
    assert lib.spx_gguf_packed_bytes(E, H, I, spx.SPX_GGUF_Q8_0) == 3 * q8 + udn(H)  # scales inside the blocks
    assert lib.spx_gguf_packed_bytes(E, H, I, spx.SPX_GGUF_Q2_K) == 2 * E * H * I * 84 // 256 + q8 + udn(H)
    # Q4_K as packed: 4736 bytes per super-block of a 16-column slice (the 6-bit
    # scales and mins unpacked to bytes: 148 bytes per 256 weights, 144 in the file)
    assert lib.spx_gguf_packed_bytes(E, H, I, spx.SPX_GGUF_Q4_K) == E * (I // 16) * (H // 256) * 4736 + q8 + udn(H)
    assert lib.spx_gguf_packed_bytes(E, H, I, spx.SPX_GGUF_Q4_K) == 2 * E * H * I * 148 // 256 + q8 + udn(H)
    assert lib.spx_gguf_packed_bytes(E, 384, I, spx.SPX_GGUF_Q2_K) == 0   # Q2_K rows: multiples of 256
    assert lib.spx_gguf_packed_bytes(E, 384, I, spx.SPX_GGUF_Q4_K) == 0
    assert lib.spx_gguf_packed_bytes(E, 384, I, spx.SPX_GGUF_Q8_0) == E * 384 * I * 34 // 32 * 3 + udn(384)
    assert lib.spx_gguf_packed_bytes(E, H, I, 7) == 0
    fake = C.c_void_p(256)
    assert lib.spx_gguf_repack(None, fake, fake, E, H, I, 0, fake, None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_gguf_repack(fake, fake, fake, E, H, I, 7, fake, None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_gguf_repack(fake, fake, fake, E, 384, I, spx.SPX_GGUF_Q2_K, fake, None) == \
        spx.SPX_ERR_UNSUPPORTED
    assert lib.spx_gguf_repack(fake, fake, fake, E, H, I, 0, C.c_void_p(264), None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_w4_zeros_repack(None, fake, fake, E, H, I, 32, fake, None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_w4_zeros_repack(fake, fake, fake, E, H, I, 24, fake, None) == spx.SPX_ERR_UNSUPPORTED
    g = spx.GgufExperts(256, 8, 256, 512, 9)
    assert lib.spx_moe_draft_gguf(fake, 4, C.byref(g), 2, fake, fake, fake, fake, fake, None, 0, None) == \
        spx.SPX_ERR_WORKSPACE


def test_verify_launch_choice_validation(lib):
    """The layer call's checks of the tensor-memory verify arguments happen on
    the host, before any CUDA call: an unknown verify_launch, a misaligned tile
    pack, a forced call without tile packs, and a forced call whose workspace
    lacks the tensor-memory scratch."""
    from quantized_expert_gb300 import spx
    fake = 1 << 20  # aligned, never dereferenced
    T, H, E, k, I, I_s = 5, 2048, 64, 6, 1408, 2816
    f16 = spx.F16Experts(fake, E, H, I, None)
    sh = spx.Shared(fake, None, H, I_s, None)

    def args(verify_launch, tc_packed=None, sh_tc=None, ws_bytes=None):
        a = spx.LayerArgs()
        a.mode, a.T, a.H, a.E, a.k = 1, T, H, E, k
        a.x = a.logits = a.topk_ids = a.topk_w = fake
        a.counts = a.offsets = a.sorted_slots = a.active = a.n_active = a.out = a.ws = fake
        a.ws_bytes = ws_bytes if ws_bytes is not None else lib.spx_workspace_size(T, H, I, E, k, I_s)
        f16.tc_packed = tc_packed
        sh.tc_packed = sh_tc
        a.f16 = C.pointer(f16)
        a.shared = C.pointer(sh)
        a.verify_launch = verify_launch
        return a

    assert lib.spx_moe_layer(C.byref(args(3)), None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_moe_layer(C.byref(args(-1)), None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_moe_layer(C.byref(args(2, tc_packed=fake + 8, sh_tc=fake)), None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_moe_layer(C.byref(args(2)), None) == spx.SPX_ERR_UNSUPPORTED
    assert lib.spx_moe_layer(C.byref(args(2, tc_packed=fake)), None) == spx.SPX_ERR_UNSUPPORTED  # shared lacks one
    # T = 5: the default workspace has no tensor-memory scratch, a forced call needs spx_workspace_size_tc
    assert lib.spx_workspace_size_tc(T, H, I, E, k, I_s) > lib.spx_workspace_size(T, H, I, E, k, I_s)
    assert lib.spx_moe_layer(C.byref(args(2, tc_packed=fake, sh_tc=fake)), None) == spx.SPX_ERR_WORKSPACE
