"""Thin Python binding of libspx (include/spx.h): argument marshalling only.

Every function here takes torch tensors that already live on the GPU, passes
their device pointers and the current CUDA stream to the C entry point of the
same name, and raises ``SpxError`` on a non-zero status.  No arithmetic of
the method happens in Python, and there is no fallback: if libspx.so is not
built, importing the library fails with an error.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import torch

from . import build as _build

_lib = None

SPX_OK, SPX_ERR_INVALID_ARG, SPX_ERR_UNSUPPORTED, SPX_ERR_WORKSPACE, SPX_ERR_CUDA, SPX_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
SPX_PLAN_COLD_START, SPX_PLAN_PREFETCH_OVERLAP, SPX_PLAN_FINAL_CLEANUP = 0, 1, 2
SPX_PLAN_EVICT, SPX_PLAN_LOAD = 0, 1


class SpxError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class W4Experts(C.Structure):
    _fields_ = [("packed", C.c_void_p), ("E", C.c_int), ("H", C.c_int), ("I", C.c_int), ("slice_cols", C.c_int),
                ("zeros", C.c_void_p)]


class F16Experts(C.Structure):
    _fields_ = [("packed", C.c_void_p), ("E", C.c_int), ("H", C.c_int), ("I", C.c_int),
                ("tc_packed", C.c_void_p)]


class GgufExperts(C.Structure):
    _fields_ = [("packed", C.c_void_p), ("E", C.c_int), ("H", C.c_int), ("I", C.c_int), ("gate_up_type", C.c_int)]


class Shared(C.Structure):
    _fields_ = [("packed", C.c_void_p), ("w_sgate", C.c_void_p), ("H", C.c_int), ("I_s", C.c_int),
                ("tc_packed", C.c_void_p)]


class PlanCfg(C.Structure):
    _fields_ = [("L", C.c_int), ("E", C.c_int), ("K", C.c_int), ("capacity", C.c_int), ("min_chunk", C.c_int),
                ("step_us", C.c_double), ("copy_us", C.c_double)]


class LayerArgs(C.Structure):
    _fields_ = [("mode", C.c_int), ("T", C.c_int), ("H", C.c_int), ("E", C.c_int), ("k", C.c_int),
                ("renorm", C.c_int), ("x", C.c_void_p), ("w_router", C.c_void_p), ("logits", C.c_void_p),
                ("w4", C.POINTER(W4Experts)), ("f16", C.POINTER(F16Experts)), ("shared", C.POINTER(Shared)),
                ("elb", C.c_void_p), ("L", C.c_int), ("layer", C.c_int),
                ("topk_ids", C.c_void_p), ("topk_w", C.c_void_p), ("counts", C.c_void_p),
                ("offsets", C.c_void_p), ("sorted_slots", C.c_void_p), ("active", C.c_void_p),
                ("n_active", C.c_void_p), ("out", C.c_void_p), ("ws", C.c_void_p), ("ws_bytes", C.c_size_t),
                ("ev_experts_begin", C.c_void_p), ("ev_experts_end", C.c_void_p),
                ("resident", C.c_void_p), ("ready", C.c_void_p), ("wait_budget_ns", C.c_uint64),
                ("gguf", C.POINTER(GgufExperts)), ("verify_launch", C.c_int)]


_SIGS = {
    "spx_status_string": (C.c_char_p, [C.c_int]),
    "spx_version": (C.c_int, []),
    "spx_last_cuda_error": (C.c_char_p, []),
    "spx_route_topk": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                 C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "spx_elb_accumulate": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_int, C.c_void_p]),
    "spx_elb_read": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "spx_elb_reset": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_void_p]),
    "spx_gather_by_expert": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p,
                                       C.c_void_p, C.c_void_p, C.c_void_p]),
    "spx_w4_packed_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int]),
    "spx_f16_packed_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int]),
    "spx_w4_repack": (C.c_int, [C.c_void_p] * 6 + [C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "spx_w4_zeros_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int]),
    "spx_gguf_packed_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int]),
    "spx_gguf_repack": (C.c_int, [C.c_void_p] * 3 + [C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "spx_w4_zeros_repack": (C.c_int, [C.c_void_p] * 3 + [C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "spx_f16_repack": (C.c_int, [C.c_void_p] * 3 + [C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "spx_workspace_size": (C.c_size_t, [C.c_int] * 6),
    "spx_workspace_size_tc": (C.c_size_t, [C.c_int] * 6),
    "spx_f16_tc_packed_bytes": (C.c_size_t, [C.c_int] * 3),
    "spx_f16_tc_repack": (C.c_int, [C.c_void_p] * 3 + [C.c_int] * 3 + [C.c_void_p, C.c_void_p]),
    "spx_shared_tc_repack": (C.c_int, [C.c_void_p] * 3 + [C.c_int] * 2 + [C.c_void_p, C.c_void_p]),
    "spx_shared_packed_bytes": (C.c_size_t, [C.c_int, C.c_int]),
    "spx_shared_repack": (C.c_int, [C.c_void_p] * 3 + [C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "spx_workspace_init": (C.c_int, [C.c_void_p, C.c_size_t, C.c_void_p]),
    "spx_workspace_status": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p]),
    "spx_moe_draft_w4a16": (C.c_int, [C.c_void_p, C.c_int, C.POINTER(W4Experts), C.c_int] + [C.c_void_p] * 5 +
                            [C.c_void_p, C.c_size_t, C.c_void_p]),
    "spx_moe_draft_gguf": (C.c_int, [C.c_void_p, C.c_int, C.POINTER(GgufExperts), C.c_int] + [C.c_void_p] * 5 +
                            [C.c_void_p, C.c_size_t, C.c_void_p]),
    "spx_moe_verify_fp16": (C.c_int, [C.c_void_p, C.c_int, C.POINTER(F16Experts), C.c_int] + [C.c_void_p] * 5 +
                            [C.c_void_p, C.c_size_t, C.c_void_p]),
    "spx_combine": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.POINTER(Shared), C.c_int, C.c_int,
                              C.c_int, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "spx_moe_layer": (C.c_int, [C.POINTER(LayerArgs), C.c_void_p]),
    "spx_moe_layer_noalloc": (C.c_int, [C.POINTER(LayerArgs), C.c_void_p]),
    "spx_noalloc_init": (C.c_int, []),
    "spx_plan_prefetch": (C.c_int, [C.POINTER(PlanCfg), C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_int,
                                    C.POINTER(C.c_int), C.POINTER(C.c_int), C.POINTER(C.c_int)]),
    "spx_prefetch_issue": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p,
                                     C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p]),
    "spx_noalloc_status": (C.c_int, [C.c_void_p, C.c_void_p]),
}


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libspx.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        p = path or library_path()
        if not os.path.exists(p):
            raise ImportError(f"libspx.so is not built ({p}); run quantized_expert_gb300.build.build() "
                              "(or __graft_entry__.build()) first -- there is no fallback path")
        L = C.CDLL(p)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def exported_symbols() -> list[str]:
    return list(_SIGS)


def status_string(st: int) -> str:
    return load().spx_status_string(st).decode()


def _chk(st: int, what: str):
    if st != SPX_OK:
        if st == SPX_ERR_CUDA:
            what = f"{what} [{load().spx_last_cuda_error().decode()}]"
        raise SpxError(st, what)


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libspx takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libspx takes contiguous tensors")
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


# ------------------------------------------------------------------ API ----
def spx_version() -> int:
    return load().spx_version()


def spx_workspace_size(T: int, H: int, I: int = 0, E: int = 1, k: int = 1, I_s: int = 0) -> int:
    return load().spx_workspace_size(T, H, I, E, k, I_s)


def new_workspace(T: int, H: int, I: int = 0, E: int = 1, k: int = 1, I_s: int = 0, device="cuda",
                  stream=None, tc: bool = False) -> torch.Tensor:
    """Allocate (through torch) and zero a workspace for up to T tokens
    (tc: for verify calls forced onto the tensor-memory launches)."""
    n = (load().spx_workspace_size_tc if tc else spx_workspace_size)(T, H, I, E, k, I_s)
    if n == 0:
        raise SpxError(SPX_ERR_UNSUPPORTED, "spx_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    spx_workspace_init(ws, stream)
    return ws


def spx_workspace_init(ws: torch.Tensor, stream=None):
    _chk(load().spx_workspace_init(_p(ws), ws.numel(), _stream(stream)), "spx_workspace_init")


def spx_workspace_status(ws: torch.Tensor, stream=None) -> int:
    out = torch.zeros(1, dtype=torch.int32, device=ws.device)
    _chk(load().spx_workspace_status(_p(ws), _p(out), _stream(stream)), "spx_workspace_status")
    return int(out.item())


def spx_route_topk(x, w_router, logits, T, H, E, k, renorm, topk_ids, topk_w, ws, stream=None):
    _chk(load().spx_route_topk(_p(x), _p(w_router), _p(logits), T, H, E, k, int(bool(renorm)), _p(topk_ids),
                               _p(topk_w), _p(ws), ws.numel() if ws is not None else 0, _stream(stream)),
         "spx_route_topk")


def spx_elb_accumulate(elb, layer, topk_ids, stream=None):
    L, E = elb.shape
    T, k = topk_ids.shape
    _chk(load().spx_elb_accumulate(_p(elb), L, E, layer, _p(topk_ids), T, k, _stream(stream)), "spx_elb_accumulate")


def spx_elb_read(elb, dst, stream=None):
    L, E = elb.shape
    dptr = dst.data_ptr()
    _chk(load().spx_elb_read(_p(elb), L, E, dptr, _stream(stream)), "spx_elb_read")


def spx_elb_reset(elb, stream=None):
    L, E = elb.shape
    _chk(load().spx_elb_reset(_p(elb), L, E, _stream(stream)), "spx_elb_reset")


def spx_gather_by_expert(topk_ids, E, counts, offsets, sorted_slots, active, n_active, stream=None):
    T, k = topk_ids.shape
    _chk(load().spx_gather_by_expert(_p(topk_ids), T, k, E, _p(counts), _p(offsets), _p(sorted_slots), _p(active),
                                     _p(n_active), _stream(stream)), "spx_gather_by_expert")


@dataclass
class PackedW4:
    buf: torch.Tensor
    E: int
    H: int
    I: int
    S: int
    zeros: torch.Tensor | None = None  # repacked per-group zero points (None: zero point 8)

    def cstruct(self) -> W4Experts:
        return W4Experts(self.buf.data_ptr(), self.E, self.H, self.I, self.S, _p(self.zeros))


SPX_GGUF_Q8_0, SPX_GGUF_Q2_K, SPX_GGUF_Q4_K = 0, 1, 2


@dataclass
class PackedGguf:
    buf: torch.Tensor
    E: int
    H: int
    I: int
    gate_up_type: int  # SPX_GGUF_Q8_0, SPX_GGUF_Q2_K or SPX_GGUF_Q4_K; down is Q8_0

    def cstruct(self) -> GgufExperts:
        return GgufExperts(self.buf.data_ptr(), self.E, self.H, self.I, self.gate_up_type)


@dataclass
class PackedF16:
    buf: torch.Tensor
    E: int
    H: int
    I: int
    tc: torch.Tensor | None = None  # tile pack of the tensor-memory verify launches

    def cstruct(self) -> F16Experts:
        return F16Experts(self.buf.data_ptr(), self.E, self.H, self.I, _p(self.tc))


@dataclass
class PackedShared:
    buf: torch.Tensor
    w_sgate: torch.Tensor | None
    H: int
    I_s: int
    tc: torch.Tensor | None = None  # tile pack of the tensor-memory verify launches

    def cstruct(self) -> Shared:
        return Shared(self.buf.data_ptr(), _p(self.w_sgate), self.H, self.I_s, _p(self.tc))


def spx_w4_repack(qw_gate, s_gate, qw_up, s_up, qw_down, s_down, slice_cols=32, stream=None) -> PackedW4:
    """Canonical GPTQ tensors ([E][K/8][N] int32, [E][K/128][N] fp16 as int16/uint16 bits) -> packed units."""
    E, H8, I = qw_gate.shape
    H = H8 * 8
    n = load().spx_w4_packed_bytes(E, H, I, slice_cols)
    if n == 0:
        raise SpxError(SPX_ERR_UNSUPPORTED, "spx_w4_packed_bytes")
    buf = torch.empty(n, dtype=torch.uint8, device=qw_gate.device)
    _chk(load().spx_w4_repack(_p(qw_gate), _p(s_gate), _p(qw_up), _p(s_up), _p(qw_down), _p(s_down), E, H, I,
                              slice_cols, _p(buf), _stream(stream)), "spx_w4_repack")
    return PackedW4(buf, E, H, I, slice_cols)


def spx_w4_zeros_repack(w4: PackedW4, qz_gate, qz_up, qz_down, stream=None) -> PackedW4:
    """Canonical qzeros ([E][K/128][N/8] int32 per matrix, low nibble first) -> the
    same experts with zero points attached (a new PackedW4 sharing w4's weights)."""
    n = load().spx_w4_zeros_bytes(w4.E, w4.H, w4.I, w4.S)
    if n == 0:
        raise SpxError(SPX_ERR_UNSUPPORTED, "spx_w4_zeros_bytes")
    buf = torch.empty(n, dtype=torch.uint8, device=w4.buf.device)
    _chk(load().spx_w4_zeros_repack(_p(qz_gate), _p(qz_up), _p(qz_down), w4.E, w4.H, w4.I, w4.S, _p(buf),
                                    _stream(stream)), "spx_w4_zeros_repack")
    return PackedW4(w4.buf, w4.E, w4.H, w4.I, w4.S, buf)


def spx_gguf_repack(w_gate, w_up, w_down, gate_up_type=SPX_GGUF_Q8_0, stream=None) -> PackedGguf:
    """Canonical GGUF experts -> packed for the draft launch: gate, up uint8
    [E][I][H/32][34] (Q8_0), [E][I][H/256][84] (Q2_K) or [E][I][H/256][144]
    (Q4_K); down [E][H][I/32][34] (Q8_0)."""
    E, I, nb, bb = w_gate.shape
    H = nb * (32 if gate_up_type == SPX_GGUF_Q8_0 else 256)
    n = load().spx_gguf_packed_bytes(E, H, I, gate_up_type)
    if n == 0:
        raise SpxError(SPX_ERR_UNSUPPORTED, "spx_gguf_packed_bytes")
    buf = torch.empty(n, dtype=torch.uint8, device=w_gate.device)
    _chk(load().spx_gguf_repack(_p(w_gate), _p(w_up), _p(w_down), E, H, I, gate_up_type, _p(buf), _stream(stream)),
         "spx_gguf_repack")
    return PackedGguf(buf, E, H, I, gate_up_type)


def spx_f16_tc_repack(w_gate, w_up, w_down, stream=None) -> torch.Tensor:
    """Canonical [E][I][H], [E][I][H], [E][H][I] fp16 -> the tile pack of the
    tensor-memory verify launches (uint8 tensor)."""
    E, I, H = w_gate.shape
    n = load().spx_f16_tc_packed_bytes(E, H, I)
    if n == 0:
        raise SpxError(SPX_ERR_UNSUPPORTED, "spx_f16_tc_packed_bytes")
    buf = torch.empty(n, dtype=torch.uint8, device=w_gate.device)
    _chk(load().spx_f16_tc_repack(_p(w_gate), _p(w_up), _p(w_down), E, H, I, _p(buf), _stream(stream)),
         "spx_f16_tc_repack")
    return buf


def spx_f16_repack(w_gate, w_up, w_down, stream=None, tc=False) -> PackedF16:
    """Canonical [E][I][H], [E][I][H], [E][H][I] fp16 -> packed units (tc: also
    the tile pack of the tensor-memory verify launches)."""
    E, I, H = w_gate.shape
    n = load().spx_f16_packed_bytes(E, H, I)
    if n == 0:
        raise SpxError(SPX_ERR_UNSUPPORTED, "spx_f16_packed_bytes")
    buf = torch.empty(n, dtype=torch.uint8, device=w_gate.device)
    _chk(load().spx_f16_repack(_p(w_gate), _p(w_up), _p(w_down), E, H, I, _p(buf), _stream(stream)), "spx_f16_repack")
    return PackedF16(buf, E, H, I, spx_f16_tc_repack(w_gate, w_up, w_down, stream) if tc else None)


def pack_shared(w_gate, w_up, w_down, w_sgate=None, stream=None, tc=False) -> PackedShared:
    """Shared expert [I_s][H], [I_s][H], [H][I_s] fp16 -> packed (spx_shared_repack);
    tc as spx_f16_repack."""
    I_s, H = w_gate.shape
    n = load().spx_shared_packed_bytes(H, I_s)
    if n == 0:
        raise SpxError(SPX_ERR_UNSUPPORTED, "spx_shared_packed_bytes")
    buf = torch.empty(n, dtype=torch.uint8, device=w_gate.device)
    _chk(load().spx_shared_repack(_p(w_gate), _p(w_up), _p(w_down), H, I_s, _p(buf), _stream(stream)),
         "spx_shared_repack")
    return PackedShared(buf, w_sgate, H, I_s, spx_f16_tc_repack(w_gate[None], w_up[None], w_down[None], stream)
                        if tc else None)


def spx_moe_draft_w4a16(x, w: PackedW4, k, offsets, sorted_slots, active, n_active, y_sorted, ws, stream=None):
    """INT4 draft experts on gathered tokens: y_sorted [T*k][H] fp32, one row per
    sorted slot (the gather arrays come from spx_gather_by_expert)."""
    T = x.shape[0]
    cs = w.cstruct()
    _chk(load().spx_moe_draft_w4a16(_p(x), T, C.byref(cs), k, _p(offsets), _p(sorted_slots), _p(active),
                                    _p(n_active), _p(y_sorted), _p(ws), ws.numel(), _stream(stream)),
         "spx_moe_draft_w4a16")


def spx_moe_draft_gguf(x, w: PackedGguf, k, offsets, sorted_slots, active, n_active, y_sorted, ws, stream=None):
    """spx_moe_draft_w4a16 with GGUF draft experts."""
    T = x.shape[0]
    cs = w.cstruct()
    _chk(load().spx_moe_draft_gguf(_p(x), T, C.byref(cs), k, _p(offsets), _p(sorted_slots), _p(active),
                                   _p(n_active), _p(y_sorted), _p(ws), ws.numel(), _stream(stream)),
         "spx_moe_draft_gguf")


def spx_moe_verify_fp16(x, w: PackedF16, k, offsets, sorted_slots, active, n_active, y_sorted, ws, stream=None):
    """FP16 verify experts on gathered tokens (each expert's weights read once
    for all of its tokens); output as spx_moe_draft_w4a16."""
    T = x.shape[0]
    cs = w.cstruct()
    _chk(load().spx_moe_verify_fp16(_p(x), T, C.byref(cs), k, _p(offsets), _p(sorted_slots), _p(active),
                                    _p(n_active), _p(y_sorted), _p(ws), ws.numel(), _stream(stream)),
         "spx_moe_verify_fp16")


def spx_combine(y_sorted, sorted_slots, topk_w, x, shared: PackedShared | None, T, H, k, out, ws, stream=None):
    cs = shared.cstruct() if shared is not None else None
    _chk(load().spx_combine(_p(y_sorted), _p(sorted_slots), _p(topk_w), _p(x), C.byref(cs) if cs else None, T, H, k,
                            _p(out), _p(ws), ws.numel(), _stream(stream)), "spx_combine")


@dataclass
class Routing:
    """Caller-owned routing buffers of one layer call."""
    topk_ids: torch.Tensor
    topk_w: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    sorted_slots: torch.Tensor
    active: torch.Tensor
    n_active: torch.Tensor

    @staticmethod
    def empty(T, E, k, device="cuda") -> "Routing":
        i32 = dict(dtype=torch.int32, device=device)
        return Routing(torch.empty(T, k, **i32), torch.empty(T, k, dtype=torch.float32, device=device),
                       torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(T * k, **i32),
                       torch.empty(E, **i32), torch.empty(1, **i32))


def layer_args(mode, x, E, k, renorm, logits, routing: Routing, out, ws, w4: PackedW4 | None = None,
               f16: PackedF16 | None = None, shared: PackedShared | None = None, w_router=None, elb=None,
               layer=0, events=None, resident=None, ready=None, wait_budget_ns=0, gguf: PackedGguf | None = None,
               verify_launch=0):
    """Build (and keep alive) the argument block of one spx_moe_layer call.
    Draft experts are INT4 (w4) or GGUF (gguf), one of the two.
    resident (uint8 [E]) and ready (int32/uint32 [E]) are the optional
    cache-aware expert order and ready flags; wait_budget_ns bounds every
    device-side wait (0 = the library default).  verify_launch: 0 automatic,
    1 the expert launch, 2 the tensor-memory launches (needs the tile packs
    on f16 and shared)."""
    T, H = x.shape
    keep = []
    a = LayerArgs()
    a.mode, a.T, a.H, a.E, a.k, a.renorm = mode, T, H, E, k, int(bool(renorm))
    a.x, a.w_router, a.logits = _p(x), _p(w_router), _p(logits)
    if w4 is not None:
        s4 = w4.cstruct()
        keep.append(s4)
        a.w4 = C.pointer(s4)
    if gguf is not None:
        sg = gguf.cstruct()
        keep.append(sg)
        a.gguf = C.pointer(sg)
    if f16 is not None:
        s16 = f16.cstruct()
        keep.append(s16)
        a.f16 = C.pointer(s16)
    if shared is not None:
        ss = shared.cstruct()
        keep.append(ss)
        a.shared = C.pointer(ss)
    if elb is not None:
        a.elb, a.L, a.layer = _p(elb), elb.shape[0], layer
    r = routing
    a.topk_ids, a.topk_w, a.counts, a.offsets = _p(r.topk_ids), _p(r.topk_w), _p(r.counts), _p(r.offsets)
    a.sorted_slots, a.active, a.n_active = _p(r.sorted_slots), _p(r.active), _p(r.n_active)
    a.out, a.ws, a.ws_bytes = _p(out), _p(ws), ws.numel()
    if events is not None:
        a.ev_experts_begin, a.ev_experts_end = events[0].cuda_event, events[1].cuda_event
        keep.append(events)
    a.resident, a.ready, a.wait_budget_ns = _p(resident), _p(ready), int(wait_budget_ns)
    a.verify_launch = int(verify_launch)
    return a, keep


def spx_moe_layer(args: LayerArgs, stream=None):
    _chk(load().spx_moe_layer(C.byref(args), _stream(stream)), "spx_moe_layer")


def spx_noalloc_init():
    """Set-up of the no-allocation layer call on the current device (once, at
    start-up, before any stream capture): loads the library's kernels and its
    fixed scratch array onto the device."""
    _chk(load().spx_noalloc_init(), "spx_noalloc_init")


def spx_moe_layer_noalloc(args: LayerArgs, stream=None):
    """The same layer with the library's fixed scratch instead of args.ws (for
    callers that cannot allocate device memory); spx_noalloc_init() must have
    run on the device.  See include/spx.h."""
    _chk(load().spx_moe_layer_noalloc(C.byref(args), _stream(stream)), "spx_moe_layer_noalloc")


def spx_noalloc_status(out: torch.Tensor, stream=None):
    """Enqueue a copy of the fixed scratch's status word into `out` (one int32
    on the device, or pinned host memory); read it after the stream syncs."""
    _chk(load().spx_noalloc_status(C.c_void_p(out.data_ptr()), _stream(stream)), "spx_noalloc_status")


# ----------------------------------------------------------- prefetch plan --
def spx_plan_prefetch(cfg: PlanCfg, elb, steps_done: int, cached):
    """One planning call at a draft-chunk boundary (host numpy arrays: elb
    uint32 [L][E], cached uint8 [L][E], updated in place).  Returns (phase,
    actions int32 [n][3] = layer, expert, SPX_PLAN_LOAD/EVICT, next_chunk)."""
    import numpy as np
    elb = np.ascontiguousarray(elb, dtype=np.uint32)
    if cached.dtype != np.uint8 or not cached.flags.c_contiguous:
        raise ValueError("cached must be a contiguous uint8 array")
    cap = 2 * cfg.L * cfg.E
    acts = np.zeros((cap, 3), np.int32)
    n, chunk, phase = C.c_int(), C.c_int(), C.c_int()
    _chk(load().spx_plan_prefetch(C.byref(cfg), elb.ctypes.data, int(steps_done), cached.ctypes.data,
                                  acts.ctypes.data, cap, C.byref(n), C.byref(chunk), C.byref(phase)),
         "spx_plan_prefetch")
    return phase.value, acts[:n.value].copy(), chunk.value


_HOST_FLAGS = None


def prefetch_host_flags():
    """The executor's page-locked flag constants {1,0,0,0, 0,0,0,0}."""
    global _HOST_FLAGS
    if _HOST_FLAGS is None:
        _HOST_FLAGS = torch.tensor([1, 0, 0, 0, 0, 0, 0, 0], dtype=torch.uint8).pin_memory()
    return _HOST_FLAGS


def spx_prefetch_issue(actions, host_experts, dev_experts, expert_bytes: int, ready, resident=None, stream=None):
    """Enqueue a plan's copies and flag updates on `stream` (host_experts: list
    of page-locked host tensors per layer; dev_experts: device tensors per
    layer; ready/resident: device [L][E])."""
    import numpy as np
    acts = np.ascontiguousarray(actions, dtype=np.int32)
    L = len(dev_experts)
    hp = (C.c_void_p * L)(*[t.data_ptr() for t in host_experts])
    dp = (C.c_void_p * L)(*[t.data_ptr() for t in dev_experts])
    E = ready.shape[-1]
    _chk(load().spx_prefetch_issue(acts.ctypes.data, int(acts.shape[0]), hp, dp, int(expert_bytes), _p(ready),
                                   _p(resident), C.c_void_p(prefetch_host_flags().data_ptr()), L, E,
                                   _stream(stream)), "spx_prefetch_issue")
