"""CPU oracle for the Specter per-layer MoE expert path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library (``quantized_expert_gb300``)
never imports it and shares no code with it: the arithmetic lives in the
plain C file ``spx_oracle.c`` (binary64, single thread); this module only
builds that file with gcc, marshals numpy arrays through ctypes, and chains
the steps in the order the pages give them:

    route (logits -> softmax -> top-k) -> ELB count -> gather by expert
    -> dequant + expert MLP per (token, expert) -> shared expert -> combine

Sources (page title + section): ai.info summary "Specter: Fast MoE Inference
via Quantization-Enabled Multi-Step Speculative Offloading", Key
Contributions 1-4, "Methodology in Plain English" and Main Findings (drafts
quantised by GPTQ, AWQ and GGUF at Q2, Q4 and Q8: the zero-point and GGUF
expert formats); richland.au "Specter previews expert routing with an INT4
copy of the model itself", "What shipped".

Parity status: every step has a pin in ``tests/test_oracle_pins.py`` (closed
forms, brute force, invariants, library routines, hand-derived format
fixtures under ``tests/golden/``); the design notes list them.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spx_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libspx_oracle.so")
_lib = None
_lock = threading.Lock()

_dp = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_fp = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_u16 = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i32 = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_u32 = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_u8 = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile spx_oracle.c with gcc (-O2, IEEE semantics: no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            L.orc_half_to_double.argtypes = [C.c_uint16]
            L.orc_half_to_double.restype = C.c_double
            L.orc_double_to_half.argtypes = [C.c_double]
            L.orc_double_to_half.restype = C.c_uint16
            L.orc_halves_to_doubles.argtypes = [_u16, _dp, C.c_int64]
            L.orc_doubles_to_halves.argtypes = [_dp, _u16, C.c_int64]
            L.orc_router_logits.argtypes = [_u16, _u16, C.c_int, C.c_int, C.c_int, _dp]
            L.orc_route_topk.argtypes = [_dp, C.c_int, C.c_int, C.c_int, C.c_int, _i32, _dp, C.c_void_p]
            L.orc_elb_accumulate.argtypes = [_u32, C.c_int, C.c_int, _i32, C.c_int, C.c_int]
            L.orc_gather_by_expert.argtypes = [_i32, C.c_int, C.c_int, C.c_int, _i32, _i32, _i32, _i32, _i32]
            L.orc_w4_dequant.argtypes = [_i32, _u16, C.c_int, C.c_int, _dp]
            L.orc_w4z_dequant.argtypes = [_i32, _u16, C.c_void_p, C.c_int, C.c_int, _dp]
            L.orc_swiglu_w4z.argtypes = [_u16, C.c_int, C.c_int, _i32, _u16, C.c_void_p, _i32, _u16, C.c_void_p,
                                         _i32, _u16, C.c_void_p, _dp, C.c_void_p]
            L.orc_swiglu_w4.argtypes = [_u16, C.c_int, C.c_int, _i32, _u16, _i32, _u16, _i32, _u16, _dp, C.c_void_p]
            L.orc_swiglu_f16.argtypes = [_u16, C.c_int, C.c_int, _u16, _u16, _u16, _dp, C.c_void_p]
            L.orc_q8_dequant.argtypes = [_u8, C.c_int, C.c_int, _dp]
            L.orc_swiglu_q8.argtypes = [_u16, C.c_int, C.c_int, _u8, _u8, _u8, _dp, C.c_void_p]
            L.orc_q2k_dequant.argtypes = [_u8, C.c_int, C.c_int, _dp]
            L.orc_q4k_dequant.argtypes = [_u8, C.c_int, C.c_int, _dp]
            L.orc_swiglu_gguf.argtypes = [_u16, C.c_int, C.c_int, C.c_int, _u8, C.c_int, _u8, C.c_int, _u8, _dp,
                                          C.c_void_p]
            L.orc_shared_gate.argtypes = [_u16, _u16, C.c_int]
            L.orc_shared_gate.restype = C.c_double
            L.orc_combine.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, C.c_void_p, C.c_void_p, _dp, _u16]
            _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- fp16 --
def half_to_double(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    lib().orc_halves_to_doubles(b.reshape(-1), out.reshape(-1), b.size)
    return out


def double_to_half(vals) -> np.ndarray:
    v = _c(vals, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().orc_doubles_to_halves(v.reshape(-1), out.reshape(-1), v.size)
    return out


# -------------------------------------------------------------- routing --
def router_logits(x, wr) -> np.ndarray:
    x = _c(x, np.uint16)
    wr = _c(wr, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    out = np.empty((T, E), np.float64)
    lib().orc_router_logits(x, wr, T, H, E, out)
    return out


def route_topk(logits, k: int, renorm: bool, want_probs: bool = False):
    """-> ids int32 [T,k], w float64 [T,k] (, probs [T,E])."""
    lg = _c(logits, np.float64)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    probs = np.empty((T, E), np.float64) if want_probs else None
    lib().orc_route_topk(lg, T, E, k, int(bool(renorm)), ids, w,
                         probs.ctypes.data if want_probs else None)
    return (ids, w, probs) if want_probs else (ids, w)


def elb_accumulate(elb: np.ndarray, layer: int, ids) -> None:
    assert elb.dtype == np.uint32 and elb.flags.c_contiguous
    ids = _c(ids, np.int32)
    T, k = ids.shape
    lib().orc_elb_accumulate(elb.reshape(-1), elb.shape[-1], layer, ids, T, k)


def gather_by_expert(ids, E: int) -> dict:
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    sorted_slots = np.empty(max(T * k, 1), np.int32)
    active = np.empty(max(E, 1), np.int32)
    n_active = np.zeros(1, np.int32)
    lib().orc_gather_by_expert(ids, T, k, E, counts, offsets, sorted_slots, active, n_active)
    return dict(counts=counts, offsets=offsets, sorted_slots=sorted_slots[:T * k],
                active=active[:E], n_active=int(n_active[0]))


# ----------------------------------------------------------- experts --
def w4_dequant(q, s, qz=None) -> np.ndarray:
    """W = (code - zero) * scale; qz [K/128][N/8] int32 zero points, or None
    for zero point 8."""
    q = _c(q, np.int32)
    s = _c(s, np.uint16)
    K, N = q.shape[0] * 8, q.shape[1]
    out = np.empty((K, N), np.float64)
    z = _c(qz, np.int32) if qz is not None else None
    lib().orc_w4z_dequant(q, s, z.ctypes.data if z is not None else None, K, N, out)
    return out


def swiglu_w4(x_row, ex: dict, want_h: bool = False):
    """INT4 expert MLP on one token; ex may carry qz_gate / qz_up / qz_down
    (per-group zero points), else zero point 8."""
    x_row = _c(x_row, np.uint16)
    H = x_row.shape[0]
    I = ex["qw_gate"].shape[1]
    y = np.empty(H, np.float64)
    h = np.empty(I, np.float64) if want_h else None
    zs = [_c(ex[k], np.int32) if ex.get(k) is not None else None for k in ("qz_gate", "qz_up", "qz_down")]
    zp = [z.ctypes.data if z is not None else None for z in zs]
    lib().orc_swiglu_w4z(x_row, H, I, _c(ex["qw_gate"], np.int32), _c(ex["s_gate"], np.uint16), zp[0],
                         _c(ex["qw_up"], np.int32), _c(ex["s_up"], np.uint16), zp[1],
                         _c(ex["qw_down"], np.int32), _c(ex["s_down"], np.uint16), zp[2], y,
                         h.ctypes.data if want_h else None)
    return (y, h) if want_h else y


def q8_dequant(w) -> np.ndarray:
    """GGUF Q8_0 matrix, uint8 [N][K/32][34] blocks ([out][in] order) -> W [N][K]."""
    w = _c(w, np.uint8)
    N, K = w.shape[0], w.shape[1] * 32
    out = np.empty((N, K), np.float64)
    lib().orc_q8_dequant(w, N, K, out)
    return out


def swiglu_q8(x_row, ex: dict, want_h: bool = False):
    """Q8_0 expert MLP on one token: ex holds q8_gate, q8_up [I][H/32][34] and
    q8_down [H][I/32][34] uint8 blocks."""
    x_row = _c(x_row, np.uint16)
    H = x_row.shape[0]
    I = ex["q8_gate"].shape[0]
    y = np.empty(H, np.float64)
    h = np.empty(I, np.float64) if want_h else None
    lib().orc_swiglu_q8(x_row, H, I, _c(ex["q8_gate"], np.uint8), _c(ex["q8_up"], np.uint8),
                        _c(ex["q8_down"], np.uint8), y, h.ctypes.data if want_h else None)
    return (y, h) if want_h else y


def q2k_dequant(w) -> np.ndarray:
    """GGUF Q2_K matrix, uint8 [N][K/256][84] super-blocks ([out][in] order) -> W [N][K]."""
    w = _c(w, np.uint8)
    N, K = w.shape[0], w.shape[1] * 256
    out = np.empty((N, K), np.float64)
    lib().orc_q2k_dequant(w, N, K, out)
    return out


def q4k_dequant(w) -> np.ndarray:
    """GGUF Q4_K matrix, uint8 [N][K/256][144] super-blocks ([out][in] order) -> W [N][K]."""
    w = _c(w, np.uint8)
    N, K = w.shape[0], w.shape[1] * 256
    out = np.empty((N, K), np.float64)
    lib().orc_q4k_dequant(w, N, K, out)
    return out


_GGUF_TYPE = {"q2k": 1, "q4k": 2}


def swiglu_kquant(x_row, ex: dict, want_h: bool = False):
    """Expert with K-quant gate/up (q2k_gate, q2k_up [I][H/256][84] or q4k_gate,
    q4k_up [I][H/256][144] uint8) and a Q8_0 down projection (q8_down
    [H][I/32][34])."""
    pre = "q2k" if "q2k_gate" in ex else "q4k"
    ty = _GGUF_TYPE[pre]
    x_row = _c(x_row, np.uint16)
    H = x_row.shape[0]
    I = ex[pre + "_gate"].shape[0]
    y = np.empty(H, np.float64)
    h = np.empty(I, np.float64) if want_h else None
    lib().orc_swiglu_gguf(x_row, H, I, ty, _c(ex[pre + "_gate"], np.uint8), ty, _c(ex[pre + "_up"], np.uint8), 0,
                          _c(ex["q8_down"], np.uint8), y, h.ctypes.data if want_h else None)
    return (y, h) if want_h else y


swiglu_q2k = swiglu_kquant
swiglu_q4k = swiglu_kquant


def swiglu_draft(x_row, ex: dict, want_h: bool = False):
    """The draft expert MLP in the expert's own format (Q2_K or Q4_K gate/up
    with Q8_0 down, Q8_0, or INT4)."""
    if "q2k_gate" in ex or "q4k_gate" in ex:
        return swiglu_kquant(x_row, ex, want_h)
    return swiglu_q8(x_row, ex, want_h) if "q8_gate" in ex else swiglu_w4(x_row, ex, want_h)


def swiglu_f16(x_row, ex: dict, want_h: bool = False):
    x_row = _c(x_row, np.uint16)
    H = x_row.shape[0]
    I = ex["w_gate"].shape[0]
    y = np.empty(H, np.float64)
    h = np.empty(I, np.float64) if want_h else None
    lib().orc_swiglu_f16(x_row, H, I, _c(ex["w_gate"], np.uint16), _c(ex["w_up"], np.uint16),
                         _c(ex["w_down"], np.uint16), y, h.ctypes.data if want_h else None)
    return (y, h) if want_h else y


def shared_gate(x_row, w_sgate) -> float:
    x_row = _c(x_row, np.uint16)
    return float(lib().orc_shared_gate(x_row, _c(w_sgate, np.uint16), x_row.shape[0]))


def combine(w, y_slot, gamma=None, sh=None):
    """-> (out float64 [T,H], out fp16 bits [T,H])."""
    w = _c(w, np.float64)
    T, k = w.shape
    y_slot = _c(y_slot, np.float64)
    H = y_slot.shape[-1]
    out = np.empty((T, H), np.float64)
    outh = np.empty((T, H), np.uint16)
    g = _c(gamma, np.float64) if gamma is not None else None
    s = _c(sh, np.float64) if sh is not None else None
    lib().orc_combine(T, H, k, w, y_slot.reshape(T * k, H),
                      g.ctypes.data if g is not None else None,
                      s.ctypes.data if s is not None else None, out, outh)
    return out, outh


def f16_copy_of_w4(ex: dict) -> dict:
    """FP16 copies of a dequantised INT4 expert in [out, in] layout (the tiny
    layer's verify weights): W rounded once to fp16, gate/up transposed to
    [I, H], down to [H, I]."""
    g = w4_dequant(ex["qw_gate"], ex["s_gate"])   # [H, I]
    u = w4_dequant(ex["qw_up"], ex["s_up"])       # [H, I]
    d = w4_dequant(ex["qw_down"], ex["s_down"])   # [I, H]
    return dict(w_gate=double_to_half(g.T), w_up=double_to_half(u.T), w_down=double_to_half(d.T))


# ------------------------------------------------------------- layer --
def moe_layer(mode: str, x, k: int, renorm: bool, expert, E: int, logits=None, w_router=None,
              shared=None, elb=None, layer: int = 0) -> dict:
    """One MoE layer for T tokens.

    mode: "draft" (INT4 routed experts, ``expert(e)`` returns the GPTQ dict)
    or "verify" (FP16 routed experts, ``expert(e)`` returns the [out,in] dict);
    a draft expert dict with ``q8_gate`` is a GGUF Q8_0 expert.
    ``logits`` (fp32 [T,E]) are used as given when ``w_router`` is None,
    otherwise computed from x . w_router^T.  ``shared``: dict of FP16 shared
    expert weights (+ optional ``w_sgate``) or None.  ``elb``: uint32 [L,E]
    counter table updated in place (draft steps feed it) or None.
    """
    x = _c(x, np.uint16)
    T, H = x.shape
    if w_router is not None:
        lg = router_logits(x, w_router)
    else:
        lg = np.asarray(logits, np.float32).astype(np.float64)
    ids, w = route_topk(lg, k, renorm)
    if elb is not None:
        elb_accumulate(elb, layer, ids)
    g = gather_by_expert(ids, E)
    mlp = swiglu_draft if mode == "draft" else swiglu_f16
    y_slot = np.zeros((T * k, H), np.float64)
    # experts in ascending id order; each expert's tokens in slot order
    for a in range(g["n_active"]):
        e = int(g["active"][a])
        ex = expert(e)
        for p in range(g["offsets"][e], g["offsets"][e + 1]):
            s = int(g["sorted_slots"][p])
            y_slot[s] = mlp(x[s // k], ex)
    gamma = sh = None
    if shared is not None:
        sh = np.stack([swiglu_f16(x[t], shared) for t in range(T)])
        if shared.get("w_sgate") is not None:
            gamma = np.array([shared_gate(x[t], shared["w_sgate"]) for t in range(T)])
    out, outh = combine(w, y_slot.reshape(T, k, H), gamma, sh)
    y_sorted = y_slot[g["sorted_slots"]]
    return dict(logits=lg, ids=ids, w=w, gather=g, y_slot=y_slot, y_sorted=y_sorted,
                gamma=gamma, sh=sh, out=out, out_half=outh)
