"""Seeded synthetic workloads for the Specter per-layer MoE expert path.

This module holds layer shapes and random draws only.  It contains no step
of the method's arithmetic (no dequantisation, routing, MLP or combine), so
the CPU oracle (``oracle/``) and the CUDA library (``quantized_expert_gb300``)
can both be fed from it without sharing any code.

Shapes follow the three MoE models named in the richland.au post "Specter
previews expert routing with an INT4 copy of the model itself" (section
"What shipped": DeepSeek-V2-Lite, Qwen1.5-MoE-A2.7B, Phi-3.5-MoE; GPTQ INT4
with group size 128 for the routed experts, FP16 routers and shared experts)
and the speculation depths from the ai.info summary of the Specter paper
("Main Findings": best K = 16 / 8 / 16, so verify runs T = K + 1 tokens).

Recipe (every array is a pure function of ``(shape.seed, tags...)``):

* activations ``x``            fp16 N(0, 1)
* router / shared-gate weights  fp16 N(0, 0.02)
* INT4 codes                   uniform on 0..15 (a uniform 32-bit word is 8
                               uniform nibbles), fp16 scales U(0.005, 0.02),
                               zero point 8 (fixed, no qzeros tensor)
* FP16 verify / shared weights fp16 N(0, 0.02)
* drawn router logits          ``ln p_rank(e) + Gumbel(0, 1)`` in fp32, with
                               ``p_r ~ r^-1.1`` over a seeded permutation
                               ("zipf") or 4 hot experts at ``ln a = 1.1510``
                               and the rest at 0 ("hot"; a = 3.1614 makes the
                               hot experts' expected share of top-2 picks 50%).

Every fp16 value is drawn in float64 and rounded once to fp16 by numpy.
Each (layer, tensor, expert) has its own stream, so any single expert can be
regenerated on the host without drawing the others.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
import math

import numpy as np

__all__ = [
    "LayerShape", "CONFIGS", "rng_for", "gen_x", "gen_router", "gen_shared_gate",
    "gen_logits", "gen_w4_expert", "gen_f16_expert", "gen_shared", "cycle_logits",
    "draft_logits", "verify_logits",
]

# stream tags (part of the seeding key, never of the arithmetic)
(TAG_X, TAG_ROUTER, TAG_LOGITS, TAG_W4, TAG_F16, TAG_SHARED, TAG_SGATE, TAG_PERM, TAG_ZEROS, TAG_Q8,
 TAG_Q2K, TAG_Q4K) = range(1, 13)
HOT_LOG_A = 1.1510  # ln a, a = 3.1614
ZIPF_S = 1.1


@dataclass(frozen=True)
class LayerShape:
    """One synthetic MoE layer.

    ``logits``: "router" = computed from a router weight (x . Wr^T),
    "zipf" / "hot" = drawn directly (see module docstring).
    ``verify_is_dequant``: the FP16 verify weights are FP16 copies of the
    dequantised INT4 draft weights (produced by the consumer, not here).
    """
    name: str
    H: int
    I: int
    E: int
    k: int
    renorm: bool
    I_s: int
    shared_gate: bool
    T_draft: int
    T_verify: int
    logits: str
    seed: int
    layers: int = 1
    verify_is_dequant: bool = False

    @property
    def K(self) -> int:  # speculation depth
        return self.T_verify - 1


CONFIGS = {
    # tiny layer: H=256, I=512, E=8, top-2 + renorm, no shared expert, T=4
    "tiny": LayerShape("tiny", 256, 512, 8, 2, True, 0, False, 4, 4, "router", 0,
                       verify_is_dequant=True),
    # DeepSeek-V2-Lite-shaped: 64 experts top-6, 2 shared experts (I_s = 2*1408)
    "deepseek_v2_lite": LayerShape("deepseek_v2_lite", 2048, 1408, 64, 6, False, 2816, False,
                                   1, 17, "zipf", 1),
    # Qwen1.5-MoE-A2.7B-shaped: 60 experts top-4, sigmoid-gated shared expert I_s=5632
    "qwen15_moe": LayerShape("qwen15_moe", 2048, 1408, 60, 4, False, 5632, True,
                             1, 9, "router", 2),
    # Phi-3.5-MoE-shaped: 16 experts top-2 + renorm, no shared expert
    "phi35_moe": LayerShape("phi35_moe", 4096, 6400, 16, 2, True, 0, False,
                            1, 17, "hot", 3),
    # 26-layer DeepSeek-V2-Lite-shaped stack, K=16 draft steps then one verify
    "deepseek_v2_lite_x26": LayerShape("deepseek_v2_lite_x26", 2048, 1408, 64, 6, False, 2816,
                                       False, 1, 17, "zipf", 4, layers=26),
}


def rng_for(shape: LayerShape, *tags: int) -> np.random.Generator:
    """Independent PCG64 stream keyed by the shape's seed and integer tags."""
    ss = np.random.SeedSequence([int(shape.seed)] + [int(t) for t in tags])
    return np.random.Generator(np.random.PCG64(ss))


def _f16_normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    v = rng.standard_normal(size=shape, dtype=np.float64)
    if std != 1.0:
        v = v * std
    return v.astype(np.float16).view(np.uint16)


def gen_x(shape: LayerShape, T: int, layer: int = 0, step: int = 0, which: int = 0) -> np.ndarray:
    """Activations [T, H] as fp16 bit patterns (uint16). ``which``: 0 draft, 1 verify."""
    return _f16_normal(rng_for(shape, TAG_X, layer, step, which, T), (T, shape.H), 1.0)


def gen_router(shape: LayerShape, layer: int = 0) -> np.ndarray:
    """Router weight [E, H] fp16 bits, N(0, 0.02)."""
    return _f16_normal(rng_for(shape, TAG_ROUTER, layer), (shape.E, shape.H), 0.02)


def gen_shared_gate(shape: LayerShape, layer: int = 0) -> np.ndarray:
    """Shared-expert sigmoid-gate weight [H] fp16 bits, N(0, 0.02)."""
    return _f16_normal(rng_for(shape, TAG_SGATE, layer), (shape.H,), 0.02)


def _gumbel(rng: np.random.Generator, shape) -> np.ndarray:
    u = rng.random(size=shape, dtype=np.float64)
    u = np.clip(u, 1e-300, 1.0 - 1e-16)
    return -np.log(-np.log(u))


def _popularity_log(shape: LayerShape, layer: int) -> np.ndarray:
    """Per-expert log-popularity offsets (fixed per layer)."""
    perm = rng_for(shape, TAG_PERM, layer).permutation(shape.E)
    logp = np.zeros(shape.E, dtype=np.float64)
    if shape.logits == "zipf":
        r = np.arange(1, shape.E + 1, dtype=np.float64)
        lw = -ZIPF_S * np.log(r)
        lw -= math.log(np.exp(lw).sum())
        logp[perm] = lw          # expert perm[r-1] has rank r
    elif shape.logits == "hot":
        logp[perm[:4]] = HOT_LOG_A
    else:
        raise ValueError(f"shape {shape.name} computes its logits from a router weight")
    return logp


def gen_logits(shape: LayerShape, T: int, layer: int = 0, step: int = 0, which: int = 0) -> np.ndarray:
    """Drawn router logits [T, E] float32 (only for 'zipf' / 'hot' shapes)."""
    logp = _popularity_log(shape, layer)
    g = _gumbel(rng_for(shape, TAG_LOGITS, layer, step, which, T), (T, shape.E))
    return (logp[None, :] + g).astype(np.float32)


def draft_logits(shape: LayerShape, layer: int, step: int) -> np.ndarray:
    """Logits [1, E] of draft step ``step`` (1-based) at ``layer`` in the K-step cycle."""
    return gen_logits(shape, 1, layer, step, 0)


def verify_logits(shape: LayerShape, layer: int) -> np.ndarray:
    """Verify logits [K+1, E]: tokens 0..K-1 reuse draft steps 1..K, token K is fresh."""
    rows = [draft_logits(shape, layer, s) for s in range(1, shape.K + 1)]
    rows.append(gen_logits(shape, 1, layer, shape.K + 1, 1))
    return np.concatenate(rows, axis=0)


cycle_logits = verify_logits


def _w4_matrix(rng: np.random.Generator, K: int, N: int):
    """GPTQ-style packed codes [K/8, N] int32 (uniform nibbles) and fp16 scales [K/128, N]."""
    q = rng.integers(0, 2 ** 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32).view(np.int32)
    s = rng.uniform(0.005, 0.02, size=(K // 128, N)).astype(np.float16).view(np.uint16)
    return q, s


def gen_w4_expert(shape: LayerShape, layer: int, e: int) -> dict:
    """INT4 draft expert e in the canonical GPTQ layout (zero point 8, group 128).

    ``qw_gate``/``qw_up``: [H/8, I] int32 (code k at bits 4*(k%8) of row k/8),
    ``s_gate``/``s_up``: [H/128, I]; ``qw_down``: [I/8, H], ``s_down``: [I/128, H].
    """
    H, I = shape.H, shape.I
    rng = rng_for(shape, TAG_W4, layer, e)
    qg, sg = _w4_matrix(rng, H, I)
    qu, su = _w4_matrix(rng, H, I)
    qd, sd = _w4_matrix(rng, I, H)
    return dict(qw_gate=qg, s_gate=sg, qw_up=qu, s_up=su, qw_down=qd, s_down=sd)


def gen_w4_zeros(shape: LayerShape, layer: int, e: int) -> dict:
    """Per-group zero points of INT4 expert e (the asymmetric, AWQ-style form),
    packed like GPTQ qzeros: ``qz_gate``/``qz_up`` [H/128, I/8] int32,
    ``qz_down`` [I/128, H/8], zero point of column n at bits 4*(n%8) of word
    n/8, uniform over 0..15."""
    H, I = shape.H, shape.I
    rng = rng_for(shape, TAG_ZEROS, layer, e)

    def words(K, N):
        return rng.integers(0, 2 ** 32, size=(K // 128, N // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)

    return dict(qz_gate=words(H, I), qz_up=words(H, I), qz_down=words(I, H))


def _q8_matrix(rng: np.random.Generator, N: int, K: int) -> np.ndarray:
    """GGUF Q8_0 blocks of an [N][K] matrix: uint8 [N][K/32][34], each block a
    little-endian fp16 scale U(0.0003, 0.00125) then 32 int8 codes uniform
    over -128..127 (weights of the INT4 experts' magnitude)."""
    d = rng.uniform(0.0003, 0.00125, size=(N, K // 32)).astype(np.float16).view(np.uint16)
    codes = rng.integers(0, 256, size=(N, K // 32, 32), dtype=np.uint8)
    out = np.empty((N, K // 32, 34), np.uint8)
    out[:, :, 0] = d & 0xFF
    out[:, :, 1] = d >> 8
    out[:, :, 2:] = codes
    return out


def gen_q8_expert(shape: LayerShape, layer: int, e: int) -> dict:
    """GGUF Q8_0 draft expert e in [out][in] order: ``q8_gate``/``q8_up``
    [I][H/32][34] uint8, ``q8_down`` [H][I/32][34]."""
    H, I = shape.H, shape.I
    rng = rng_for(shape, TAG_Q8, layer, e)
    return dict(q8_gate=_q8_matrix(rng, I, H), q8_up=_q8_matrix(rng, I, H), q8_down=_q8_matrix(rng, H, I))


def _q2k_matrix(rng: np.random.Generator, N: int, K: int) -> np.ndarray:
    """GGUF Q2_K super-blocks of an [N][K] matrix: uint8 [N][K/256][84]; the
    sub-block bytes and codes uniform, d U(0.001, 0.003) and dmin
    U(0.001, 0.004) fp16 little-endian (weights of the INT4 experts' scale)."""
    out = rng.integers(0, 256, size=(N, K // 256, 84), dtype=np.uint8)
    d = rng.uniform(0.001, 0.003, size=(N, K // 256)).astype(np.float16).view(np.uint16)
    dmin = rng.uniform(0.001, 0.004, size=(N, K // 256)).astype(np.float16).view(np.uint16)
    out[:, :, 80], out[:, :, 81] = d & 0xFF, d >> 8
    out[:, :, 82], out[:, :, 83] = dmin & 0xFF, dmin >> 8
    return out


def gen_q2k_expert(shape: LayerShape, layer: int, e: int) -> dict:
    """Draft expert e with GGUF Q2_K gate/up (``q2k_gate``/``q2k_up``
    [I][H/256][84] uint8) and a GGUF Q8_0 down projection (``q8_down``
    [H][I/32][34]): Q2_K rows need a multiple of 256 values, which the down
    rows (I values) of the 1408-wide shapes are not."""
    H, I = shape.H, shape.I
    rng = rng_for(shape, TAG_Q2K, layer, e)
    return dict(q2k_gate=_q2k_matrix(rng, I, H), q2k_up=_q2k_matrix(rng, I, H), q8_down=_q8_matrix(rng, H, I))


def _q4k_matrix(rng: np.random.Generator, N: int, K: int) -> np.ndarray:
    """GGUF Q4_K super-blocks of an [N][K] matrix: uint8 [N][K/256][144]; the
    scale/min bytes and codes uniform, d U(0.00015, 0.0004) and dmin
    U(0.0003, 0.001) fp16 little-endian (weights of the INT4 experts' scale)."""
    out = rng.integers(0, 256, size=(N, K // 256, 144), dtype=np.uint8)
    d = rng.uniform(0.00015, 0.0004, size=(N, K // 256)).astype(np.float16).view(np.uint16)
    dmin = rng.uniform(0.0003, 0.001, size=(N, K // 256)).astype(np.float16).view(np.uint16)
    out[:, :, 0], out[:, :, 1] = d & 0xFF, d >> 8
    out[:, :, 2], out[:, :, 3] = dmin & 0xFF, dmin >> 8
    return out


def gen_q4k_expert(shape: LayerShape, layer: int, e: int) -> dict:
    """Draft expert e with GGUF Q4_K gate/up (``q4k_gate``/``q4k_up``
    [I][H/256][144] uint8) and a GGUF Q8_0 down projection (``q8_down``
    [H][I/32][34]), for the reason given at gen_q2k_expert."""
    H, I = shape.H, shape.I
    rng = rng_for(shape, TAG_Q4K, layer, e)
    return dict(q4k_gate=_q4k_matrix(rng, I, H), q4k_up=_q4k_matrix(rng, I, H), q8_down=_q8_matrix(rng, H, I))


def gen_f16_expert(shape: LayerShape, layer: int, e: int) -> dict:
    """FP16 verify expert e, PyTorch [out, in] layout: gate/up [I, H], down [H, I]."""
    H, I = shape.H, shape.I
    rng = rng_for(shape, TAG_F16, layer, e)
    return dict(w_gate=_f16_normal(rng, (I, H), 0.02),
                w_up=_f16_normal(rng, (I, H), 0.02),
                w_down=_f16_normal(rng, (H, I), 0.02))


def gen_shared(shape: LayerShape, layer: int = 0) -> dict | None:
    """FP16 shared expert (all shared experts concatenated along I_s), [out, in] layout."""
    if shape.I_s == 0:
        return None
    H, I = shape.H, shape.I_s
    rng = rng_for(shape, TAG_SHARED, layer)
    d = dict(w_gate=_f16_normal(rng, (I, H), 0.02),
             w_up=_f16_normal(rng, (I, H), 0.02),
             w_down=_f16_normal(rng, (H, I), 0.02))
    if shape.shared_gate:
        d["w_sgate"] = gen_shared_gate(shape, layer)
    return d


def scaled(shape: LayerShape, **kw) -> LayerShape:
    """Copy of a shape with some fields replaced (small parity cases)."""
    return replace(shape, **kw)
