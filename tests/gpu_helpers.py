"""Helpers for the GPU parity tests: upload seeded inputs, repack them through
the library, and compare library outputs with the CPU oracle.

Tolerance (fp32 accumulate, fp16 activations and intermediate):
  max |gpu - ref| <= 1e-2 * max |ref|   and
  sum |gpu - ref| / sum |ref| <= 1e-3   (mean relative error, the stable form).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import spx_workloads as W
from quantized_expert_gb300 import spx

MAX_REL = 1e-2
MEAN_REL = 1e-3


def dev_f16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_close(gpu, ref, what: str, max_rel=MAX_REL, mean_rel=MEAN_REL) -> dict:
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    err = np.abs(gpu - ref)
    scale = np.abs(ref).max()
    st = dict(max_err=float(err.max()), max_ref=float(scale),
              mean_rel=float(err.sum() / max(np.abs(ref).sum(), 1e-300)))
    assert st["max_err"] <= max_rel * scale, f"{what}: {st}"
    assert st["mean_rel"] <= mean_rel, f"{what}: {st}"
    return st


def f16_out(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().astype(np.float64)


class Layer:
    """One synthetic layer: host experts (for the oracle) and packed device
    weights (for the library).  Only experts in `needed` are generated; the
    others are zero on the device (the kernels never read them)."""

    def __init__(self, shape: W.LayerShape, layer: int = 0, needed=None, draft=True, verify=True, slice_cols=32,
                 zeros=False, gguf=None):
        self.shape = s = shape
        self.layer = layer
        needed = sorted(set(range(s.E) if needed is None else needed))
        self.needed = needed
        self.w4_host = {e: W.gen_w4_expert(s, layer, e) for e in needed} if (draft or s.verify_is_dequant) else {}
        self.gguf = None
        if gguf:  # GGUF draft experts instead of INT4: "q8_0", or "q2_k" / "q4_k" gate/up with a Q8_0 down
            assert draft and not zeros and not (verify and s.verify_is_dequant)
            gen = {"q8_0": W.gen_q8_expert, "q2_k": W.gen_q2k_expert, "q4_k": W.gen_q4k_expert}[gguf]
            self.w4_host = {e: gen(s, layer, e) for e in needed}
        self.zeros = zeros
        if zeros:  # asymmetric INT4: per-group zero points on every draft expert
            assert draft and not (verify and s.verify_is_dequant)
            for e in needed:
                self.w4_host[e] = dict(self.w4_host[e], **W.gen_w4_zeros(s, layer, e))
        self.f16_host = {}
        if verify:
            for e in needed:
                self.f16_host[e] = (oracle.f16_copy_of_w4(self.w4_host[e]) if s.verify_is_dequant
                                    else W.gen_f16_expert(s, layer, e))
        self.shared_host = W.gen_shared(s, layer)
        self.router_host = W.gen_router(s, layer) if s.logits == "router" else None
        self.w4 = self.f16 = self.shared = None
        if draft and gguf:
            self.gguf = self._pack_gguf(gguf)
        elif draft:
            self.w4 = self._pack_w4(slice_cols)
        if verify:
            self.f16 = self._pack_f16()
        if self.shared_host is not None:
            sh = self.shared_host
            self.shared = spx.pack_shared(dev_f16(sh["w_gate"]), dev_f16(sh["w_up"]), dev_f16(sh["w_down"]),
                                          dev_f16(sh["w_sgate"]) if "w_sgate" in sh else None,
                                          tc=s.I_s % 64 == 0 and s.H % 128 == 0)
        self.w_router = dev_f16(self.router_host) if self.router_host is not None else None

    def _pack_w4(self, S):
        s = self.shape
        E, H, I = s.E, s.H, s.I
        qg = np.zeros((E, H // 8, I), np.int32)
        qu = np.zeros_like(qg)
        qd = np.zeros((E, I // 8, H), np.int32)
        sg = np.zeros((E, H // 128, I), np.uint16)
        su = np.zeros_like(sg)
        sd = np.zeros((E, I // 128, H), np.uint16)
        for e, ex in self.w4_host.items():
            qg[e], sg[e], qu[e], su[e], qd[e], sd[e] = (ex["qw_gate"], ex["s_gate"], ex["qw_up"], ex["s_up"],
                                                        ex["qw_down"], ex["s_down"])
        p = spx.spx_w4_repack(dev(qg), dev(sg.view(np.int16)), dev(qu), dev(su.view(np.int16)), dev(qd),
                              dev(sd.view(np.int16)), slice_cols=S)
        if self.zeros:
            zg = np.zeros((E, H // 128, I // 8), np.int32)
            zu = np.zeros_like(zg)
            zd = np.zeros((E, I // 128, H // 8), np.int32)
            for e, ex in self.w4_host.items():
                zg[e], zu[e], zd[e] = ex["qz_gate"], ex["qz_up"], ex["qz_down"]
            p = spx.spx_w4_zeros_repack(p, dev(zg), dev(zu), dev(zd))
        torch.cuda.synchronize()
        return p

    def _pack_gguf(self, kind):
        s = self.shape
        E, H, I = s.E, s.H, s.I
        blk, pre, ty = {"q8_0": ((H // 32, 34), "q8_", spx.SPX_GGUF_Q8_0),
                        "q2_k": ((H // 256, 84), "q2k_", spx.SPX_GGUF_Q2_K),
                        "q4_k": ((H // 256, 144), "q4k_", spx.SPX_GGUF_Q4_K)}[kind]
        wg = np.zeros((E, I) + blk, np.uint8)
        wu = np.zeros_like(wg)
        wd = np.zeros((E, H, I // 32, 34), np.uint8)
        for e, ex in self.w4_host.items():
            wg[e], wu[e], wd[e] = ex[pre + "gate"], ex[pre + "up"], ex["q8_down"]
        p = spx.spx_gguf_repack(dev(wg), dev(wu), dev(wd), ty)
        torch.cuda.synchronize()
        return p

    def _pack_f16(self):
        s = self.shape
        E, H, I = s.E, s.H, s.I
        wg = np.zeros((E, I, H), np.uint16)
        wu = np.zeros_like(wg)
        wd = np.zeros((E, H, I), np.uint16)
        for e, ex in self.f16_host.items():
            wg[e], wu[e], wd[e] = ex["w_gate"], ex["w_up"], ex["w_down"]
        # the tile pack of the tensor-memory verify launches where the shape allows one
        p = spx.spx_f16_repack(dev_f16(wg), dev_f16(wu), dev_f16(wd), tc=I % 64 == 0 and H % 128 == 0)
        torch.cuda.synchronize()
        return p

    def oracle_layer(self, mode, x, logits=None, elb=None):
        s = self.shape
        if mode == "draft":
            expert = lambda e: self.w4_host[e]  # noqa: E731
        else:
            expert = lambda e: self.f16_host[e]  # noqa: E731
        return oracle.moe_layer(mode, x, s.k, s.renorm, expert, s.E, logits=logits, w_router=self.router_host,
                                shared=self.shared_host, elb=elb, layer=self.layer)


def needed_experts(shape: W.LayerShape, logits_list=None, x_list=None, layer=0):
    """Experts the oracle routes to for the given inputs (to limit generation)."""
    out = set()
    if shape.logits == "router":
        wr = W.gen_router(shape, layer)
        for x in x_list:
            ids, _ = oracle.route_topk(oracle.router_logits(x, wr), shape.k, shape.renorm)
            out |= set(ids.reshape(-1).tolist())
    else:
        for lg in logits_list:
            ids, _ = oracle.route_topk(np.asarray(lg, np.float64), shape.k, shape.renorm)
            out |= set(ids.reshape(-1).tolist())
    return sorted(out)
