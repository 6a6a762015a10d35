"""Helpers for the GPU parity tests: upload the seeded inputs, run the layer through the C ABI,
bring results back, and compute the fp64 oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import grouped_gemm_device_gb300 as g
from grouped_gemm_device_gb300 import synth
from oracle import moe as om

BF16_TOL = 5e-3
MX_TOL = 3e-2


def bf16_dev(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.cpu().numpy().astype(np.float64) if t.is_floating_point() else t.cpu().numpy()


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    if nb == 0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def act_params(cfg) -> om.ActParams:
    return om.ActParams(cfg.activation, cfg.beta, cfg.gate_max, cfg.lin_lo, cfg.lin_hi,
                        cfg.lin_offset)


class Inputs:
    def __init__(self, cfg: synth.LayerConfig, logits=None):
        self.cfg = cfg
        self.logits = synth.gen_logits(cfg) if logits is None else logits
        self.x = synth.gen_x(cfg)
        self.w1 = synth.gen_w1(cfg)
        self.w2 = synth.gen_w2(cfg)
        self.dy = synth.gen_dy(cfg)

    def oracle(self, backward=True, keep=True, recompute=False):
        c = self.cfg
        return om.layer(self.logits, om.bf16_to_f64(self.x), om.bf16_to_f64(self.w1),
                        om.bf16_to_f64(self.w2), c.k, act_params(c), mx=c.precision == "mxfp8",
                        align=c.align, dy=om.bf16_to_f64(self.dy) if backward else None,
                        keep_intermediates=keep, recompute=recompute)


class LayerRun:
    """Runs route -> fwd -> bwd for the inputs on cuda and keeps the results."""

    def __init__(self, inp: Inputs, T_max=None, sm_margin=0, backward=True, recompute=False):
        cfg = inp.cfg
        self.cfg = cfg
        self.desc = g.desc_from_config(cfg, T_max=T_max, sm_margin=sm_margin, recompute=recompute)
        self.layer = g.MoELayer(self.desc)
        self.w1p = g.pack_w1(bf16_dev(inp.w1), gated=cfg.gated, ilv=cfg.ilv)
        self.w2 = bf16_dev(inp.w2)
        self.logits_d = torch.from_numpy(inp.logits).cuda()
        self.x_d = bf16_dev(inp.x)
        self.dy_d = bf16_dev(inp.dy)
        self.T = cfg.T
        self.run(backward)

    def run(self, backward=True, sync=True):
        L = self.layer
        L.route_permute(self.logits_d, self.x_d, self.T)
        self.y = L.forward(self.w1p, self.w2, self.T)
        if backward:
            self.dx, self.dw1p, self.dw2, self.d_probs = L.backward(self.dy_d, self.w1p, self.w2,
                                                                    self.T)
        if sync:
            torch.cuda.synchronize()

    def dw1_logical(self):
        c = self.cfg
        out = torch.empty(c.E, c.H, c.N1, dtype=torch.bfloat16, device="cuda")
        g.moe_pack_fc1_weight(self.dw1p, out, c.E, c.H, c.F, int(c.gated), c.ilv, 1)
        torch.cuda.synchronize()
        return to_np(out)

    def ws(self, name, dtype, cols):
        R = self.layer.layout.R_cap
        return self.layer.ws_view(name, dtype, (R, cols) if cols else (R,))

    def unpack_cols(self, packed: np.ndarray) -> np.ndarray:
        """[rows, N1] in packed column order -> logical [gate | linear] order (test-side view
        of the documented interleave)."""
        c = self.cfg
        if not c.gated:
            return packed
        N1 = packed.shape[1]
        p = np.arange(N1)
        b = p // c.ilv
        logical = (b % 2) * c.F + (b // 2) * c.ilv + p % c.ilv
        out = np.empty_like(packed)
        out[:, logical] = packed
        return out


def check_weight_grads_16_byte_aligned(cfg):
    """Weight gradients written to buffers that are 16- but not 32-byte aligned take the
    128-bit store path of the GEMM epilogue; they must equal the 256-bit path bit for bit."""
    run = LayerRun(Inputs(cfg))
    dw1, dw2 = run.dw1p.clone(), run.dw2.clone()
    L = run.layer
    b1 = torch.zeros(L.dw1.numel() + 8, dtype=torch.bfloat16, device="cuda")
    b2 = torch.zeros(L.dw2.numel() + 8, dtype=torch.bfloat16, device="cuda")
    L.dw1 = b1[8:].view(L.dw1.shape)
    L.dw2 = b2[8:].view(L.dw2.shape)
    assert L.dw1.data_ptr() % 32 == 16 and L.dw2.data_ptr() % 32 == 16
    run.run()
    assert torch.equal(run.dw1p, dw1) and torch.equal(run.dw2, dw2)
    assert not b1[:8].any() and not b2[:8].any()
