"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI and the oracle on
the same seeded inputs. Importing this module never touches the GPU by itself."""
from __future__ import annotations

import numpy as np
import torch

from block_scaled_fp8_moe_gb300 import synth
from oracle import formats as F
from oracle import moe as M

SWIGLU_REL = 1e-5          # pre-requant SwiGLU: |d| <= 1e-5 * max(|a_ref|, rms_row(a_ref))
OUT_REL_RMS = 2e-2         # final bf16 output: max |d| <= 2e-2 * rms(out_ref)


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy()


def oracle_weights(w_fp32: torch.Tensor, experts=None) -> M.ExpertWeights:
    """Oracle-side MXFP4 quantisation of fp32 expert weights [E, R, K] (only `experts` filled)."""
    E, R, K = w_fp32.shape
    codes = np.zeros((E, R, K // 2), dtype=np.uint8)
    scales = np.zeros((E, R, K // 32), dtype=np.uint8)
    for e in (range(E) if experts is None else experts):
        q, s = M.quant_mxfp4(w_fp32[e].detach().cpu().numpy())
        codes[e], scales[e] = q, s
    return M.ExpertWeights(codes, scales, cache=8)


class GpuLayer:
    """Inputs on the device, quantised and packed by the product kernels."""

    def __init__(self, inp: synth.MoeInputs, device="cuda"):
        from block_scaled_fp8_moe_gb300 import binding as B
        self.B = B
        cfg = inp.cfg
        self.cfg = cfg
        self.x = inp.x.to(device).contiguous()
        self.wr = inp.w_router.to(device).contiguous()
        self.bias = inp.bias.to(device).contiguous()
        self.dead = inp.dead.to(device).contiguous()
        w13 = inp.w13.to(device).contiguous()
        w2 = inp.w2.to(device).contiguous()
        self.layer = B.MoeLayer.from_fp32(self.wr, self.bias, w13, w2, cfg.k)
        self.q13, self.s13 = B.moe_quant_mxfp4(w13)
        self.q2, self.s2 = B.moe_quant_mxfp4(w2)

    def shape(self, T=None, flags=0):
        return self.layer.shape(self.cfg.T if T is None else T, flags)

    def forward(self, x=None, dead=None, inter=None, anchor=None, shared=None, side_stream=None):
        x = self.x if x is None else x
        return self.layer.forward(x, dead=dead, inter=inter, anchor=anchor, shared=shared, side_stream=side_stream)

    def run_steps(self, use_dead=True):
        """Route -> quant -> W13 (debug on) -> W2+combine through the four step entry points."""
        B = self.B
        cfg = self.cfg
        shp = self.shape(flags=B.MOE_FLAG_SWIGLU_DEBUG)
        ws = B.alloc_workspace(shp)
        dead = self.dead if use_dead else None
        plan = B.moe_route_topk(shp, self.x, self.wr, self.bias, dead, ws)
        xq, xs = B.moe_quant_mxfp8(self.x)
        S = cfg.T * cfg.k
        dbg = torch.full((max(S, 1), cfg.I), float("nan"), dtype=torch.float32, device=self.x.device)
        hq, hs = B.moe_w13_swiglu_grouped(shp, xq, xs, self.layer.w13p, self.layer.w13sp, plan, ws, debug=dbg)
        out = B.moe_w2_combine_grouped(shp, hq, hs, self.layer.w2p, self.layer.w2sp, plan, ws, dead=dead)
        B.moe_check_device_status(ws)
        return dict(plan=plan, xq=xq, xs=xs, hq=hq, hs=hs, dbg=dbg, out=out)


def oracle_forward(inp: synth.MoeInputs, tokens=None, w13=None, w2=None, use_dead=True, anchor=None, shared=None):
    cfg = inp.cfg
    x = bf16_to_np(inp.x)
    wr = bf16_to_np(inp.w_router)
    bias = inp.bias.cpu().numpy()
    dead = inp.dead.cpu().numpy().astype(bool) if use_dead else None
    if w13 is None or w2 is None:
        # quantise only the experts the requested tokens reach
        r = M.route(x if tokens is None else x[tokens], wr, bias, cfg.k)
        used = sorted(set(r.topk_idx.reshape(-1).tolist()))
        w13 = oracle_weights(inp.w13, used) if w13 is None else w13
        w2 = oracle_weights(inp.w2, used) if w2 is None else w2
    return (M.forward(x, wr, bias, cfg.k, w13, w2, cfg.I, dead=dead, tokens=tokens, anchor=anchor, shared=shared),
            w13, w2)


def assert_out_close(got: np.ndarray, ref_exact: np.ndarray, rel=OUT_REL_RMS):
    """The bf16 output must be the round-to-nearest-even image of a value within rel * rms of the
    oracle's exact (float64, unrounded) output: max-abs error <= rel * rms before the output's own
    rounding, so a rounding-boundary flip of the last bf16 bit is allowed like an FP8 requant flip.
    RNE is monotonic, so that is got in [bf16(ref - tol), bf16(ref + tol)]."""
    ref_exact = np.asarray(ref_exact, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref_exact ** 2))) if ref_exact.size else 0.0
    tol = rel * max(rms, 1e-30)
    lo = F.round_to_bf16(ref_exact - tol)
    hi = F.round_to_bf16(ref_exact + tol)
    bad = (got < lo) | (got > hi)
    err = float(np.max(np.abs(got - ref_exact))) if got.size else 0.0
    assert not np.any(bad), (f"{int(bad.sum())} outputs outside the rounding of exact +- {rel} * rms "
                             f"{rms:.4g}; max|d| = {err:.4g}")
    return err, rms


def e4m3_codes_match(got_q, got_s, ref_q, ref_s, flip_ok):
    """Requant codes must equal the oracle's except where the oracle marks a legitimate flip."""
    bad_q = (got_q != ref_q) & ~flip_ok
    nb = ref_s.shape[1]
    block_ok = flip_ok.reshape(flip_ok.shape[0], nb, F.BLOCK).any(-1)
    bad_s = (got_s[:, :nb] != ref_s) & ~block_ok
    return int(bad_q.sum()), int(bad_s.sum())
