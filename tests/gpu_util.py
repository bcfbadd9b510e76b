"""Helpers for the GPU tests: move a seeded workload to the device, run the
library through its C ABI, read the results back."""

from __future__ import annotations

import numpy as np
import torch

import beam_decode_attention_gb300 as gr


def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class DeviceWorkload:
    """The workload's tensors on cuda:0 (bf16 as int16 bit patterns)."""

    def __init__(self, inp):
        self.inp = inp
        self.shape = gr.Shape.of(inp)
        self.ctx_k = to_dev(inp["ctx_k"])
        self.ctx_v = to_dev(inp["ctx_v"])
        self.ctx_len = to_dev(inp["ctx_len"])
        self.beam_k = to_dev(inp["beam_k"])
        self.beam_v = to_dev(inp["beam_v"])
        self.beam_path = to_dev(inp["beam_path"])
        self.q = [to_dev(x) for x in inp["q"]]
        self.widths = [int(w) for w in inp["widths"]]

    def outputs(self, step, guard=0):
        R, Hq, D = self.inp["num_requests"], self.inp["num_q_heads"], self.inp["head_dim"]
        W_s = self.widths[step]
        n = R * W_s * Hq
        out = torch.full((n * D + 2 * guard,), 0x5A5A, dtype=torch.int16, device="cuda")
        lse = torch.full((n + 2 * guard,), 7.25, dtype=torch.float32, device="cuda")
        return out, lse

    def run(self, step, guard=0, stream=None, workspace=None):
        """Returns (out float32 [R, W_s, Hq, D], lse [R, W_s, Hq]) as numpy."""
        R, Hq, D = self.inp["num_requests"], self.inp["num_q_heads"], self.inp["head_dim"]
        W_s = self.widths[step]
        n = R * W_s * Hq
        out, lse = self.outputs(step, guard)
        out_v = out[guard:guard + n * D]
        lse_v = lse[guard:guard + n]
        if workspace is None:
            ws_bytes = gr.gr_decode_attn_workspace_size(self.shape, self.widths, step)
            workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
        gr.gr_decode_attn(self.shape, self.q[step], self.ctx_k, self.ctx_v, self.ctx_len,
                          self.beam_k, self.beam_v, self.beam_path, self.widths, step,
                          out_v, lse_v, workspace, stream=stream)
        torch.cuda.synchronize()
        if guard:
            assert torch.all(out[:guard] == 0x5A5A) and torch.all(out[guard + n * D:] == 0x5A5A), \
                "write outside out"
            assert torch.all(lse[:guard] == 7.25) and torch.all(lse[guard + n:] == 7.25), \
                "write outside lse"
        o = out_v.cpu().numpy().view(np.uint16)
        o = (o.astype(np.uint32) << 16).view(np.float32).reshape(R, W_s, Hq, D)
        return o, lse_v.cpu().numpy().reshape(R, W_s, Hq)

    def ancestors(self, step):
        R = self.inp["num_requests"]
        W_s = self.widths[step]
        anc = torch.full((R, W_s, step + 1), -7, dtype=torch.int32, device="cuda")
        gr.gr_resolve_ancestors(self.shape, self.beam_path, self.widths, step, anc)
        torch.cuda.synchronize()
        return anc.cpu().numpy()


def bf16_half_ulp(x):
    """Half a unit in the last place of bf16 (8 significant bits) at |x|: the
    largest error of rounding the exact value x to a bf16 output."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(np.maximum(e, -133.0) - 8.0), 0.0)


def compare(out, lse, ref_out, ref_lse, tol_out=1e-2, tol_lse=1e-3):
    """Asserts the parity gate and returns a small report.

    out: |out - oracle| <= tol_out + half a bf16 ulp of the oracle value.
    The output format itself cannot hold the exact result: at |out| >= 4 a
    bf16 step is 2^-5, so even the exactly computed, correctly rounded
    result can sit 0.0156 from the fp64 oracle.  The 1e-2 gate therefore
    bounds the error the kernel adds beyond that rounding.  lse (fp32):
    |lse - oracle| <= tol_lse.  The plain max-abs errors are reported too.
    """
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse)), "non-finite output"
    diff = np.abs(out.astype(np.float64) - ref_out)
    e_out = float(np.max(diff)) if out.size else 0.0
    excess = float(np.max(diff - bf16_half_ulp(ref_out))) if out.size else 0.0
    e_lse = float(np.max(np.abs(lse.astype(np.float64) - ref_lse))) if lse.size else 0.0
    assert excess <= tol_out, (f"max |out - oracle| beyond the bf16 output rounding = {excess:.3e} > {tol_out} "
                               f"(max-abs {e_out:.3e})")
    assert e_lse <= tol_lse, f"max |lse - oracle| = {e_lse:.3e} > {tol_lse}"
    return dict(max_abs_out=e_out, max_out_beyond_rounding=excess, max_abs_lse=e_lse)
