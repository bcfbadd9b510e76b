"""Brute-force numpy restatement of the attention, for tiny inputs only.

TEST INFRASTRUCTURE ONLY.  Written separately from ``gr_oracle.c`` (no
shared helpers) so that each can check the other.  Pure Python loops over
rows; every step is spelled out as the pages' three-stage attention reads:
follow the parent indices back to step 0 (GR-Inference blog, "system
design": BeamPath), gather the chain's K/V from BeamKV, put them after the
request's shared ContextKV, and take an ordinary softmax over the joined
keys (xGR review, "xAttention": shared + unshared + merge is exact).
"""

from __future__ import annotations

import math

import numpy as np


def _widen(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def chain_of(beam_path, widths, r, b, step):
    """Slots [a_0, ..., a_s] visited from beam b at `step` back to step 0."""
    slots = [b]
    slot = b
    for t in range(step, 0, -1):
        parent = int(beam_path[r, t, slot])
        if not 0 <= parent < int(widths[t - 1]):
            raise ValueError(f"parent {parent} outside [0, {widths[t - 1]}) at step {t}")
        slot = parent
        slots.append(slot)
    return slots[::-1]


def attention(inp, step):
    """Return (out [R, W_s, Hq, D], lse [R, W_s, Hq], anc [R, W_s, s+1])."""
    R, Hq, Hkv, D = (inp["num_requests"], inp["num_q_heads"], inp["num_kv_heads"],
                     inp["head_dim"])
    G = Hq // Hkv
    W_s = int(inp["widths"][step])
    scale = float(np.float32(inp["softmax_scale"]))
    q = _widen(inp["q"][step])
    out = np.zeros((R, W_s, Hq, D))
    lse = np.zeros((R, W_s, Hq))
    anc = np.zeros((R, W_s, step + 1), dtype=np.int32)
    for r in range(R):
        n_ctx = int(inp["ctx_len"][r])
        for b in range(W_s):
            slots = chain_of(inp["beam_path"], inp["widths"], r, b, step)
            anc[r, b] = slots
            for h in range(Hq):
                g = h // G
                keys = [_widen(inp["ctx_k"][r, g, j]) for j in range(n_ctx)]
                vals = [_widen(inp["ctx_v"][r, g, j]) for j in range(n_ctx)]
                for t, a in enumerate(slots):
                    keys.append(_widen(inp["beam_k"][r, t, a, g]))
                    vals.append(_widen(inp["beam_v"][r, t, a, g]))
                scores = [scale * float(np.dot(q[r, b, h], k)) for k in keys]
                top = max(scores)
                weights = [math.exp(x - top) for x in scores]
                total = sum(weights)
                lse[r, b, h] = top + math.log(total)
                acc = np.zeros(D)
                for w, v in zip(weights, vals):
                    acc += (w / total) * v
                out[r, b, h] = acc
    return out, lse, anc
