"""The decode loop as the oracle runs it (test infrastructure).

For each decode step s (SID-GR Inference README, section 9: one decode step
is the attention call followed by log_softmax + top-K + beam selection;
GR-Inference blog, "system design": BeamKV grows by the token each beam adds,
BeamPath records each beam's parent):

  1. the step's new K/V go to BeamKV[:, s, :W_s] (the append);
  2. attention at step s (oracle.Oracle.decode_attn);
  3. before the last step, the beam selection over the step's logits
     (oracle.select.beam_select) gives BeamPath[:, s+1, :W_{s+1}] and the
     next beam scores.  The scores are kept in fp32 between steps, the type
     the selection's interface stores them in.

``margin`` is the smallest gap between consecutive scores among each
request's best W_{s+1} + 1 candidates, over every selection of the loop: when
it is far above the fp32 rounding of a score, the selection and its order
are fixed by the mathematics and any correct implementation picks the same
parents, tokens and slots.
"""

from __future__ import annotations

import numpy as np

import oracle
from oracle import select

CASES = {
    # widths 8 -> 32 -> 32 over a 50-token vocabulary, Qwen3-0.6B heads
    "w8-32-32_d128": dict(R=2, Hq=16, Hkv=8, D=128, ctx_len=[300, 777], widths=(8, 32, 32), vocab=50,
                          logit_std=4.0, seed=18),
    # widths 4 -> 64 -> 64 over 128 tokens, D = 64, four query heads per kv head
    "w4-64-64_d64": dict(R=3, Hq=8, Hkv=2, D=64, ctx_len=[129, 1000, 64], widths=(4, 64, 64), vocab=128,
                         logit_std=12.0, seed=19),
}


# a margin this wide is two orders of magnitude above the fp32 rounding of
# scores of magnitude < 100 summed over a vocabulary of <= 128 tokens
MARGIN = 5e-4


def make_case(name):
    import workloads
    c = CASES[name]
    return workloads.make_decode_loop(c["R"], c["Hq"], c["Hkv"], c["D"], c["ctx_len"], c["widths"], c["vocab"],
                                      c["logit_std"], c["seed"])


def run_oracle_loop(inp):
    """Returns (per-step records, margin, final state)."""
    orc = oracle.Oracle()
    R = inp["num_requests"]
    W = [int(w) for w in inp["widths"]]
    st = dict(inp)
    st["beam_k"], st["beam_v"] = inp["beam_k"].copy(), inp["beam_v"].copy()
    st["beam_path"] = inp["beam_path"].copy()
    scores = inp["beam_scores"]
    records, margin = [], np.inf
    for s in range(len(W)):
        st["beam_k"][:, s, :W[s]] = inp["k_new"][s]
        st["beam_v"][:, s, :W[s]] = inp["v_new"][s]
        out, lse, _ = orc.decode_attn(st, s)
        rec = dict(out=out, lse=lse)
        if s + 1 < len(W):
            par, tok, sco = select.beam_select(inp["logits"][s], scores, W[s + 1])
            flat = select.scores(inp["logits"][s], scores).reshape(R, -1)
            top = -np.sort(-flat, axis=1)[:, :W[s + 1] + 1]
            margin = min(margin, float(np.min(-np.diff(top, axis=1))))
            st["beam_path"][:, s + 1, :W[s + 1]] = par
            scores = sco.astype(np.float32)
            rec.update(parent=par, token=tok, score=sco)
        records.append(rec)
    return records, margin, st
