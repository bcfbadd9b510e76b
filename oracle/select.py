"""Oracle for beam selection (TEST INFRASTRUCTURE ONLY).

Only ``tests/`` and ``bench.py``'s CPU-baseline leg may import this module;
the product library never calls it and shares no code with it.

What it computes (SID-GR README, section 10 "TODO and Roadmap", the "beam
selection graph" row: log_softmax + topK + beam selection after each decode
forward; section 9 "Performance Breakdown", the "topK / beam selection"
bucket; xGR review, "xBeam": a size-BW selection over every beam's
candidates, with early termination of the sort as an optimisation that does
not change the result):

  for request r, active beam b < W_s with cumulative log-probability
  S[r, b] and next-token logits z[r, b, v] (v < V):
      lp[r, b, v]    = z[r, b, v] - ln sum_v' exp(z[r, b, v'])   (log_softmax)
      score[r, b, v] = S[r, b] + lp[r, b, v]
  the next W' beams of request r are the W' candidates (b, v) of largest
  score; equal scores are ordered by the smaller flat index b * V + v.  Each
  chosen candidate gives the next BeamPath entry (its parent b), its token v
  and its score, in that order.

Readings where the pages are silent (they list score normalisation, length
penalty and tie-break policy as open): no length penalty or normalisation;
ties go to the smaller flat index; a logit of -inf is a masked token (its
candidates rank last, by index), and a row needs at least one finite logit.

Everything here is fp64 numpy: the log-sum-exp is taken after subtracting
the row maximum, and the ordering is numpy's stable sort on (score, flat
index).  At full size (W_s * V in the hundreds of millions) ``top_candidates``
narrows each request with ``np.argpartition`` before the exact ordering.
"""

from __future__ import annotations

from typing import Tuple

import numpy as np


def log_softmax(z: np.ndarray) -> np.ndarray:
    """fp64 log_softmax over the last axis (row maximum subtracted first)."""
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    return z - (m + np.log(np.sum(np.exp(z - m), axis=-1, keepdims=True)))


def scores(logits: np.ndarray, beam_scores: np.ndarray) -> np.ndarray:
    """score[r, b, v] = S[r, b] + log_softmax(z[r, b, :])[v], fp64, [R, W_s, V]."""
    return np.asarray(beam_scores, dtype=np.float64)[..., None] + log_softmax(logits)


def _order(flat_scores: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Positions of `idx` sorted by score descending, then flat index ascending."""
    return np.lexsort((idx, -flat_scores[idx]))


def beam_select(logits: np.ndarray, beam_scores: np.ndarray,
                next_width: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Exact selection over every candidate (small and medium sizes).

    Returns parent int32 [R, W'], token int32 [R, W'], score fp64 [R, W'].
    """
    sc = scores(logits, beam_scores)
    R, W, V = sc.shape
    if not 1 <= next_width <= W * V:
        raise ValueError("next_width outside [1, W_s * V]")
    flat = sc.reshape(R, W * V)
    parent = np.empty((R, next_width), np.int32)
    token = np.empty((R, next_width), np.int32)
    best = np.empty((R, next_width), np.float64)
    allidx = np.arange(W * V)
    for r in range(R):
        pick = allidx[_order(flat[r], allidx)[:next_width]]
        parent[r], token[r], best[r] = pick // V, pick % V, flat[r, pick]
    return parent, token, best


def top_candidates(logits: np.ndarray, beam_scores: np.ndarray, next_width: int,
                   extra: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """The next_width + extra best candidates of each request, exactly ordered.

    For full-size inputs: each request's scores are narrowed with
    np.argpartition (every candidate scoring at least the cut is kept, so
    ties at the cut are not lost), then ordered exactly.  Returns the flat
    indices int64 [R, n] and the fp64 scores [R, n], n = next_width + extra
    (capped at W_s * V).
    """
    R, W, V = logits.shape
    n = min(next_width + extra, W * V)
    flats, vals = [], []
    for r in range(R):
        sc = scores(logits[r:r + 1], beam_scores[r:r + 1]).reshape(W * V)
        if n < W * V:
            part = np.argpartition(-sc, n - 1)[:n]
            cut = sc[part].min()
            part = np.nonzero(sc >= cut)[0]
        else:
            part = np.arange(W * V)
        keep = part[_order(sc, part)][:n]
        flats.append(keep)
        vals.append(sc[keep])
    return np.stack(flats), np.stack(vals)


# --------------------------------------------------------------------------- item-constrained selection
#
# GR-Inference blog, "kernel design" (the item-constrained fused kernel: the
# SID trie resident on the device in CSR form; prefix traversal, gather of
# the legal tokens and a local top-K, with no full-vocabulary mask); xGR
# review, "xBeam" (an item mask on the logits filters invalid token ids).
#
# Trie in CSR form: node n's children are the edges k in
# [offsets[n], offsets[n+1]), each with a token tokens[k] (strictly
# increasing within a node) and a child node children[k].  Beam b of request
# r sits at node beam_node[r, b] (the node its SID prefix reached; the root
# at the first step).  Its legal next tokens are that node's edge tokens, and
# masking every other logit to -inf before log_softmax means:
#
#     lp[r, b, k] = z[r, b, tokens[k]] - ln sum_{k' legal} exp(z[r, b, tokens[k']])
#     score       = S[r, b] + lp
#
# The next W' beams are the W' largest scores over every beam's legal
# candidates, equal scores ordered by the smaller flat index b * V + token;
# each keeps its parent b, its token, its score and its child node (the
# traversal advances one level per step).  A beam at a leaf has no
# candidates; when a request has fewer than W' candidates the remaining
# slots hold parent -1, token -1, score -inf and node -1.


def trie_select(logits: np.ndarray, beam_scores: np.ndarray, beam_node: np.ndarray,
                offsets: np.ndarray, tokens: np.ndarray, children: np.ndarray,
                next_width: int):
    """Returns parent, token, node (int32 [R, W']) and score (fp64 [R, W'])."""
    z = np.asarray(logits, dtype=np.float64)
    S = np.asarray(beam_scores, dtype=np.float64)
    R, W, V = z.shape
    parent = np.full((R, next_width), -1, np.int32)
    token = np.full((R, next_width), -1, np.int32)
    node = np.full((R, next_width), -1, np.int32)
    best = np.full((R, next_width), -np.inf)
    for r in range(R):
        flats, vals, kids = [], [], []
        for b in range(W):
            n = int(beam_node[r, b])
            ks = np.arange(int(offsets[n]), int(offsets[n + 1]))
            if ks.size == 0:
                continue
            toks = np.asarray(tokens)[ks]
            lz = z[r, b, toks]
            m = lz.max()
            lp = lz - (m + np.log(np.sum(np.exp(lz - m))))
            flats.append(b * V + toks.astype(np.int64))
            vals.append(S[r, b] + lp)
            kids.append(np.asarray(children)[ks])
        if not flats:
            continue
        flat = np.concatenate(flats)
        val = np.concatenate(vals)
        kid = np.concatenate(kids)
        order = np.lexsort((flat, -val))[:next_width]
        n_take = order.size
        parent[r, :n_take] = flat[order] // V
        token[r, :n_take] = flat[order] % V
        node[r, :n_take] = kid[order]
        best[r, :n_take] = val[order]
    return parent, token, node, best
