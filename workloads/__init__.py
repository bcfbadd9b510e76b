"""Seeded synthetic inputs for large-beam decode attention.

This module draws random inputs only. It holds none of the attention
arithmetic: both the CPU oracle (``oracle/``) and the CUDA path
(``beam_decode_attention_gb300``) consume what it returns, and neither
imports the other.

Geometry follows the workloads the GR-Inference blog ("GR-Inference",
system design section) and the SID-GR Inference README (section 9, Nsight
breakdown) describe: Qwen3-0.6B / 1.7B / 4B attention heads, beam widths of
128 to 900, contexts of 1k to 4k tokens, three decode steps, a first step
that expands from the single prefill row.

Recipe (fixed, so that any two runs draw the same bits):

* ``numpy.random.Generator(PCG64(seed))`` with ``seed = 1000 + index`` where
  ``index`` is the workload's position in :data:`WORKLOADS`.
* Draw order: context lengths (ragged workloads only, integers uniform in
  ``[lc_lo, lc_hi]``), ``ctx_k``, ``ctx_v``, then for each step ``t``:
  ``beam_k[t]``, ``beam_v[t]``, ``q[t]``, ``parents[t]``.
* Values are standard normal float32 rounded to bfloat16 (round to nearest,
  ties to even) and stored as ``uint16`` bit patterns.
* Parents at step 0 are all 0 (every beam expands from the one prefill row);
  at step ``t >= 1`` they are uniform in ``[0, W[t-1])``.
* Storage that no active row may read is poisoned: bf16 NaN for K/V slots
  past a context length or past the step's width, ``-1`` for unused
  BeamPath entries.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

BF16_NAN = np.uint16(0x7FC0)


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    num_requests: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    lc: int                     # fixed context length (0 when ragged)
    lc_range: Optional[tuple]   # (lo, hi) inclusive when ragged
    widths: tuple               # active beam width per decode step
    description: str

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def steps(self) -> int:
        return len(self.widths)


WORKLOADS: List[WorkloadSpec] = [
    WorkloadSpec("tiny_r1_h4x2_d64_lc64_w4", 1, 4, 2, 64, 64, None, (4, 4, 4),
                 "1 request, Hq=4, Hkv=2, D=64, Lc=64, widths 4/4/4"),
    WorkloadSpec("qwen3_0.6b_r8_lc1024_w128", 8, 16, 8, 128, 1024, None, (128, 128, 128),
                 "Qwen3-0.6B heads, 8 requests, Lc=1024, width 128"),
    WorkloadSpec("qwen3_0.6b_r4_lc2048_w900", 4, 16, 8, 128, 2048, None, (900, 900, 900),
                 "Qwen3-0.6B heads, 4 requests, Lc=2048, width 900"),
    WorkloadSpec("qwen3_4b_r4_lc3072_w512", 4, 32, 8, 128, 3072, None, (512, 512, 512),
                 "Qwen3-4B heads, 4 requests, Lc=3072, width 512"),
    WorkloadSpec("qwen3_1.7b_r16_lc512-4096_w20-300-900", 16, 16, 8, 128, 0, (512, 4096),
                 (20, 300, 900),
                 "Qwen3-1.7B heads, 16 requests, Lc uniform in [512,4096], widths 20/300/900"),
]

WORKLOAD_BY_NAME: Dict[str, WorkloadSpec] = {w.name: w for w in WORKLOADS}
# the headline workload: beam width 900 over a 2048-token context
HEADLINE = WORKLOADS[2].name
SMALL = WORKLOADS[0].name


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16, nearest-even, returning uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    out = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def make_inputs(spec: WorkloadSpec, seed: Optional[int] = None,
                widths: Optional[Sequence[int]] = None) -> Dict[str, object]:
    """Draw one workload. Returns a dict of numpy arrays (bf16 as uint16).

    Keys: ``q`` (list per step, ``[R, W_t, Hq, D]``), ``ctx_k``/``ctx_v``
    (``[R, Hkv, Lc_max, D]``), ``ctx_len`` (``[R]`` int32), ``beam_k``/``beam_v``
    (``[R, S_max, W_max, Hkv, D]``), ``beam_path`` (``[R, S_max, W_max]``
    int32), ``widths`` (``[S_max]`` int32) and the shape scalars.
    """
    if seed is None:
        seed = 1000 + WORKLOADS.index(spec)
    W = tuple(int(w) for w in (widths if widths is not None else spec.widths))
    R, Hq, Hkv, D = spec.num_requests, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    S = len(W)
    W_max = max(W)
    rng = np.random.Generator(np.random.PCG64(seed))

    if spec.lc_range is not None:
        lo, hi = spec.lc_range
        ctx_len = rng.integers(lo, hi, size=R, endpoint=True).astype(np.int32)
    else:
        ctx_len = np.full(R, spec.lc, dtype=np.int32)
    lc_max = int(ctx_len.max()) if R else 0

    ctx_k = _normal_bf16(rng, (R, Hkv, lc_max, D))
    ctx_v = _normal_bf16(rng, (R, Hkv, lc_max, D))
    for r in range(R):
        ctx_k[r, :, ctx_len[r]:, :] = BF16_NAN
        ctx_v[r, :, ctx_len[r]:, :] = BF16_NAN

    beam_k = np.full((R, S, W_max, Hkv, D), BF16_NAN, dtype=np.uint16)
    beam_v = np.full((R, S, W_max, Hkv, D), BF16_NAN, dtype=np.uint16)
    beam_path = np.full((R, S, W_max), -1, dtype=np.int32)
    q = []
    for t in range(S):
        beam_k[:, t, :W[t]] = _normal_bf16(rng, (R, W[t], Hkv, D))
        beam_v[:, t, :W[t]] = _normal_bf16(rng, (R, W[t], Hkv, D))
        q.append(_normal_bf16(rng, (R, W[t], Hq, D)))
        if t == 0:
            beam_path[:, 0, :W[0]] = 0
        else:
            beam_path[:, t, :W[t]] = rng.integers(0, W[t - 1], size=(R, W[t])).astype(np.int32)

    return dict(
        name=spec.name, num_requests=R, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
        ctx_capacity=lc_max, step_capacity=S, beam_capacity=W_max,
        softmax_scale=float(np.float32(1.0 / np.sqrt(D))),
        q=q, ctx_k=ctx_k, ctx_v=ctx_v, ctx_len=ctx_len,
        beam_k=beam_k, beam_v=beam_v, beam_path=beam_path,
        widths=np.asarray(W, dtype=np.int32),
    )


def make_custom(R: int, Hq: int, Hkv: int, D: int, ctx_len: Sequence[int],
                widths: Sequence[int], seed: int, lc_max: Optional[int] = None,
                q_scale: float = 1.0) -> Dict[str, object]:
    """Same recipe with arbitrary shapes (edge cases in the tests).

    ``q_scale`` multiplies the float32 draw of ``q`` before rounding, which
    sharpens the softmax so that single keys carry visible weight.
    """
    W = tuple(int(w) for w in widths)
    S = len(W)
    W_max = max(W)
    ctx_len = np.asarray(ctx_len, dtype=np.int32)
    if lc_max is None:
        lc_max = int(ctx_len.max()) if R else 0
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx_k = _normal_bf16(rng, (R, Hkv, lc_max, D))
    ctx_v = _normal_bf16(rng, (R, Hkv, lc_max, D))
    for r in range(R):
        ctx_k[r, :, ctx_len[r]:, :] = BF16_NAN
        ctx_v[r, :, ctx_len[r]:, :] = BF16_NAN
    beam_k = np.full((R, S, W_max, Hkv, D), BF16_NAN, dtype=np.uint16)
    beam_v = np.full((R, S, W_max, Hkv, D), BF16_NAN, dtype=np.uint16)
    beam_path = np.full((R, S, W_max), -1, dtype=np.int32)
    q = []
    for t in range(S):
        beam_k[:, t, :W[t]] = _normal_bf16(rng, (R, W[t], Hkv, D))
        beam_v[:, t, :W[t]] = _normal_bf16(rng, (R, W[t], Hkv, D))
        q.append(f32_to_bf16_bits(
            rng.standard_normal(size=(R, W[t], Hq, D), dtype=np.float32) * np.float32(q_scale)))
        if t == 0:
            beam_path[:, 0, :W[0]] = 0
        else:
            beam_path[:, t, :W[t]] = rng.integers(0, W[t - 1], size=(R, W[t])).astype(np.int32)
    return dict(
        name="custom", num_requests=R, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
        ctx_capacity=lc_max, step_capacity=S, beam_capacity=W_max,
        softmax_scale=float(np.float32(1.0 / np.sqrt(D))),
        q=q, ctx_k=ctx_k, ctx_v=ctx_v, ctx_len=ctx_len,
        beam_k=beam_k, beam_v=beam_v, beam_path=beam_path,
        widths=np.asarray(W, dtype=np.int32),
    )


# --------------------------------------------------------------------------- beam selection
#
# Inputs of the beam-selection step that follows a decode forward: next-token
# logits of every active beam and the beams' cumulative log-probabilities.
# Recipe: Generator(PCG64(seed)); logits are float32 draws of N(0, sigma^2)
# (sigma = logit_std), then beam scores -|N(0, 1)| * 3 (cumulative
# log-probabilities are negative).  The vocabulary defaults to 151,936
# entries, the Qwen3 tokenizer's embedding rows; the pages measure a fixed
# width of 900 with full-vocabulary log-probabilities.

# --------------------------------------------------------------------------- layouts of the context and widths
#
# A paged ContextKV pool built from a dense [R, Hkv, Lc_max, D] context: the
# pages of all requests in a shuffled order (Generator(PCG64(seed))) with
# `extra_pages` spare pages, each [Hkv, page_size, D]; positions past Lc_max
# hold NaN.  Returns the pool [P, Hkv, page_size, D], the block table
# [R, pages_per_request] int32, pages_per_request and P.

def paged_pool(ctx: np.ndarray, page_size: int, extra_pages: int, seed: int):
    R, Hkv, Lc, D = ctx.shape
    ppr = max(1, -(-Lc // page_size))
    P = R * ppr + extra_pages
    order = np.random.Generator(np.random.PCG64(seed)).permutation(P)
    pool = np.full((P, Hkv, page_size, D), BF16_NAN, np.uint16)
    table = np.empty((R, ppr), np.int32)
    for r in range(R):
        for i in range(ppr):
            page = int(order[r * ppr + i])
            table[r, i] = page
            seg = ctx[r, :, i * page_size:(i + 1) * page_size]
            pool[page, :, :seg.shape[1]] = seg
    return pool, table, ppr, P


# Per-request widths over a workload laid out at each step's largest width:
# request r has width widths[r][t] at step t, and its BeamPath parents are
# folded into its own previous width (parent mod W[r][t-1]).  Returns the
# modified inputs and W int32 [R, S].

def make_ragged(spec: WorkloadSpec, widths: Sequence[Sequence[int]], seed: Optional[int] = None):
    W = np.asarray(widths, np.int32)
    if W.shape != (spec.num_requests, spec.steps) or np.any(W < 1):
        raise ValueError("widths must be [requests][steps] of positive widths")
    if np.any(W.max(axis=0) != np.asarray(spec.widths)):
        raise ValueError("each step's largest width must be the workload's width")
    inp = make_inputs(spec, seed)
    bp = inp["beam_path"]
    for r in range(W.shape[0]):
        for t in range(1, W.shape[1]):
            bp[r, t, :spec.widths[t]] %= W[r, t - 1]
    return inp, W


# A short decode loop: the inputs of `len(widths)` steps of append ->
# attention -> beam selection, for one fixed context.  Recipe:
# Generator(PCG64(seed)); draw order ctx_k, ctx_v (standard normal, bf16),
# then per step t: k_new[t], v_new[t] ([R, W_t, Hkv, D]), q[t]
# ([R, W_t, Hq, D]), all standard normal rounded to bf16, and for every step
# but the last the next-token logits[t] ([R, W_t, V] float32, N(0,
# logit_std^2)).  The loop starts from an empty BeamKV (NaN), a BeamPath of
# -1 with step 0's parents 0, and beam scores 0.

def make_decode_loop(R: int, Hq: int, Hkv: int, D: int, ctx_len: Sequence[int], widths: Sequence[int],
                     vocab: int, logit_std: float, seed: int) -> Dict[str, object]:
    W = tuple(int(w) for w in widths)
    S, W_max = len(W), max(W)
    ctx_len = np.asarray(ctx_len, dtype=np.int32)
    lc_max = int(ctx_len.max())
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx_k = _normal_bf16(rng, (R, Hkv, lc_max, D))
    ctx_v = _normal_bf16(rng, (R, Hkv, lc_max, D))
    for r in range(R):
        ctx_k[r, :, ctx_len[r]:, :] = BF16_NAN
        ctx_v[r, :, ctx_len[r]:, :] = BF16_NAN
    k_new, v_new, q, logits = [], [], [], []
    for t in range(S):
        k_new.append(_normal_bf16(rng, (R, W[t], Hkv, D)))
        v_new.append(_normal_bf16(rng, (R, W[t], Hkv, D)))
        q.append(_normal_bf16(rng, (R, W[t], Hq, D)))
        if t + 1 < S:
            logits.append(rng.standard_normal(size=(R, W[t], vocab), dtype=np.float32) * np.float32(logit_std))
    beam_path = np.full((R, S, W_max), -1, dtype=np.int32)
    beam_path[:, 0, :W[0]] = 0
    return dict(
        name="decode_loop", num_requests=R, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
        ctx_capacity=lc_max, step_capacity=S, beam_capacity=W_max,
        softmax_scale=float(np.float32(1.0 / np.sqrt(D))),
        ctx_k=ctx_k, ctx_v=ctx_v, ctx_len=ctx_len,
        beam_k=np.full((R, S, W_max, Hkv, D), BF16_NAN, dtype=np.uint16),
        beam_v=np.full((R, S, W_max, Hkv, D), BF16_NAN, dtype=np.uint16),
        beam_path=beam_path, widths=np.asarray(W, dtype=np.int32),
        k_new=k_new, v_new=v_new, q=q, logits=logits,
        beam_scores=np.zeros((R, W[0]), dtype=np.float32), vocab=int(vocab),
    )


SELECT_HEADLINE = dict(num_requests=4, width=900, vocab=151936, next_width=900)


def make_select_inputs(num_requests: int, width: int, vocab: int, seed: int,
                       logit_std: float = 2.0) -> Dict[str, np.ndarray]:
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = rng.standard_normal(size=(num_requests, width, vocab), dtype=np.float32)
    if logit_std != 1.0:
        logits *= np.float32(logit_std)
    scores = (-np.abs(rng.standard_normal(size=(num_requests, width), dtype=np.float32))
              * np.float32(3.0))
    return dict(logits=logits, beam_scores=scores)


# --------------------------------------------------------------------------- item-constrained selection
#
# A synthetic SID catalogue: `items` items, each a path of `levels` codes in
# [0, codebook) drawn uniformly (Generator(PCG64(seed))); the codes of level l
# are the vocabulary tokens token_base + l * codebook + code (the SID tokens
# sit at the end of the vocabulary).  The trie of the distinct paths is
# returned in CSR form with nodes numbered level by level (root 0), each
# node's edges sorted by token.

SELECT_TRIE_HEADLINE = dict(num_requests=4, width=900, vocab=151936, next_width=900,
                            codebook=256, levels=3, items=200_000, level=1)


def make_sid_trie(items: int, levels: int, codebook: int, vocab: int, seed: int):
    rng = np.random.Generator(np.random.PCG64(seed))
    codes = rng.integers(0, codebook, size=(items, levels), dtype=np.int64)
    token_base = vocab - levels * codebook
    if token_base < 0:
        raise ValueError("vocabulary smaller than the SID tokens")
    # nodes level by level: the distinct prefixes of each length
    level_nodes = [np.array([0])]
    prefix_id = {(): 0}
    edges = {}   # node -> list of (token, child)
    next_id = 1
    for lv in range(levels):
        prefixes = np.unique(codes[:, :lv + 1], axis=0)
        ids = []
        for p in map(tuple, prefixes):
            parent = prefix_id[p[:-1]]
            prefix_id[p] = next_id
            edges.setdefault(parent, []).append((int(token_base + lv * codebook + p[-1]), next_id))
            ids.append(next_id)
            next_id += 1
        level_nodes.append(np.array(ids))
    offsets = np.zeros(next_id + 1, np.int32)
    tokens, children = [], []
    for n in range(next_id):
        for t, c in sorted(edges.get(n, [])):
            tokens.append(t)
            children.append(c)
        offsets[n + 1] = len(tokens)
    return dict(offsets=offsets, tokens=np.array(tokens, np.int32), children=np.array(children, np.int32),
                num_nodes=next_id, level_nodes=level_nodes)


def make_trie_select_inputs(num_requests: int, width: int, vocab: int, trie, level: int, seed: int,
                            logit_std: float = 2.0) -> Dict[str, np.ndarray]:
    """Logits and beam scores as make_select_inputs, plus each beam's trie
    node: a uniformly drawn node of the given level (0 = the root)."""
    d = make_select_inputs(num_requests, width, vocab, seed, logit_std)
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    nodes = trie["level_nodes"][level]
    d["beam_node"] = nodes[rng.integers(0, len(nodes), size=(num_requests, width))].astype(np.int32)
    return d
