"""Pins for the CPU oracle: checks against facts other than the oracle itself.

Each pin takes an :class:`oracle.Oracle` and raises ``AssertionError`` when
the oracle disagrees with the mathematics.  ``tests/test_oracle_pins.py`` runs
them on the oracle; ``tests/test_oracle_mutants.py`` runs them on variants of
the oracle with one planted mistake each and requires that some pin fails.

No page prints a worked numerical example for this attention, so the pins
are closed forms, invariants, library routines for the special cases that
reduce to ordinary attention, a separately written brute force, and
hand-enumerated BeamPath chains.
"""

from __future__ import annotations

import math
import os

import numpy as np
import torch

import workloads
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _f64(bits):
    return workloads.bf16_bits_to_f32(bits).astype(np.float64)


def tiny_inputs(seed=1000):
    return workloads.make_inputs(workloads.WORKLOAD_BY_NAME[workloads.SMALL], seed=seed)


def load_hand_ancestors():
    """Parse tests/golden/ancestors_hand.txt into (inputs, expected chains)."""
    widths, paths, chains, R = None, [], [], None
    with open(os.path.join(GOLDEN, "ancestors_hand.txt")) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "requests":
                R = int(tok[1])
            elif tok[0] == "widths":
                widths = [int(x) for x in tok[1:]]
            elif tok[0] == "path":
                paths.append((int(tok[1]), int(tok[2]), [int(x) for x in tok[3:]]))
            elif tok[0] == "chain":
                chains.append((int(tok[1]), int(tok[2]), int(tok[3]), [int(x) for x in tok[4:]]))
    S, W_max = len(widths), max(widths)
    bp = np.full((R, S, W_max), -1, dtype=np.int32)
    for r, t, ent in paths:
        bp[r, t, :len(ent)] = ent
    inp = dict(num_requests=R, step_capacity=S, beam_capacity=W_max, beam_path=bp,
               widths=np.asarray(widths, dtype=np.int32))
    return inp, chains


# --------------------------------------------------------------------------
# A0: ancestor walk


def pin_ancestors_hand(orc):
    """Hand-enumerated chains (tests/golden/ancestors_hand.txt), integer equality."""
    inp, chains = load_hand_ancestors()
    for r, step, b, want in chains:
        got = orc.ancestors(inp, step, rows=[(r, b)])[0]
        assert list(got) == want, f"chain r={r} s={step} b={b}: got {list(got)} want {want}"


def pin_ancestors_structured(orc):
    """Closed forms: identity parents, all-zero parents, reversed parents."""
    R, S, W = 2, 4, 6
    widths = np.full(S, W, dtype=np.int32)
    base = dict(num_requests=R, step_capacity=S, beam_capacity=W, widths=widths)
    ident = np.broadcast_to(np.arange(W, dtype=np.int32), (R, S, W)).copy()
    ident[:, 0] = 0
    zero = np.zeros((R, S, W), dtype=np.int32)
    rev = np.broadcast_to((W - 1 - np.arange(W)).astype(np.int32), (R, S, W)).copy()
    rev[:, 0] = 0
    for step in range(S):
        a = orc.ancestors(dict(base, beam_path=ident), step)
        for b in range(W):
            assert list(a[0, b]) == [b] * (step + 1), "identity parents keep the slot"
        a = orc.ancestors(dict(base, beam_path=zero), step)
        for b in range(W):
            assert list(a[1, b]) == [0] * step + [b], "all-zero parents lead to slot 0"
        a = orc.ancestors(dict(base, beam_path=rev), step)
        for b in range(W):
            want = [b if (step - t) % 2 == 0 else W - 1 - b for t in range(step + 1)]
            assert list(a[1, b]) == want, "reversed parents alternate"


# --------------------------------------------------------------------------
# A1: context stage reduces to ordinary GQA decode attention at width 1


def pin_width1_is_gqa_decode(orc):
    """W=1 on every step: one chain, so this is plain GQA decode attention over
    ctx ++ [beam tokens of steps 0..s] -- compared with torch's SDPA in fp64."""
    for (Hq, Hkv, D, lc) in [(4, 2, 64, 37), (8, 2, 32, 5), (6, 6, 16, 0)]:
        inp = workloads.make_custom(2, Hq, Hkv, D, [lc, max(lc - 3, 0)], [1, 1, 1], seed=7 + Hq)
        G = Hq // Hkv
        scale = float(np.float32(inp["softmax_scale"]))
        for step in range(3):
            out, lse, _ = orc.decode_attn(inp, step)
            for r in range(2):
                n = int(inp["ctx_len"][r])
                k = np.concatenate([_f64(inp["ctx_k"][r, :, :n]),
                                    _f64(inp["beam_k"][r, :step + 1, 0]).transpose(1, 0, 2)], axis=1)
                v = np.concatenate([_f64(inp["ctx_v"][r, :, :n]),
                                    _f64(inp["beam_v"][r, :step + 1, 0]).transpose(1, 0, 2)], axis=1)
                qq = torch.from_numpy(_f64(inp["q"][step][r, 0]))[None, :, None, :]
                kk = torch.from_numpy(k).repeat_interleave(G, dim=0)[None]
                vv = torch.from_numpy(v).repeat_interleave(G, dim=0)[None]
                ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale)
                ref_lse = torch.logsumexp((qq @ kk.transpose(-1, -2)) * scale, dim=-1)
                np.testing.assert_allclose(out[r, 0], ref[0, :, 0].numpy(), rtol=0, atol=1e-12)
                np.testing.assert_allclose(lse[r, 0], ref_lse[0, :, 0].numpy(), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# A2/A4: split + log-sum-exp merge equals the unsplit softmax


def _merge(parts):
    lses = np.stack([p[1] for p in parts])          # [k, n, Hq]
    outs = np.stack([p[0] for p in parts])          # [k, n, Hq, D]
    top = np.max(lses, axis=0)
    top_safe = np.where(np.isfinite(top), top, 0.0)
    w = np.exp(lses - top_safe)
    total = w.sum(axis=0)
    lse = top_safe + np.log(total)
    out = (w[..., None] * outs).sum(axis=0) / total[..., None]
    return out, lse


def pin_split_merge_identity(orc):
    """Any split of the key set, merged by LSE, equals the unsplit softmax."""
    inp = workloads.make_custom(2, 4, 2, 32, [23, 9], [3, 5, 4], seed=99)
    rows = [(r, b) for r in range(2) for b in range(4)]
    for step in (1, 2):
        full_o, full_l, _ = orc.decode_attn(inp, step, rows=rows)
        for cut in (0, 1, 4, 9, 17, 23):
            a = orc.decode_attn(inp, step, rows=rows, ctx_range=(0, cut), include_beam=False)
            b = orc.decode_attn(inp, step, rows=rows, ctx_range=(cut, -1), include_beam=False)
            c = orc.decode_attn(inp, step, rows=rows, ctx_range=(0, 0), include_beam=True)
            o, l = _merge([a, b, c])
            np.testing.assert_allclose(o, full_o, rtol=0, atol=1e-12)
            np.testing.assert_allclose(l, full_l, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# A3 and the whole: brute force, empty context, tagged values


def pin_brute_force_tiny(orc):
    """The numpy brute force agrees with the C oracle to 1e-12 (tiny, every step)."""
    inp = tiny_inputs()
    for step in range(3):
        o, l, a = orc.decode_attn(inp, step)
        bo, bl, ba = brute.attention(inp, step)
        assert np.array_equal(a, ba), "ancestor tables differ"
        np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, bl, rtol=0, atol=1e-12)


def pin_empty_context(orc):
    """ctx_len = 0: only the beam chain is attended (brute force, ragged batch)."""
    inp = workloads.make_custom(3, 4, 2, 64, [0, 5, 0], [2, 3, 3], seed=5)
    for step in range(3):
        o, l, _ = orc.decode_attn(inp, step)
        bo, bl, _ = brute.attention(inp, step)
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
        np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, bl, rtol=0, atol=1e-12)


def pin_closed_form_two_keys(orc):
    """One context key, step 0, one head: softmax of two scores in closed form."""
    D = 16
    inp = workloads.make_custom(1, 1, 1, D, [1], [1], seed=3)
    one, two, half = 0x3F80, 0x4000, 0x3F00           # 1.0, 2.0, 0.5 in bf16
    q = np.zeros((1, 1, 1, D), np.uint16); q[..., 0] = two
    inp["q"] = [q]
    inp["ctx_k"][:] = 0; inp["ctx_k"][0, 0, 0, 0] = one            # key . q = 2
    inp["beam_k"][:] = 0; inp["beam_k"][0, 0, 0, 0, 0] = half      # key . q = 1
    inp["ctx_v"][:] = 0; inp["ctx_v"][0, 0, 0, 1] = one            # value e_1
    inp["beam_v"][:] = 0; inp["beam_v"][0, 0, 0, 0, 2] = one       # value e_2
    s = float(np.float32(1 / math.sqrt(D)))
    x_ctx, x_beam = 2 * s, 1 * s
    w_ctx = 1 / (1 + math.exp(x_beam - x_ctx))
    o, l, _ = orc.decode_attn(inp, 0)
    want = np.zeros(D); want[1] = w_ctx; want[2] = 1 - w_ctx
    np.testing.assert_allclose(o[0, 0, 0], want, rtol=0, atol=1e-14)
    assert abs(l[0, 0, 0] - (x_ctx + math.log(1 + math.exp(x_beam - x_ctx)))) < 1e-14


def pin_tagged_beam_values(orc):
    """Context V = 0 and each beam token's V = one-hot of its (step, slot) code:
    out[code] is the weight the row gives that token, so the non-zero codes
    name exactly the chain the hand walk gives, and their weights are the
    softmax weights of the chain tokens."""
    D = 64
    inp = workloads.make_custom(2, 4, 2, D, [6, 0], [3, 4, 2], seed=11, q_scale=4.0)
    hand, chains = load_hand_ancestors()
    inp["beam_path"][:] = hand["beam_path"]
    inp["widths"] = hand["widths"]
    inp["ctx_v"][:] = 0
    W_max = inp["beam_capacity"]
    for t in range(3):
        for a in range(W_max):
            inp["beam_v"][:, t, a] = 0
            inp["beam_v"][:, t, a, :, t * W_max + a] = 0x3F80
    scale = float(np.float32(inp["softmax_scale"]))
    for r, step, b, chain in chains:
        o, _, _ = orc.decode_attn(inp, step, rows=[(r, b)])
        for h in range(4):
            g = h // 2
            qv = _f64(inp["q"][step][r, b, h])
            n = int(inp["ctx_len"][r])
            keys = [_f64(inp["ctx_k"][r, g, j]) for j in range(n)]
            keys += [_f64(inp["beam_k"][r, t, chain[t], g]) for t in range(step + 1)]
            x = np.array([scale * float(np.dot(qv, k)) for k in keys])
            w = np.exp(x - x.max()); w /= w.sum()
            want = np.zeros(D)
            for t in range(step + 1):
                want[t * W_max + chain[t]] = w[n + t]
            np.testing.assert_allclose(o[0, h], want, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# invariants


def pin_identical_paths_identical_rows(orc):
    """All beams share one chain (every parent 0, current-step K/V equal in
    every slot) and the same query: every output row is the same."""
    inp = workloads.make_custom(2, 8, 2, 32, [17, 4], [5, 5, 5], seed=21)
    inp["beam_path"][:, 1:, :5] = 0
    for t in range(3):
        inp["beam_k"][:, t, :5] = inp["beam_k"][:, t, :1]
        inp["beam_v"][:, t, :5] = inp["beam_v"][:, t, :1]
        inp["q"][t][:] = inp["q"][t][:, :1]
    for step in range(3):
        o, l, _ = orc.decode_attn(inp, step)
        for b in range(1, 5):
            assert np.array_equal(o[:, b], o[:, 0]) and np.array_equal(l[:, b], l[:, 0])


def pin_relabel_invariance(orc):
    """Renumbering the slots of one step (moving K/V and fixing the parent
    indices that point at them) leaves every output row unchanged."""
    inp = workloads.make_custom(2, 4, 2, 32, [11, 7], [3, 5, 4], seed=31)
    o_ref, l_ref, _ = orc.decode_attn(inp, 2)
    rng = np.random.default_rng(5)
    for t in (0, 1):
        W_t = int(inp["widths"][t])
        perm = rng.permutation(W_t)                    # old slot i -> new slot perm[i]
        new = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in inp.items()}
        new["q"] = inp["q"]
        new["beam_k"][:, t, perm] = inp["beam_k"][:, t, :W_t]
        new["beam_v"][:, t, perm] = inp["beam_v"][:, t, :W_t]
        new["beam_path"][:, t, perm] = inp["beam_path"][:, t, :W_t]
        W_n = int(inp["widths"][t + 1])
        new["beam_path"][:, t + 1, :W_n] = perm[inp["beam_path"][:, t + 1, :W_n]]
        o, l, _ = orc.decode_attn(new, 2)
        np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l, l_ref, rtol=0, atol=1e-13)


def pin_convex_and_lse_bounds(orc):
    """Outputs are convex combinations of the attended values; the LSE lies
    between the largest score and the largest score + ln(#keys)."""
    inp = workloads.make_custom(2, 4, 2, 32, [40, 13], [4, 6, 5], seed=41, q_scale=2.0)
    scale = float(np.float32(inp["softmax_scale"]))
    for step in range(3):
        o, l, a = orc.decode_attn(inp, step)
        for r in range(2):
            n = int(inp["ctx_len"][r])
            for b in range(int(inp["widths"][step])):
                for h in range(4):
                    g = h // 2
                    k = np.concatenate([_f64(inp["ctx_k"][r, g, :n]),
                                        _f64(inp["beam_k"][r, np.arange(step + 1), a[r, b], g])])
                    v = np.concatenate([_f64(inp["ctx_v"][r, g, :n]),
                                        _f64(inp["beam_v"][r, np.arange(step + 1), a[r, b], g])])
                    x = scale * (k @ _f64(inp["q"][step][r, b, h]))
                    assert np.all(o[r, b, h] >= v.min(axis=0) - 1e-12)
                    assert np.all(o[r, b, h] <= v.max(axis=0) + 1e-12)
                    assert x.max() - 1e-12 <= l[r, b, h] <= x.max() + math.log(len(x)) + 1e-12


ALL_PINS = [
    pin_ancestors_hand,
    pin_ancestors_structured,
    pin_width1_is_gqa_decode,
    pin_split_merge_identity,
    pin_brute_force_tiny,
    pin_empty_context,
    pin_closed_form_two_keys,
    pin_tagged_beam_values,
    pin_identical_paths_identical_rows,
    pin_relabel_invariance,
    pin_convex_and_lse_bounds,
]
