"""Pins for the beam-selection oracle (oracle/select.py): hand-worked cases,
SciPy's log_softmax, a separately written brute force, and invariances."""

import math
import os

import numpy as np
import pytest

from oracle import select

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_VALUES = {"ln3": math.log(3.0), "-ln4": -math.log(4.0), "ln(3/4)": math.log(0.75),
           "ln(1/4)": math.log(0.25)}


def _num(tok):
    return _VALUES[tok] if tok in _VALUES else float(tok)


def hand_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "beam_select_hand.txt")) as fh:
        for line in fh:
            f = line.split()
            if not f or f[0].startswith("#"):
                continue
            if f[0] == "case":
                W, V, n = int(f[2]), int(f[3]), int(f[4])
                cur = dict(name=f[1], z=np.zeros((1, W, V)), S=np.zeros((1, W)), n=n, want=[])
                cases.append(cur)
            elif f[0] == "S":
                cur["S"][0] = [_num(x) for x in f[1:]]
            elif f[0] == "z":
                cur["z"][0, int(f[1])] = [_num(x) for x in f[2:]]
            elif f[0] == "want":
                cur["want"].append((int(f[1]), int(f[2]), _num(f[3])))
    return cases


@pytest.mark.parametrize("case", hand_cases(), ids=lambda c: c["name"])
def test_hand_worked_cases(case):
    parent, token, score = select.beam_select(case["z"], case["S"], case["n"])
    want = case["want"]
    assert [int(x) for x in parent[0]] == [w[0] for w in want]
    assert [int(x) for x in token[0]] == [w[1] for w in want]
    assert np.allclose(score[0], [w[2] for w in want], rtol=0, atol=1e-14)


def test_log_softmax_matches_scipy():
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    z = rng.standard_normal((3, 5, 1000)) * 4.0 + rng.standard_normal((3, 5, 1)) * 200.0
    assert np.max(np.abs(select.log_softmax(z) - sp.log_softmax(z, axis=-1))) < 1e-11


def _brute(z, S, n):
    """Every candidate, ordered by Python's sort on (-score, flat index)."""
    sp = pytest.importorskip("scipy.special")
    lp = sp.log_softmax(np.asarray(z, np.float64), axis=-1)
    R, W, V = lp.shape
    out = []
    for r in range(R):
        cand = sorted(((-(S[r, b] + lp[r, b, v]), b * V + v) for b in range(W) for v in range(V)))
        out.append([(f // V, f % V, -s) for s, f in cand[:n]])
    return out


@pytest.mark.parametrize("R,W,V,n", [(1, 1, 7, 3), (2, 4, 9, 5), (3, 6, 5, 30), (2, 3, 4, 12)])
def test_against_brute_force(R, W, V, n):
    rng = np.random.default_rng(R * 100 + W * 10 + V)
    z = rng.standard_normal((R, W, V)) * 2.0
    S = -np.abs(rng.standard_normal((R, W))) * 3.0
    parent, token, score = select.beam_select(z, S, n)
    for r, ref in enumerate(_brute(z, S, n)):
        assert [int(x) for x in parent[r]] == [p for p, _, _ in ref]
        assert [int(x) for x in token[r]] == [t for _, t, _ in ref]
        assert np.allclose(score[r], [s for _, _, s in ref], rtol=0, atol=1e-12)


def test_masked_tokens_rank_last_by_index():
    z = np.array([[[0.0, -np.inf, 1.0], [-np.inf, 2.0, -np.inf]]])
    S = np.zeros((1, 2))
    parent, token, score = select.beam_select(z, S, 6)
    # finite candidates by score, then the three masked ones by flat index 1, 3, 5
    assert [(int(p), int(t)) for p, t in zip(parent[0], token[0])][3:] == [(0, 1), (1, 0), (1, 2)]
    assert np.all(np.isneginf(score[0, 3:])) and np.all(np.isfinite(score[0, :3]))
    assert (int(parent[0, 0]), int(token[0, 0])) == (1, 1)   # a lone finite logit: log-prob 0


def test_invariances():
    rng = np.random.default_rng(11)
    z = rng.standard_normal((2, 5, 40))
    S = -np.abs(rng.standard_normal((2, 5)))
    p0, t0, s0 = select.beam_select(z, S, 17)
    # a constant added to a beam's logits leaves its log-probabilities unchanged
    p1, t1, s1 = select.beam_select(z + rng.standard_normal((2, 5, 1)) * 30.0, S, 17)
    assert np.array_equal(p0, p1) and np.array_equal(t0, t1) and np.allclose(s0, s1, atol=1e-10)
    # reversing the beams maps each parent b to W-1-b (no ties in this draw)
    p2, t2, s2 = select.beam_select(z[:, ::-1], S[:, ::-1], 17)
    assert np.array_equal(p2, 4 - p0) and np.array_equal(t2, t0) and np.allclose(s2, s0, atol=1e-12)
    # each beam's probabilities sum to one
    assert np.allclose(np.exp(select.log_softmax(z)).sum(-1), 1.0, atol=1e-12)


def test_top_candidates_agrees_with_exact_selection():
    rng = np.random.default_rng(5)
    z = rng.standard_normal((2, 30, 300)).astype(np.float32)
    S = (-np.abs(rng.standard_normal((2, 30))) * 2).astype(np.float32)
    parent, token, score = select.beam_select(z, S, 50)
    flat, vals = select.top_candidates(z, S, 50, extra=10)
    assert np.array_equal(flat[:, :50] // 300, parent) and np.array_equal(flat[:, :50] % 300, token)
    assert np.allclose(vals[:, :50], score, atol=1e-12)
    assert np.all(np.diff(vals, axis=1) <= 0)
