"""Pins for the item-constrained selection oracle (oracle.select.trie_select):
a hand-worked trie, the reduction to unconstrained selection when a node's
edges cover the vocabulary, a brute force and invariances."""

import math
import os

import numpy as np
import pytest

from oracle import select

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_VALUES = {"ln3": math.log(3.0), "ln(3/4)": math.log(0.75), "ln(1/4)": math.log(0.25), "-inf": -math.inf}


def _num(tok):
    return _VALUES[tok] if tok in _VALUES else float(tok)


def hand_case():
    d = {"z": {}, "want": []}
    with open(os.path.join(GOLDEN, "trie_select_hand.txt")) as fh:
        for line in fh:
            f = line.split()
            if not f or f[0].startswith("#"):
                continue
            if f[0] in ("offsets", "tokens", "children", "beam_node"):
                d[f[0]] = np.array([int(x) for x in f[1:]], np.int32)
            elif f[0] == "S":
                d["S"] = np.array([[_num(x) for x in f[1:]]])
            elif f[0] == "z":
                d["z"][int(f[1])] = [_num(x) for x in f[2:]]
            elif f[0] == "next_width":
                d["n"] = int(f[1])
            elif f[0] == "want":
                d["want"].append((int(f[1]), int(f[2]), int(f[3]), _num(f[4])))
    W = len(d["beam_node"])
    d["logits"] = np.array([[d["z"][b] for b in range(W)]])
    d["beam_node"] = d["beam_node"][None, :]
    return d


def test_hand_worked_trie():
    d = hand_case()
    parent, token, node, score = select.trie_select(d["logits"], d["S"], d["beam_node"], d["offsets"],
                                                    d["tokens"], d["children"], d["n"])
    want = d["want"]
    assert [int(x) for x in parent[0]] == [w[0] for w in want]
    assert [int(x) for x in token[0]] == [w[1] for w in want]
    assert [int(x) for x in node[0]] == [w[2] for w in want]
    fin = [np.isfinite(w[3]) for w in want]
    assert np.allclose(score[0][fin], [w[3] for w in want if np.isfinite(w[3])], rtol=0, atol=1e-14)
    assert np.all(np.isneginf(score[0][[not f for f in fin]]))


def random_trie(rng, V, fanout, depth):
    """A CSR trie of `depth` levels below the root, each node with a random
    sorted subset of at most `fanout` of the V tokens."""
    offsets, tokens, children = [0], [], []
    level, next_id = [0], 1
    frontier = []
    nodes = {0: None}
    for _ in range(depth):
        frontier = []
        for n in level:
            k = int(rng.integers(1, fanout + 1))
            toks = np.sort(rng.choice(V, size=k, replace=False))
            nodes[n] = [(int(t), next_id + i) for i, t in enumerate(toks)]
            frontier += [next_id + i for i in range(k)]
            next_id += k
        level = frontier
    N = next_id
    for n in range(N):
        for t, c in (nodes.get(n) or []):
            tokens.append(t)
            children.append(c)
        offsets.append(len(tokens))
    return (np.array(offsets, np.int32), np.array(tokens, np.int32), np.array(children, np.int32), N)


def _brute(z, S, bn, offsets, tokens, children, n):
    sp = pytest.importorskip("scipy.special")
    R, W, V = z.shape
    out = []
    for r in range(R):
        cand = []
        for b in range(W):
            ks = list(range(offsets[bn[r, b]], offsets[bn[r, b] + 1]))
            if not ks:
                continue
            lp = sp.log_softmax(np.array([z[r, b, tokens[k]] for k in ks], np.float64))
            cand += [(-(S[r, b] + lp[i]), b * V + int(tokens[k]), int(children[k])) for i, k in enumerate(ks)]
        cand.sort()
        out.append([(f // V, f % V, c, -s) for s, f, c in cand[:n]])
    return out


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_against_brute_force(seed):
    rng = np.random.default_rng(seed)
    V = 40
    offsets, tokens, children, N = random_trie(rng, V, 6, 3)
    R, W = 2, 7
    z = rng.standard_normal((R, W, V)) * 2.0
    S = -np.abs(rng.standard_normal((R, W))) * 3.0
    bn = rng.integers(0, N, size=(R, W)).astype(np.int32)
    n = 9
    parent, token, node, score = select.trie_select(z, S, bn, offsets, tokens, children, n)
    for r, ref in enumerate(_brute(z, S, bn, offsets, tokens, children, n)):
        k = len(ref)
        assert [int(x) for x in parent[r, :k]] == [p for p, _, _, _ in ref]
        assert [int(x) for x in token[r, :k]] == [t for _, t, _, _ in ref]
        assert [int(x) for x in node[r, :k]] == [c for _, _, c, _ in ref]
        assert np.allclose(score[r, :k], [s for _, _, _, s in ref], rtol=0, atol=1e-12)
        assert np.all(parent[r, k:] == -1) and np.all(np.isneginf(score[r, k:]))


def test_full_fanout_reduces_to_unconstrained_selection():
    """A node whose edges are every token of the vocabulary, and every beam on
    it: the constrained selection is the plain one (next nodes = the edges'
    children)."""
    rng = np.random.default_rng(8)
    V = 30
    offsets = np.array([0, V] + [V] * V, np.int32)
    tokens = np.arange(V, dtype=np.int32)
    children = np.arange(1, V + 1, dtype=np.int32)
    z = rng.standard_normal((2, 5, V))
    S = -np.abs(rng.standard_normal((2, 5)))
    bn = np.zeros((2, 5), np.int32)
    p0, t0, s0 = select.beam_select(z, S, 12)
    p1, t1, n1, s1 = select.trie_select(z, S, bn, offsets, tokens, children, 12)
    assert np.array_equal(p0, p1) and np.array_equal(t0, t1) and np.allclose(s0, s1, atol=1e-12)
    assert np.array_equal(n1, t1 + 1)


def test_masked_logits_do_not_matter():
    rng = np.random.default_rng(4)
    offsets, tokens, children, N = random_trie(rng, 25, 5, 2)
    z = rng.standard_normal((1, 6, 25))
    S = -np.abs(rng.standard_normal((1, 6)))
    bn = rng.integers(0, N, size=(1, 6)).astype(np.int32)
    legal = np.zeros((1, 6, 25), bool)
    for b in range(6):
        legal[0, b, tokens[offsets[bn[0, b]]:offsets[bn[0, b] + 1]]] = True
    a = select.trie_select(z, S, bn, offsets, tokens, children, 8)
    z2 = np.where(legal, z + 3.0, rng.standard_normal(z.shape) * 50)   # shift legal, scramble the rest
    b_ = select.trie_select(z2, S, bn, offsets, tokens, children, 8)
    for x, y in zip(a[:3], b_[:3]):
        assert np.array_equal(x, y)
    assert np.allclose(a[3], b_[3], atol=1e-12)
