"""Parity of gr_trie_select (item-constrained beam selection, through the C
ABI) with its oracle: a hand-worked trie, random SID tries at every level
(leaves, padding), a node with more edges than one chunk, out-of-range trie
indices, and the measured size on two requests."""

import numpy as np
import pytest

import workloads
from oracle import select
import test_oracle_trie_select as hand

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():   # pragma: no cover - CPU-only machines
    pytest.skip("needs a GPU", allow_module_level=True)

import beam_decode_attention_gb300 as gr  # noqa: E402

TOL = 1e-4


def dev(a, dtype=None):
    return torch.from_numpy(np.ascontiguousarray(a if dtype is None else a.astype(dtype))).cuda()


def run(logits, scores, beam_node, offsets, tokens, children, n, num_nodes=None):
    R, W, V = logits.shape
    N = len(offsets) - 1 if num_nodes is None else num_nodes
    shape = gr.TrieSelectShape(R, W, V, n, N, len(tokens))
    ws = torch.empty(max(16, gr.gr_trie_select_workspace_size(shape)), dtype=torch.uint8, device="cuda")
    par = torch.empty((R, n), dtype=torch.int32, device="cuda")
    tok = torch.empty_like(par)
    nod = torch.empty_like(par)
    sco = torch.empty((R, n), dtype=torch.float32, device="cuda")
    tk = dev(tokens, np.int32) if len(tokens) else torch.zeros(4, dtype=torch.int32, device="cuda")
    ch = dev(children, np.int32) if len(children) else torch.zeros(4, dtype=torch.int32, device="cuda")
    gr.gr_trie_select(shape, dev(logits, np.float32), dev(scores, np.float32), dev(beam_node, np.int32),
                      dev(offsets, np.int32), tk, ch, par, tok, sco, nod, ws)
    torch.cuda.synchronize()
    return par.cpu().numpy(), tok.cpu().numpy(), nod.cpu().numpy(), sco.cpu().numpy()


def check(logits, scores, beam_node, offsets, tokens, children, n, got, requests=None):
    par, tok, nod, sco = got
    rp, rt, rn, rs = select.trie_select(logits, scores, beam_node, offsets, tokens, children, n)
    R, W, V = logits.shape
    for r in (range(R) if requests is None else requests):
        real = rp[r] >= 0
        k = int(real.sum())
        # padding where the oracle has no candidate
        assert np.all(par[r, k:] == -1) and np.all(tok[r, k:] == -1) and np.all(nod[r, k:] == -1)
        assert np.all(np.isneginf(sco[r, k:]))
        assert np.allclose(sco[r, :k], rs[r, :k], rtol=0, atol=TOL * max(1.0, np.abs(rs[r, :k]).max(initial=0)))
        gaps = -np.diff(rs[r, :k])
        if k <= 1 or np.all(gaps > 2 * TOL * max(1.0, np.abs(rs[r, :k]).max())):
            assert np.array_equal(par[r, :k], rp[r, :k]) and np.array_equal(tok[r, :k], rt[r, :k])
            assert np.array_equal(nod[r, :k], rn[r, :k])
        else:
            # near-ties: same multiset of candidates up to the tolerance, each pick a real edge
            got_flat = set(zip(par[r, :k].tolist(), tok[r, :k].tolist()))
            clear = [(p, t) for p, t, s in zip(rp[r, :k], rt[r, :k], rs[r, :k]) if s > rs[r, k - 1] + 2 * TOL]
            assert set(clear) <= got_flat
            for p, t, c in zip(par[r, :k], tok[r, :k], nod[r, :k]):
                nd = beam_node[r, p]
                e = np.arange(offsets[nd], offsets[nd + 1])
                assert t in tokens[e] and c == children[e[np.searchsorted(tokens[e], t)]]


def test_hand_worked_trie():
    d = hand.hand_case()
    got = run(d["logits"].astype(np.float32), d["S"].astype(np.float32), d["beam_node"], d["offsets"],
              d["tokens"], d["children"], d["n"])
    want = d["want"]
    assert [int(x) for x in got[0][0]] == [w[0] for w in want]
    assert [int(x) for x in got[1][0]] == [w[1] for w in want]
    assert [int(x) for x in got[2][0]] == [w[2] for w in want]
    assert np.allclose(got[3][0][:3], [w[3] for w in want[:3]], atol=1e-6) and np.isneginf(got[3][0][3])


@pytest.mark.parametrize("level,W,n", [(0, 5, 7), (1, 16, 40), (2, 30, 64), (3, 4, 5), (1, 3, 200)])
def test_random_sid_tries(level, W, n):
    t = workloads.make_sid_trie(3000, 3, 24, 500, seed=level * 10 + W)
    inp = workloads.make_trie_select_inputs(2, W, 500, t, level, seed=level + W + n)
    got = run(inp["logits"], inp["beam_scores"], inp["beam_node"], t["offsets"], t["tokens"], t["children"], n)
    check(inp["logits"], inp["beam_scores"], inp["beam_node"], t["offsets"], t["tokens"], t["children"], n, got)


def test_node_with_more_edges_than_a_chunk():
    t = workloads.make_sid_trie(8000, 1, 3000, 4000, seed=77)   # the root has ~2800 edges
    assert t["offsets"][1] > 2048
    inp = workloads.make_trie_select_inputs(2, 6, 4000, t, 0, seed=78)
    got = run(inp["logits"], inp["beam_scores"], inp["beam_node"], t["offsets"], t["tokens"], t["children"], 1000)
    check(inp["logits"], inp["beam_scores"], inp["beam_node"], t["offsets"], t["tokens"], t["children"], 1000, got)


def test_entries_keep_the_token_when_edge_indices_overflow():
    """The list entries carry the edge index while W * num_edges fits 32 bits,
    and the token otherwise (the merge then finds the child by a search of the
    parent's node).  4096 beams over 513 nodes of 2048 edges each (1,050,624
    edges) take the second form, through the wide-row kernel."""
    W, V, N, n = 4096, 2048, 513, 64
    assert W * N * V >= 1 << 32
    rng = np.random.default_rng(513)
    offsets = (np.arange(N + 1) * V).astype(np.int32)
    tokens = np.tile(np.arange(V, dtype=np.int32), N)
    children = rng.integers(0, N, size=N * V).astype(np.int32)
    logits = rng.standard_normal(size=(1, W, V), dtype=np.float32) * np.float32(2.0)
    scores = (-np.abs(rng.standard_normal(size=(1, W), dtype=np.float32)) * np.float32(3.0))
    beam_node = rng.integers(0, N, size=(1, W)).astype(np.int32)
    got = run(logits, scores, beam_node, offsets, tokens, children, n)
    check(logits, scores, beam_node, offsets, tokens, children, n, got)


def test_rows_wide_and_narrow_in_one_request():
    """Beams at a node with more edges than one warp holds (the block kernel)
    and beams at small nodes (the warp kernel) in the same requests: both
    feed one merge."""
    t = workloads.make_sid_trie(4000, 2, 600, 2000, seed=91)   # the root has ~600 edges
    assert t["offsets"][1] > 256
    inp = workloads.make_trie_select_inputs(2, 10, 2000, t, 1, seed=92)
    bn = inp["beam_node"].copy()
    bn[:, ::3] = 0   # every third beam at the root
    got = run(inp["logits"], inp["beam_scores"], bn, t["offsets"], t["tokens"], t["children"], 40)
    check(inp["logits"], inp["beam_scores"], bn, t["offsets"], t["tokens"], t["children"], 40, got)


def test_rows_with_fewer_and_more_candidates_than_the_width():
    """Beams at a node of 16 edges keep every candidate (fewer than W' = 20:
    only the merge's head keys are put in order), beams at a node of 30 edges
    keep their best 20 in full order and publish their 20th as a bound; both
    kinds of list feed one merge."""
    V, W, n = 64, 40, 20
    # node 0: the root (edges to nodes 1 and 2); node 1: 16 edges; node 2: 30 edges; nodes 3..48: leaves
    deg = [2, 16, 30]
    offsets = np.concatenate([[0], np.cumsum(deg), np.full(46, sum(deg))]).astype(np.int32)
    tokens = np.concatenate([[0, 1], np.arange(10, 26), np.arange(30, 60)]).astype(np.int32)
    children = np.concatenate([[1, 2], np.arange(3, 19), np.arange(19, 49)]).astype(np.int32)
    rng = np.random.default_rng(2020)
    logits = (rng.standard_normal(size=(2, W, V)) * 2.0).astype(np.float32)
    scores = (-np.abs(rng.standard_normal(size=(2, W))) * 3.0).astype(np.float32)
    beam_node = np.where(np.arange(W) % 2 == 0, 1, 2)[None, :].repeat(2, axis=0).astype(np.int32)
    got = run(logits, scores, beam_node, offsets, tokens, children, n)
    check(logits, scores, beam_node, offsets, tokens, children, n, got)


def test_exact_ties_overflow_the_merge_buffer():
    """Every candidate ties exactly (equal legal logits, equal beam scores):
    a row list orders only its head entries, every list's head reaches the
    merge's bound, and the candidates at or above it (12,800) overflow the
    merge's shared memory.  The rows' unordered tails are then sorted in
    place and the lists walked where they are; the selection is the
    flat-index order."""
    W, V, deg, n = 64, 300, 200, 64
    offsets = np.array([0] + [deg] * (deg + 1), dtype=np.int32)   # the root's deg edges, then deg leaves
    tokens = np.arange(deg, dtype=np.int32)
    children = np.arange(1, deg + 1, dtype=np.int32)
    logits = np.zeros((1, W, V), np.float32)
    scores = np.full((1, W), -1.0, np.float32)
    beam_node = np.zeros((1, W), np.int32)
    par, tok, nod, sco = run(logits, scores, beam_node, offsets, tokens, children, n)
    assert np.array_equal(par[0], np.zeros(n)) and np.array_equal(tok[0], np.arange(n))
    assert np.array_equal(nod[0], np.arange(1, n + 1))
    assert np.allclose(sco[0], -1.0 - np.log(deg), atol=1e-5)


def test_out_of_range_nodes_are_skipped():
    """Beams whose node index lies outside the trie contribute nothing (the
    kernel checks the index before reading the trie)."""
    t = workloads.make_sid_trie(500, 2, 10, 100, seed=5)
    inp = workloads.make_trie_select_inputs(1, 6, 100, t, 1, seed=6)
    bn = inp["beam_node"].copy()
    bn[0, 1] = -5
    bn[0, 4] = t["num_nodes"] + 3
    got = run(inp["logits"], inp["beam_scores"], bn, t["offsets"], t["tokens"], t["children"], 12)
    keep = bn.copy()
    leaf = t["level_nodes"][-1][0]          # a leaf stands in for the skipped beams in the oracle
    keep[0, 1] = keep[0, 4] = leaf
    check(inp["logits"], inp["beam_scores"], keep, t["offsets"], t["tokens"], t["children"], 12, got)


def test_headline_size_sampled_requests():
    cfg = workloads.SELECT_TRIE_HEADLINE
    t = workloads.make_sid_trie(cfg["items"], cfg["levels"], cfg["codebook"], cfg["vocab"], seed=31)
    inp = workloads.make_trie_select_inputs(cfg["num_requests"], cfg["width"], cfg["vocab"], t, cfg["level"], seed=32)
    got = run(inp["logits"], inp["beam_scores"], inp["beam_node"], t["offsets"], t["tokens"], t["children"],
              cfg["next_width"])
    check(inp["logits"], inp["beam_scores"], inp["beam_node"], t["offsets"], t["tokens"], t["children"],
          cfg["next_width"], got, requests=[0, 3])
