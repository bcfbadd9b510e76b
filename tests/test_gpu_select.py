"""Parity of gr_beam_select (through the C ABI) with the selection oracle.

Integer outputs (parents, tokens) are compared exactly wherever the oracle's
order is decided by a clear margin or by exact ties (then the flat-index
rule fixes it); where two candidates' fp64 scores lie within the fp32
rounding of the kernel's scores, the selection is checked for validity
instead: every pick is a real candidate, the picked scores equal the
oracle's best scores within the tolerance, and every candidate clearly
inside the oracle's selection is picked.
"""

import numpy as np
import pytest

import workloads
from oracle import select

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():   # pragma: no cover - CPU-only machines
    pytest.skip("needs a GPU", allow_module_level=True)

import beam_decode_attention_gb300 as gr  # noqa: E402

TOL = 2e-4   # fp32 log-normaliser over up to ~1.5e5 exponentials, plus the score's rounding


def run_select(logits, scores, next_width, parent_stride=None):
    R, W, V = logits.shape
    shape = gr.SelectShape(R, W, V, next_width)
    ws = torch.empty(max(16, gr.gr_beam_select_workspace_size(shape)), dtype=torch.uint8, device="cuda")
    stride = next_width if parent_stride is None else parent_stride
    par = torch.full((R * stride,), -7, dtype=torch.int32, device="cuda")
    tok = torch.empty((R, next_width), dtype=torch.int32, device="cuda")
    sco = torch.empty((R, next_width), dtype=torch.float32, device="cuda")
    gr.gr_beam_select(shape, torch.from_numpy(logits).cuda(), torch.from_numpy(scores).cuda(),
                      par, tok, sco, ws, parent_stride=stride)
    torch.cuda.synchronize()
    par = par.cpu().numpy().reshape(R, stride)
    return par[:, :next_width], tok.cpu().numpy(), sco.cpu().numpy(), par


def check(logits, scores, next_width, par, tok, sco, requests=None):
    R, W, V = logits.shape
    for r in (range(R) if requests is None else requests):
        assert np.all((par[r] >= 0) & (par[r] < W)) and np.all((tok[r] >= 0) & (tok[r] < V))
        flat = par[r].astype(np.int64) * V + tok[r]
        assert len(np.unique(flat)) == next_width, "a candidate was picked twice"
        lp = select.log_softmax(logits[r, np.unique(par[r])])
        row_of = {b: i for i, b in enumerate(np.unique(par[r]))}
        exact = np.array([scores[r, b] + lp[row_of[b], v] for b, v in zip(par[r], tok[r])])
        fin = np.isfinite(exact)
        assert np.array_equal(fin, np.isfinite(sco[r]))
        assert np.all(np.abs(sco[r][fin] - exact[fin]) <= TOL * np.maximum(1.0, np.abs(exact[fin])))
        assert np.all(np.diff(sco[r].astype(np.float64)) <= 0), "scores not in descending order"
        ref_flat, ref_val = select.top_candidates(logits[r:r + 1], scores[r:r + 1], next_width, extra=1)
        ref_flat, ref_val = ref_flat[0], ref_val[0]
        top = ref_val[:next_width]
        got = np.sort(exact)[::-1]
        same = np.isfinite(top)
        assert np.all(np.abs(got[same] - top[same]) <= 2 * TOL * np.maximum(1.0, np.abs(top[same])))
        cut = top[-1]
        if np.isfinite(cut):
            clear = ref_flat[:next_width][top > cut + 2 * TOL * max(1.0, abs(cut))]
            assert np.all(np.isin(clear, flat)), "a clearly selected candidate is missing"
        gaps = np.diff(ref_val)
        if np.all(np.isfinite(ref_val)) and np.all(-gaps > 2 * TOL * np.maximum(1.0, np.abs(ref_val[1:]))):
            assert np.array_equal(flat, ref_flat[:next_width])


@pytest.mark.parametrize("R,W,V,n", [(2, 5, 37, 11), (3, 16, 1000, 64), (1, 8, 3, 20), (2, 40, 4099, 1024),
                                     (1, 1, 5000, 1), (2, 300, 2048, 300)])
def test_random_cases(R, W, V, n):
    inp = workloads.make_select_inputs(R, W, V, seed=R * 1000 + W * 10 + V + n)
    par, tok, sco, _ = run_select(inp["logits"], inp["beam_scores"], n)
    check(inp["logits"], inp["beam_scores"], n, par, tok, sco)


def test_exact_ties_follow_flat_index():
    """Every beam holds the same logits and score: all candidates of a token
    tie exactly, so the selection is the flat-index order of the best tokens."""
    rng = np.random.default_rng(3)
    row = rng.standard_normal(300).astype(np.float32)
    logits = np.broadcast_to(row, (2, 6, 300)).copy()
    scores = np.full((2, 6), -1.5, np.float32)
    par, tok, sco, _ = run_select(logits, scores, 20)
    order = np.argsort(-row, kind="stable")
    want = [(b, v) for v in order for b in range(6)][:20]   # best token on every beam, then the next
    for r in range(2):
        assert [(int(p), int(t)) for p, t in zip(par[r], tok[r])] == want


def test_constant_rows_take_the_exact_fallback():
    """Constant logits (a whole row ties at the boundary, more than the
    shared-memory candidate slots): the exact radix path picks the first
    tokens by index."""
    logits = np.zeros((2, 3, 20000), np.float32)
    logits[1, 1] = 1.0                      # request 1: beam 1 is ahead of the others only by S
    scores = np.array([[-1.0, -1.0, -1.0], [-2.0, -0.5, -2.0]], np.float32)
    par, tok, sco, _ = run_select(logits, scores, 700)
    assert np.array_equal(par[0], np.zeros(700)) and np.array_equal(tok[0], np.arange(700))
    assert np.array_equal(par[1], np.ones(700)) and np.array_equal(tok[1], np.arange(700))
    assert np.allclose(sco[0], -1.0 - np.log(20000.0), atol=1e-5)


@pytest.mark.parametrize("skew", ["prefix_high", "prefix_low", "tail_high", "mixed_scales", "prefix_masked"])
def test_threshold_prefix_skews(skew):
    """The row kernel sets its candidate threshold from each row's first
    logits: rows whose prefix is not representative (its best far above or
    below the rest, or rows of different scales) must still select exactly,
    through the completeness check or the exact fallback."""
    R, W, V, n = 2, 24, 20000, 64
    inp = workloads.make_select_inputs(R, W, V, seed={"prefix_high": 1, "prefix_low": 2, "tail_high": 3,
                                                      "mixed_scales": 4, "prefix_masked": 5}[skew])
    z = inp["logits"]
    if skew == "prefix_high":
        z[:, :, :4096] += np.float32(3.0)
    elif skew == "prefix_low":
        z[:, :, :4096] -= np.float32(10.0)
    elif skew == "tail_high":
        z[:, :, 15000:] += np.float32(6.0)
    elif skew == "prefix_masked":
        z[:, :, :4096] = -np.inf
    else:
        z[:, ::2, :] *= np.float32(0.05)
    par, tok, sco, _ = run_select(z, inp["beam_scores"], n)
    check(z, inp["beam_scores"], n, par, tok, sco)


def test_guessed_threshold_after_an_unlike_row():
    """More rows than the row kernel has CTAs (four per SM), so each CTA
    streams rows one after another: flat rows first, then rows whose first
    4096 logits are raised by 6.  Once the request has a bound, a row's
    threshold is guessed from it with the normaliser correction (c - c_pre)
    the CTA saw on its previous row; for a raised row after a flat one that
    guess is too high, so the completeness check must send the row to a
    complete k-th selection or the exact path.  The selection stays exact."""
    grid = torch.cuda.get_device_properties(0).multi_processor_count * 4
    R, V, n = 1, 20000, 256
    W = 3 * grid
    inp = workloads.make_select_inputs(R, W, V, seed=77)
    z = inp["logits"]
    z[:, 2 * grid:, :4096] += np.float32(6.0)
    par, tok, sco, _ = run_select(z, inp["beam_scores"], n)
    check(z, inp["beam_scores"], n, par, tok, sco)


def test_masked_tokens_and_width_past_the_finite_candidates():
    """-inf logits mask tokens; asking for more beams than there are finite
    candidates returns the finite ones by score, then masked ones by index."""
    rng = np.random.default_rng(9)
    logits = np.full((1, 3, 8), -np.inf, np.float32)
    logits[0, :, [1, 6]] = rng.standard_normal((2, 3)).astype(np.float32)
    scores = np.array([[-0.5, -1.0, -0.25]], np.float32)
    par, tok, sco, _ = run_select(logits, scores, 10)
    ref_p, ref_t, ref_s = select.beam_select(logits, scores, 10)
    assert np.array_equal(par, ref_p) and np.array_equal(tok, ref_t)
    assert np.all(np.isneginf(sco[0, 6:])) and np.allclose(sco[0, :6], ref_s[0, :6], atol=TOL)


def test_parent_rows_written_in_place():
    """next_parent rows at a stride (the next BeamPath row inside a
    [R, S_max, W_max] array): the gaps between rows stay untouched."""
    inp = workloads.make_select_inputs(3, 10, 500, seed=21)
    par, tok, sco, raw = run_select(inp["logits"], inp["beam_scores"], 7, parent_stride=24)
    assert np.all(raw[:, 7:] == -7)
    check(inp["logits"], inp["beam_scores"], 7, par, tok, sco)


def test_headline_size_sampled_requests():
    """R=4, W=900 -> 900, V=151,936 (the measured configuration): requests 0
    and 3 against the oracle."""
    cfg = workloads.SELECT_HEADLINE
    inp = workloads.make_select_inputs(cfg["num_requests"], cfg["width"], cfg["vocab"], seed=4242)
    par, tok, sco, _ = run_select(inp["logits"], inp["beam_scores"], cfg["next_width"])
    check(inp["logits"], inp["beam_scores"], cfg["next_width"], par, tok, sco, requests=[0, 3])
