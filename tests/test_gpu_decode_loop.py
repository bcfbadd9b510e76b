"""Three decode steps run on the device through the C ABI, with no host
round trip between them: gr_beam_append writes each step's new K/V,
gr_decode_attn attends, and gr_beam_select writes the next BeamPath row in
place (next_parent pointing into BeamPath) and the next beam scores.  The
oracle runs the same loop on the CPU (tests/decode_loop.py).

Each step's attention meets the oracle's gate; parents, tokens and the
BeamPath rows are bit-exact (the seeded inputs decide every selection by a
margin far above the scores' fp32 rounding, a property the CPU suite checks
on the oracle alone); scores agree within the selection tolerance.

The xGR variant reorders the per-beam cache in place after each selection
(gr_beam_reorder_inplace) and attends through the identity path: its rows
equal the BeamPath loop's bit for bit.
"""

import numpy as np
import pytest

import decode_loop

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():   # pragma: no cover - CPU-only machines
    pytest.skip("needs a GPU", allow_module_level=True)

import beam_decode_attention_gb300 as gr  # noqa: E402
from gpu_util import compare, to_dev  # noqa: E402

SCORE_TOL = 1e-4   # fp32 log-normaliser over <= 128 logits plus the score's rounding


def device_loop(inp, inplace):
    """Runs the loop on one stream; returns the per-step device tensors."""
    shape = gr.Shape.of(inp)
    R, Hq, D = inp["num_requests"], inp["num_q_heads"], inp["head_dim"]
    S, W_max, V = inp["step_capacity"], inp["beam_capacity"], inp["vocab"]
    W = [int(w) for w in inp["widths"]]
    ck, cv, cl = to_dev(inp["ctx_k"]), to_dev(inp["ctx_v"]), to_dev(inp["ctx_len"])
    bk, bv, bp = to_dev(inp["beam_k"]), to_dev(inp["beam_v"]), to_dev(inp["beam_path"])
    k_new = [to_dev(x) for x in inp["k_new"]]
    v_new = [to_dev(x) for x in inp["v_new"]]
    q = [to_dev(x) for x in inp["q"]]
    logits = [to_dev(x) for x in inp["logits"]]
    scores = to_dev(inp["beam_scores"])
    steps = []
    for s in range(S):
        # widths as the attention call sees them: the schedule itself, or,
        # once the cache has been reordered in place, W_s at every level
        widths = [W[s]] * (s + 1) if inplace else W[:s + 1]
        gr.gr_beam_append(shape, widths, s, k_new[s], v_new[s], bk, bv)
        out = torch.empty(R * W[s] * Hq * D, dtype=torch.int16, device="cuda")
        lse = torch.empty(R * W[s] * Hq, dtype=torch.float32, device="cuda")
        ws = torch.empty(max(16, gr.gr_decode_attn_workspace_size(shape, widths, s)), dtype=torch.uint8,
                         device="cuda")
        gr.gr_decode_attn(shape, q[s], ck, cv, cl, bk, bv, bp, widths, s, out, lse, ws)
        rec = dict(out=out, lse=lse)
        if s + 1 < S:
            sel = gr.SelectShape(R, W[s], V, W[s + 1])
            sws = torch.empty(max(16, gr.gr_beam_select_workspace_size(sel)), dtype=torch.uint8, device="cuda")
            tok = torch.empty((R, W[s + 1]), dtype=torch.int32, device="cuda")
            sco = torch.empty((R, W[s + 1]), dtype=torch.float32, device="cuda")
            gr.gr_beam_select(sel, logits[s], scores, bp[0, s + 1], tok, sco, sws, parent_stride=S * W_max)
            rec.update(token=tok, score=sco, path=bp[:, s + 1, :W[s + 1]].clone())
            if inplace:
                gr.gr_beam_reorder_inplace(shape, bk, bv, bp, [W[s]] * (s + 1) + [W[s + 1]], s + 1)
            scores = sco
        steps.append(rec)
    torch.cuda.synchronize()
    assert gr.gr_get_device_error() == 0
    return steps


def f32_of(out):
    return (out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("name", sorted(decode_loop.CASES))
def test_three_step_loop_meets_the_oracle(name):
    inp = decode_loop.make_case(name)
    ref, margin, _ = decode_loop.run_oracle_loop(inp)
    assert margin >= decode_loop.MARGIN
    got = device_loop(inp, inplace=False)
    for s, (g, r) in enumerate(zip(got, ref)):
        compare(f32_of(g["out"]).reshape(r["out"].shape), g["lse"].cpu().numpy().reshape(r["lse"].shape),
                r["out"], r["lse"])
        if "parent" in r:
            assert np.array_equal(g["path"].cpu().numpy(), r["parent"]), f"BeamPath row {s + 1}"
            assert np.array_equal(g["token"].cpu().numpy(), r["token"]), f"tokens after step {s}"
            sc = g["score"].cpu().numpy().astype(np.float64)
            assert np.all(np.abs(sc - r["score"]) <= SCORE_TOL * np.maximum(1.0, np.abs(r["score"])))


@pytest.mark.parametrize("name", sorted(decode_loop.CASES))
def test_loop_on_the_cache_reordered_in_place_gives_the_same_rows(name):
    inp = decode_loop.make_case(name)
    a = device_loop(inp, inplace=False)
    b = device_loop(inp, inplace=True)
    for s, (x, y) in enumerate(zip(a, b)):
        assert torch.equal(x["out"], y["out"]), f"step {s} out"
        assert torch.equal(x["lse"], y["lse"]), f"step {s} lse"
        if "token" in x:
            assert torch.equal(x["token"], y["token"]) and torch.equal(x["score"], y["score"])
            assert torch.equal(x["path"], y["path"])
