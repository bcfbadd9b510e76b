"""The oracle's decode loop on its own (CPU): the seeded loop inputs fix
every selection by a clear margin, and the BeamPath rows the loop writes are
valid parents whose chains the oracle's ancestor walk follows."""

import numpy as np
import pytest

import decode_loop
import oracle


@pytest.mark.parametrize("name", sorted(decode_loop.CASES))
def test_loop_selections_are_decided_by_a_clear_margin(name):
    inp = decode_loop.make_case(name)
    records, margin, st = decode_loop.run_oracle_loop(inp)
    assert margin >= decode_loop.MARGIN
    W = [int(w) for w in inp["widths"]]
    for s, rec in enumerate(records):
        assert rec["out"].shape == (inp["num_requests"], W[s], inp["num_q_heads"], inp["head_dim"])
        assert np.all(np.isfinite(rec["out"])) and np.all(np.isfinite(rec["lse"]))
        if s + 1 < len(W):
            assert np.all((rec["parent"] >= 0) & (rec["parent"] < W[s]))
            assert np.all(np.diff(rec["score"], axis=1) <= 0)
            assert np.array_equal(st["beam_path"][:, s + 1, :W[s + 1]], rec["parent"])
    # the last step's chains follow the parents the selections recorded
    anc = oracle.Oracle().ancestors(st, len(W) - 1)
    last = len(W) - 1
    for r in range(inp["num_requests"]):
        for b in range(W[last]):
            assert anc[r, b, last] == b
            assert anc[r, b, last - 1] == records[last - 1]["parent"][r, b]
            assert anc[r, b, last - 2] == records[last - 2]["parent"][r, anc[r, b, last - 1]]
