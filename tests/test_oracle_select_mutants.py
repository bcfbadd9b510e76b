"""The beam-selection pins must reject plausible mistakes: each variant of the
oracle below plants one (in a copy, on the CPU) and some pin has to fail."""

import numpy as np
import pytest

from oracle import select
import test_oracle_select as pins


def _select_with(lp_fn, order="desc", ties="flat_asc", beam_sign=1.0):
    def fn(z, S, n):
        lp = lp_fn(np.asarray(z, np.float64))
        sc = beam_sign * np.asarray(S, np.float64)[..., None] + lp
        R, W, V = sc.shape
        flat = sc.reshape(R, W * V)
        idx = np.arange(W * V)
        par, tok, best = [], [], []
        for r in range(R):
            key = -flat[r] if order == "desc" else flat[r]
            tie = idx if ties == "flat_asc" else -idx
            pick = np.lexsort((tie, key))[:n]
            par.append(pick // V)
            tok.append(pick % V)
            best.append(flat[r, pick])
        return np.array(par), np.array(tok), np.array(best)
    return fn


def _no_norm(z):
    return z


def _max_only(z):
    return z - z.max(axis=-1, keepdims=True)


def _log_of_sum(z):   # forgets the exponentials
    return z - np.log(np.abs(z).sum(axis=-1, keepdims=True))


MUTANTS = {
    "no log-normaliser": _select_with(_no_norm),
    "max subtracted only": _select_with(_max_only),
    "log of the plain sum": _select_with(_log_of_sum),
    "ascending scores": _select_with(select.log_softmax, order="asc"),
    "ties to the larger flat index": _select_with(select.log_softmax, ties="flat_desc"),
    "beam score ignored": _select_with(select.log_softmax, beam_sign=0.0),
    "beam score subtracted": _select_with(select.log_softmax, beam_sign=-1.0),
}


def _pins_pass(fn):
    try:
        for case in pins.hand_cases():
            parent, token, score = fn(case["z"], case["S"], case["n"])
            want = case["want"]
            assert [int(x) for x in parent[0]] == [w[0] for w in want]
            assert [int(x) for x in token[0]] == [w[1] for w in want]
            assert np.allclose(score[0], [w[2] for w in want], rtol=0, atol=1e-14)
        rng = np.random.default_rng(123)
        z = rng.standard_normal((2, 4, 9)) * 2.0
        S = -np.abs(rng.standard_normal((2, 4))) * 3.0
        parent, token, score = fn(z, S, 5)
        for r, ref in enumerate(pins._brute(z, S, 5)):
            assert [int(x) for x in parent[r]] == [p for p, _, _ in ref]
            assert [int(x) for x in token[r]] == [t for _, t, _ in ref]
            assert np.allclose(score[r], [s for _, _, s in ref], rtol=0, atol=1e-12)
    except AssertionError:
        return False
    return True


def test_the_oracle_itself_passes():
    assert _pins_pass(select.beam_select)
    assert _pins_pass(_select_with(select.log_softmax))   # the harness's own copy


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_each_planted_mistake_is_caught(name):
    assert not _pins_pass(MUTANTS[name]), f"no pin caught: {name}"
