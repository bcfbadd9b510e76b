"""The input builders for the paged and per-request-width layouts (CPU):
the pool holds every context position at its block-table page, and each
request's BeamPath parents stay inside its own previous width."""

import numpy as np
import pytest

import workloads


def test_paged_pool_holds_the_context():
    inp = workloads.make_custom(3, 4, 2, 64, [300, 0, 257], [2, 3], seed=5, lc_max=300)
    for page_size in (128, 256):
        pool, table, ppr, P = workloads.paged_pool(inp["ctx_k"], page_size, 4, seed=2)
        assert ppr == -(-300 // page_size) and P == 3 * ppr + 4
        assert sorted(table.ravel().tolist()) == sorted(set(table.ravel().tolist()))   # distinct pages
        for r in range(3):
            for j in range(300):
                page, off = table[r, j // page_size], j % page_size
                assert np.array_equal(pool[page, :, off], inp["ctx_k"][r, :, j])
        # past the context capacity, and on spare pages, the pool holds NaN
        tail = ppr * page_size - 300
        if tail:
            assert np.all(pool[table[0, -1], :, page_size - tail:] == workloads.BF16_NAN)
        spare = sorted(set(range(P)) - set(table.ravel().tolist()))
        assert len(spare) == 4 and np.all(pool[spare] == workloads.BF16_NAN)


def test_make_ragged_keeps_parents_in_each_request_width():
    spec = workloads.WORKLOADS[1]                     # 8 requests, width 128 at each of 3 steps
    assert spec.num_requests == 8 and tuple(spec.widths) == (128, 128, 128)
    W = [[128, 128, 128]] + [[w, max(1, w // 2), w] for w in (7, 50, 1, 128, 64, 3, 100)]
    inp, Wa = workloads.make_ragged(spec, W)
    assert Wa.shape == (spec.num_requests, spec.steps)
    bp = inp["beam_path"]
    for r in range(spec.num_requests):
        assert np.all(bp[r, 0, :spec.widths[0]] == 0)
        for t in range(1, spec.steps):
            rows = bp[r, t, :Wa[r, t]]
            assert rows.min() >= 0 and rows.max() < Wa[r, t - 1]


def test_make_ragged_rejects_bad_widths():
    spec = workloads.WORKLOADS[1]
    good = [list(spec.widths)] * spec.num_requests
    with pytest.raises(ValueError):
        workloads.make_ragged(spec, good[:-1])                      # a request missing
    with pytest.raises(ValueError):
        workloads.make_ragged(spec, [[0] * spec.steps] + good[1:])  # a width below 1
    with pytest.raises(ValueError):
        workloads.make_ragged(spec, [[max(1, w - 1) for w in spec.widths]] * spec.num_requests)   # no request at the padded width


def test_parity_gate_rounding_allowance():
    """The GPU parity gate allows half a bf16 ulp of the oracle value on top
    of 1e-2: check that allowance against the bf16 rounding the workloads
    use (it bounds every rounding error and is reached)."""
    from gpu_util import bf16_half_ulp
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(200000) * s for s in (0.01, 1.0, 3.0, 100.0)]).astype(np.float32)
    r = workloads.bf16_bits_to_f32(workloads.f32_to_bf16_bits(x)).astype(np.float64)
    err = np.abs(r - x.astype(np.float64))
    hu = bf16_half_ulp(x)
    assert np.all(err <= hu)
    assert np.max(err / hu) > 0.999
    assert bf16_half_ulp(np.array([4.0]))[0] == 2.0 ** -6 and bf16_half_ulp(np.array([3.99]))[0] == 2.0 ** -7
