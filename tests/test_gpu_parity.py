"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Gate (stated with the target): BeamPath handling bit-exact; max |out - oracle|
<= 1e-2 on the bf16 outputs; max |lse - oracle| <= 1e-3.  The oracle is fp64;
the CUDA path computes in fp32 with bf16 P on the tensor cores.
"""

import os

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():   # pragma: no cover - CPU-only machines
    pytest.skip("needs a GPU", allow_module_level=True)

from gpu_util import DeviceWorkload, compare  # noqa: E402

ORC = oracle.Oracle()
_CACHE = {}


def workload(name):
    if name not in _CACHE:
        inp = workloads.make_inputs(workloads.WORKLOAD_BY_NAME[name])
        _CACHE[name] = (inp, DeviceWorkload(inp))
    return _CACHE[name]


def sample_rows(inp, step, n_random=40, seed=0):
    """Rows the oracle recomputes one by one at full size: the first and last
    beams of every request, beams on either side of 128-row tile edges, and
    random beams."""
    R, W_s, G = inp["num_requests"], int(inp["widths"][step]), inp["num_q_heads"] // inp["num_kv_heads"]
    per_tile = max(1, 128 // G)
    rows = set()
    for r in range(R):
        for b in (0, W_s - 1, per_tile - 1, per_tile, 2 * per_tile - 1, 2 * per_tile):
            if 0 <= b < W_s:
                rows.add((r, b))
    rng = np.random.default_rng(seed + step)
    for _ in range(n_random):
        rows.add((int(rng.integers(R)), int(rng.integers(W_s))))
    return sorted(rows)


@pytest.mark.parametrize("name", [workloads.WORKLOADS[0].name, workloads.WORKLOADS[1].name])
@pytest.mark.parametrize("step", [0, 1, 2])
def test_small_workloads_every_row(name, step):
    inp, dev = workload(name)
    out, lse = dev.run(step, guard=64)
    ref_out, ref_lse, ref_anc = ORC.decode_attn(inp, step)
    compare(out, lse, ref_out, ref_lse)
    assert np.array_equal(dev.ancestors(step), ref_anc)


@pytest.mark.parametrize("step", [0, 1, 2])
def test_headline_workload_every_row(step):
    """The measured workload (4 requests, 2048 context keys, 900 beams) in the
    plan and launch configuration the benchmark times: every row."""
    import beam_decode_attention_gb300 as gr
    inp, dev = workload(workloads.HEADLINE)
    assert gr.gr_decode_attn_plan(dev.shape, dev.widths, step)["fused_merge"] == 1
    out, lse = dev.run(step, guard=64)
    ref_out, ref_lse, ref_anc = ORC.decode_attn(inp, step)
    compare(out, lse, ref_out, ref_lse)
    assert np.array_equal(dev.ancestors(step), ref_anc)


@pytest.mark.parametrize("name", [w.name for w in workloads.WORKLOADS[2:]])
@pytest.mark.parametrize("step", [0, 1, 2])
def test_full_size_sampled_rows(name, step):
    inp, dev = workload(name)
    out, lse = dev.run(step, guard=64)
    # every row: finite, and bounded by the largest |value| it could average
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    vmax = max(float(np.nanmax(np.abs(workloads.bf16_bits_to_f32(inp["ctx_v"])))),
               float(np.nanmax(np.abs(workloads.bf16_bits_to_f32(inp["beam_v"])))))
    assert float(np.max(np.abs(out))) <= vmax * (1 + 2 ** -7)
    rows = sample_rows(inp, step)
    ref_out, ref_lse, _ = ORC.decode_attn(inp, step, rows=rows)
    idx_r = np.array([r for r, _ in rows])
    idx_b = np.array([b for _, b in rows])
    compare(out[idx_r, idx_b], lse[idx_r, idx_b], ref_out, ref_lse)
    # BeamPath: bit-exact on every row
    assert np.array_equal(dev.ancestors(step), ORC.ancestors(inp, step))


def _run_custom(inp, steps=None, splits=None):
    dev = DeviceWorkload(inp)
    for step in (steps if steps is not None else range(len(inp["widths"]))):
        if splits is not None:
            os.environ["GR_ATTN_FORCE_SPLITS"] = str(splits)
        try:
            out, lse = dev.run(step, guard=32)
        finally:
            os.environ.pop("GR_ATTN_FORCE_SPLITS", None)
        ref_out, ref_lse, ref_anc = ORC.decode_attn(inp, step)
        compare(out, lse, ref_out, ref_lse)
        assert np.array_equal(dev.ancestors(step), ref_anc)


def test_multi_tile_ragged():
    """Several 128-row tiles per (request, kv head) with a ragged last tile,
    several key blocks, ragged context lengths."""
    inp = workloads.make_custom(3, 16, 8, 128, [300, 1000, 129], [5, 70, 133], seed=101)
    _run_custom(inp)


@pytest.mark.parametrize("R", [31, 33])
def test_requests_ranked_by_context_length(R):
    """The tile-pair kernel takes the CTAs of the longest contexts first: the
    grid's request index is a rank by key blocks (ties by request index),
    computed in every warp for up to 32 requests and left as the index past
    that.  Ragged lengths with ties, empty contexts and a long one, on both
    sides of the 32-request limit: every row still lands in its own place."""
    rng = np.random.default_rng(500 + R)
    lens = [int(x) for x in rng.choice([0, 1, 128, 129, 300, 300, 700], size=R)]
    lens[R // 2] = 1500
    inp = workloads.make_custom(R, 4, 2, 64, lens, [3, 70, 140], seed=R)
    os.environ["GR_ATTN_FORCE_PATH"] = "pair"
    try:
        _run_custom(inp, splits=1)
    finally:
        os.environ.pop("GR_ATTN_FORCE_PATH", None)


@pytest.mark.parametrize("lens", [[0, 0], [1, 7], [127, 128], [129, 255], [0, 256]])
def test_context_length_edges(lens):
    inp = workloads.make_custom(2, 16, 8, 128, lens, [3, 9, 65], seed=sum(lens) + 3, lc_max=300)
    _run_custom(inp)


def test_no_context_capacity():
    inp = workloads.make_custom(2, 4, 2, 64, [0, 0], [2, 3, 4], seed=5, lc_max=0)
    _run_custom(inp)


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 8, 128), (16, 4, 128), (32, 4, 64), (4, 2, 64), (12, 4, 128)])
def test_head_geometries(Hq, Hkv, D):
    inp = workloads.make_custom(2, Hq, Hkv, D, [200, 77], [7, 33, 50], seed=Hq * 7 + Hkv + D)
    _run_custom(inp)


@pytest.mark.parametrize("lens", [[0, 300], [130, 1]])
def test_two_chain_blocks_per_level(lens):
    """One query head per kv head (G = 1) and up to 256 beams: a CTA of the
    fused single-split path holds two 128-beam tiles, so its per-beam stage
    walks 256 chains; with no context (ctx_len 0) the rows are the chain
    tokens alone, and with one context key few tokens carry all the weight."""
    import beam_decode_attention_gb300 as gr
    inp = workloads.make_custom(2, 4, 4, 128, lens, [5, 140, 256], seed=sum(lens) + 11)
    dev = DeviceWorkload(inp)
    os.environ["GR_ATTN_FORCE_SPLITS"] = "1"
    try:
        assert gr.gr_decode_attn_plan(dev.shape, dev.widths, 2)["fused_merge"] == 1
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)
    _run_custom(inp, splits=1)


def test_fused_chain_of_eight_levels():
    """Steps 5 and 7 in one key split: chains of six and eight tokens, the
    longest the fused single-split path takes."""
    import beam_decode_attention_gb300 as gr
    inp = workloads.make_custom(2, 16, 8, 128, [200, 90], [2, 3, 4, 5, 6, 7, 8, 9], seed=92)
    dev = DeviceWorkload(inp)
    os.environ["GR_ATTN_FORCE_SPLITS"] = "1"
    try:
        assert gr.gr_decode_attn_plan(dev.shape, dev.widths, 7)["fused_merge"] == 1
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)
    _run_custom(inp, steps=[5, 7], splits=1)


@pytest.mark.parametrize("path", ["persistent", "pair"])
def test_many_tiles_per_cta_mixed_contexts(path):
    """More 128-row tiles than SMs, so each CTA of the persistent kernel
    walks several items, with requests whose context is empty, one key,
    ragged and long mixed in the same grid (items without context have no
    key blocks; ragged tails are zeroed per ring slot) -- and the same call on
    the tile-pair kernel."""
    import beam_decode_attention_gb300 as gr
    inp = workloads.make_custom(8, 16, 8, 128, [0, 1, 127, 128, 129, 0, 3000, 700], [40, 200, 300], seed=121)
    dev = DeviceWorkload(inp)
    os.environ["GR_ATTN_FORCE_PATH"] = path
    try:
        for step in range(3):
            plan = gr.gr_decode_attn_plan(dev.shape, dev.widths, step)
            if plan["n_splits"] == 1:
                assert plan["persistent"] == (0 if path == "pair" else 1)
            out, lse = dev.run(step, guard=32)
            ref_out, ref_lse, ref_anc = ORC.decode_attn(inp, step)
            compare(out, lse, ref_out, ref_lse)
    finally:
        os.environ.pop("GR_ATTN_FORCE_PATH", None)
    assert gr.gr_get_device_error() == 0


@pytest.mark.parametrize("step", [0, 2])
def test_headline_on_the_persistent_kernel(step):
    """The measured workload on the persistent kernel (480 tiles on at most
    one CTA per SM, so each CTA takes three or four of them), which the
    planner leaves for calls whose tiles fit one round."""
    import beam_decode_attention_gb300 as gr
    inp, dev = workload(workloads.HEADLINE)
    os.environ["GR_ATTN_FORCE_PATH"] = "persistent"
    try:
        plan = gr.gr_decode_attn_plan(dev.shape, dev.widths, step)
        assert plan["persistent"] == 1 and plan["fused_merge"] == 1
        out, lse = dev.run(step, guard=64)
    finally:
        os.environ.pop("GR_ATTN_FORCE_PATH", None)
    rows = sample_rows(inp, step, n_random=200)
    ref_out, ref_lse, _ = ORC.decode_attn(inp, step, rows=rows)
    idx_r = np.array([r for r, _ in rows]); idx_b = np.array([b for _, b in rows])
    compare(out[idx_r, idx_b], lse[idx_r, idx_b], ref_out, ref_lse)


def test_width_one():
    inp = workloads.make_custom(3, 16, 8, 128, [64, 500, 3], [1, 1, 1], seed=17)
    _run_custom(inp)


@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_forced_splits(splits):
    inp = workloads.make_custom(2, 16, 8, 128, [777, 1024], [16, 40, 72], seed=29)
    _run_custom(inp, steps=[2], splits=splits)


@pytest.mark.parametrize("splits", [2, 3, 4])
def test_split_merge_in_kernel_several_tile_pairs(splits):
    """Several key splits merged inside the context kernel (the last split of
    each (request, kv head, tile pair) to finish merges): three tile pairs
    per (request, kv head) with a ragged last pair, a request whose context
    ends inside a split and one whose later splits are empty, every step in
    a row (the arrival counters start from zero in every call)."""
    import beam_decode_attention_gb300 as gr
    inp = workloads.make_custom(3, 16, 8, 128, [1024, 130, 777], [16, 140, 300], seed=31 + splits)
    dev = DeviceWorkload(inp)
    os.environ["GR_ATTN_FORCE_SPLITS"] = str(splits)
    try:
        plan = gr.gr_decode_attn_plan(dev.shape, dev.widths, 2)
        assert plan["n_splits"] == splits and plan["fused_merge"] == 1 and plan["kernels"] == 1
        assert gr.gr_decode_attn_workspace_size(dev.shape, dev.widths, 2) > 0
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)
    _run_custom(inp, splits=splits)
    _run_custom(inp, splits=splits)      # the same workspace again


def test_tagged_beam_values():
    """Context V = 0, each beam token's V is a one-hot code of (step, slot),
    queries sharpened x4: out names the chain tokens and their weights, so a
    wrong ancestor or a missing beam term gives an O(0.1) error."""
    D = 128
    inp = workloads.make_custom(2, 16, 8, D, [40, 300], [5, 9, 12], seed=61, q_scale=4.0)
    inp["ctx_v"][:] = 0
    W_max = inp["beam_capacity"]
    for t in range(3):
        for a in range(W_max):
            inp["beam_v"][:, t, a] = 0
            inp["beam_v"][:, t, a, :, t * W_max + a] = 0x3F80
    dev = DeviceWorkload(inp)
    for step in range(3):
        out, lse = dev.run(step)
        ref_out, ref_lse, _ = ORC.decode_attn(inp, step)
        assert float(np.max(np.abs(ref_out))) > 0.2
        compare(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("path", ["default", "persistent"])
def test_tagged_values_at_the_headline_geometry_fused(path):
    """The fused single-split epilogue at the headline geometry (Qwen3-0.6B
    heads, G = 2, 64 beams per 128-row tile, 900 beams: 14 full tiles and an
    8-row tail tile) with a strong signal.  Context V = 0 and each chain
    token's V is a random +-1 code of (request, step, slot, kv head), so out
    is the chain tokens' weights times their codes: a wrong ancestor, a
    missing chain term or a row written to the wrong place gives an O(0.1-1)
    error.  Queries x4 and chain keys x3 make the chain tokens carry a large
    share of the weight even against 2048 context keys; ctx_len 0 and 1 give
    chain-only rows.  Every row of every request at every step."""
    import beam_decode_attention_gb300 as gr
    inp = workloads.make_custom(4, 16, 8, 128, [2048, 0, 1, 2048], [900, 900, 900], seed=303, q_scale=4.0)
    inp["ctx_v"][:, :, :, :] = np.where(inp["ctx_v"] == workloads.BF16_NAN, workloads.BF16_NAN, 0).astype(np.uint16)
    bk = workloads.bf16_bits_to_f32(inp["beam_k"])
    inp["beam_k"] = workloads.f32_to_bf16_bits(bk * 3.0)
    rng = np.random.default_rng(304)
    signs = rng.integers(0, 2, size=inp["beam_v"].shape)
    inp["beam_v"] = np.where(signs == 1, 0x3F80, 0xBF80).astype(np.uint16)   # bf16 +1 / -1
    dev = DeviceWorkload(inp)
    os.environ["GR_ATTN_FORCE_SPLITS"] = "1"
    if path == "persistent":
        os.environ["GR_ATTN_FORCE_PATH"] = "persistent"
    try:
        for step in range(3):
            plan = gr.gr_decode_attn_plan(dev.shape, dev.widths, step)
            assert plan["fused_merge"] == 1 and plan["n_splits"] == 1
            assert plan["persistent"] == (1 if path == "persistent" else 0)
            out, lse = dev.run(step, guard=64)
            ref_out, ref_lse, ref_anc = ORC.decode_attn(inp, step)
            # the signal: chain-only rows are pure +-1 mixtures, and the
            # context rows still carry large chain weights
            assert float(np.max(np.abs(ref_out[1]))) > 0.9
            assert float(np.mean(np.abs(ref_out[0]))) > 0.08
            compare(out, lse, ref_out, ref_lse)
            assert np.array_equal(dev.ancestors(step), ref_anc)
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)
        os.environ.pop("GR_ATTN_FORCE_PATH", None)
    assert gr.gr_get_device_error() == 0


@pytest.mark.parametrize("jump", [3.0, 40.0])
def test_running_max_jumps(jump):
    """Context keys past position 300 are scaled up so that the scores of
    later key blocks exceed the running maximum by far (x3: the block sums
    pass the rescale limit; x40: exp2 overflows to inf before the rescale),
    and the first keys are scaled down: the online softmax must rescale O and
    l and redo the block, in either key split.  V is scaled by 1/4 (exact in
    bf16): such peaked weights make out nearly one V row, and with |v| up to
    ~4 the bf16 rounding of P and of out alone approaches the 1e-2 gate."""
    inp = workloads.make_custom(2, 16, 8, 128, [700, 1000], [4, 6, 9], seed=83, q_scale=2.0)
    k = workloads.bf16_bits_to_f32(inp["ctx_k"])
    k[:, :, 300:] *= jump
    k[:, :, :60] *= 0.25
    inp["ctx_k"] = workloads.f32_to_bf16_bits(k)
    for key in ("ctx_v", "beam_v"):
        inp[key] = workloads.f32_to_bf16_bits(workloads.bf16_bits_to_f32(inp[key]) * 0.25)
    for splits in (1, 2):
        _run_custom(inp, steps=[0, 2], splits=splits)
    os.environ["GR_ATTN_FORCE_PATH"] = "persistent"   # the O rescale of the persistent kernel
    try:
        _run_custom(inp, steps=[0, 2])
    finally:
        os.environ.pop("GR_ATTN_FORCE_PATH", None)


def test_repeatable_and_stream():
    inp = workloads.make_custom(2, 16, 8, 128, [333, 64], [8, 20, 30], seed=71)
    dev = DeviceWorkload(inp)
    a = dev.run(2)
    s = torch.cuda.Stream()
    b = dev.run(2, stream=s)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("splits,path", [(1, "pair"), (1, "persistent"), (2, "pair")])
def test_bad_parent_is_reported_not_followed(splits, path):
    """A parent outside [0, W_{t-1}) is counted by gr_validate_beam_path; the
    decode call reads nothing out of range, writes NaN to the rows whose
    chain meets it, flags the device error word, and leaves the other rows
    right -- in the fused single-split epilogue of both kernels and in the
    split path."""
    import beam_decode_attention_gb300 as gr
    inp = workloads.make_custom(2, 4, 2, 64, [150, 300], [3, 4, 5], seed=83)
    inp["beam_path"][1, 2, 2] = 4            # widths[1] == 4: out of range
    inp["beam_path"][0, 1, 0] = -3
    dev = DeviceWorkload(inp)
    assert gr.gr_get_device_error() == 0
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    gr.gr_validate_beam_path(dev.shape, dev.beam_path, dev.widths, 2, dev.ctx_len, bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == 2
    os.environ["GR_ATTN_FORCE_SPLITS"] = str(splits)
    if path == "persistent":
        os.environ["GR_ATTN_FORCE_PATH"] = "persistent"
    try:
        plan = gr.gr_decode_attn_plan(dev.shape, dev.widths, 2)
        assert plan["fused_merge"] == 1 and plan["kernels"] == 1 and plan["n_splits"] == splits
        assert plan["persistent"] == (1 if path == "persistent" else 0)
        out, lse = dev.run(2)
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)
        os.environ.pop("GR_ATTN_FORCE_PATH", None)
    assert gr.gr_get_device_error() == -8    # GR_ERR_BAD_BEAM_PATH
    assert gr.gr_get_device_error() == 0     # reading clears the word

    def hits_bad(r, b):
        slot = b
        for t in (2, 1):
            p = int(inp["beam_path"][r, t, slot])
            if not 0 <= p < int(inp["widths"][t - 1]):
                return True
            slot = p
        return False

    affected = [(r, b) for r in range(2) for b in range(5) if hits_bad(r, b)]
    good = [(r, b) for r in range(2) for b in range(5) if not hits_bad(r, b)]
    assert (1, 2) in affected and good
    for r, b in affected:
        assert np.isnan(out[r, b]).all() and np.isnan(lse[r, b]).all()
    anc = dev.ancestors(2)
    assert list(anc[1, 2]) == [-1, -1, 2]
    fixed = dict(inp, beam_path=np.where((inp["beam_path"] == 4) | (inp["beam_path"] == -3), 0,
                                         inp["beam_path"]))
    ref_out, ref_lse, _ = ORC.decode_attn(fixed, 2, rows=good)
    idx_r = np.array([r for r, _ in good]); idx_b = np.array([b for _, b in good])
    compare(out[idx_r, idx_b], lse[idx_r, idx_b], ref_out, ref_lse)


def test_error_statuses():
    import beam_decode_attention_gb300 as gr
    inp = workloads.make_custom(1, 4, 2, 64, [300], [2, 2], seed=3)
    dev = DeviceWorkload(inp)
    out, lse = dev.outputs(1)
    os.environ["GR_ATTN_FORCE_SPLITS"] = "2"     # a plan that needs a workspace
    try:
        need = gr.gr_decode_attn_workspace_size(dev.shape, dev.widths, 1)
        assert need > 0
        _error_statuses(gr, dev, out, lse, need)
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)


def _error_statuses(gr, dev, out, lse, need):
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gr.GRError) as e:
        gr.gr_decode_attn(dev.shape, dev.q[1], dev.ctx_k, dev.ctx_v, dev.ctx_len, dev.beam_k,
                          dev.beam_v, dev.beam_path, dev.widths, 1, out, lse, small)
    assert e.value.status == -5
    big = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(gr.GRError) as e:
        gr.gr_decode_attn(dev.shape, dev.q[1], dev.ctx_k, dev.ctx_v, dev.ctx_len, dev.beam_k,
                          dev.beam_v, dev.beam_path, dev.widths, 1, out[1:], lse, big)
    assert e.value.status == -4
    with pytest.raises(gr.GRError) as e:
        gr.gr_decode_attn(dev.shape, dev.q[1], dev.ctx_k, dev.ctx_v, dev.ctx_len, dev.beam_k,
                          dev.beam_v, dev.beam_path, [2, 3], 1, out, lse, big)
    assert e.value.status == -2


@pytest.mark.parametrize("path", ["simt", "default"])
def test_context_stage_paths_agree_with_oracle(path):
    """The CUDA-core context stage (GR_ATTN_FORCE_PATH=simt, the cross-check)
    and the default tensor-core stage both meet the gate on a multi-tile
    ragged case."""
    import beam_decode_attention_gb300 as gr
    inp = workloads.make_custom(2, 16, 8, 128, [520, 129], [9, 40, 140], seed=202)
    if path == "simt":
        os.environ["GR_ATTN_FORCE_PATH"] = "simt"
    try:
        dev = DeviceWorkload(inp)
        assert gr.gr_decode_attn_plan(dev.shape, dev.widths, 2)["path"] == (1 if path == "simt" else 0)
        for step in range(3):
            out, lse = dev.run(step, guard=16)
            ref_out, ref_lse, _ = ORC.decode_attn(inp, step)
            compare(out, lse, ref_out, ref_lse)
    finally:
        os.environ.pop("GR_ATTN_FORCE_PATH", None)


def test_long_chain_beyond_fused_epilogue():
    """Nine decode steps: longer than the fused epilogue holds, so the call
    takes the partial + merge path; still exact against the oracle."""
    import beam_decode_attention_gb300 as gr
    inp = workloads.make_custom(2, 16, 8, 128, [200, 90], [2, 3, 4, 5, 6, 7, 8, 9, 10], seed=91)
    dev = DeviceWorkload(inp)
    assert gr.gr_decode_attn_plan(dev.shape, dev.widths, 8)["fused_merge"] == 0
    assert gr.gr_decode_attn_plan(dev.shape, dev.widths, 7)["fused_merge"] in (0, 1)
    for splits in (None, 2):
        if splits is not None:
            os.environ["GR_ATTN_FORCE_SPLITS"] = str(splits)
        try:
            plan = gr.gr_decode_attn_plan(dev.shape, dev.widths, 8)
            assert plan["kernels"] == 2 and plan["fused_merge"] == 0
            for step in (7, 8):
                out, lse = dev.run(step, guard=16)
                ref_out, ref_lse, ref_anc = ORC.decode_attn(inp, step)
                compare(out, lse, ref_out, ref_lse)
                assert np.array_equal(dev.ancestors(step), ref_anc)
        finally:
            os.environ.pop("GR_ATTN_FORCE_SPLITS", None)
