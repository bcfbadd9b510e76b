"""gr_beam_reorder: the reordered per-beam cache equals, byte for byte, the
gather the CPU oracle's ancestor table defines; decode attention over it
(the identity path, every level W_s wide) meets the oracle's gate on the
original inputs, and equals attention over the original cache through
BeamPath bit for bit, in the fused and the split path."""

import os

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():   # pragma: no cover - CPU-only machines
    pytest.skip("needs a GPU", allow_module_level=True)

import beam_decode_attention_gb300 as gr  # noqa: E402
from gpu_util import DeviceWorkload, compare  # noqa: E402

ORC = oracle.Oracle()


def oracle_gather(inp, step):
    """The reordered cache the oracle's ancestor table defines:
    out[r, t, b] = beam_kv[r, t, a_t(b)] for t <= step, b < W_step, and the
    identity path; every other entry keeps the poison it started with."""
    anc = ORC.ancestors(inp, step)                      # [R, W_s, step+1]
    W_s = int(inp["widths"][step])
    ok = np.full_like(inp["beam_k"], 0x7FC0)
    ov = np.full_like(inp["beam_v"], 0x7FC0)
    op = np.full_like(inp["beam_path"], -1)
    for r in range(inp["num_requests"]):
        for t in range(step + 1):
            ok[r, t, :W_s] = inp["beam_k"][r, t, anc[r, :, t]]
            ov[r, t, :W_s] = inp["beam_v"][r, t, anc[r, :, t]]
            op[r, t, :W_s] = np.arange(W_s) if t > 0 else 0
    return ok, ov, op


def _bits(t):
    return t.cpu().numpy().view(np.uint16) if t.dtype == torch.int16 else t.cpu().numpy()


@pytest.mark.parametrize("name", ["qwen3_0.6b_r8_lc1024_w128", "qwen3_0.6b_r4_lc2048_w900"])
@pytest.mark.parametrize("step", [0, 1, 2])
def test_reordered_bytes_equal_the_oracle_gather(name, step):
    inp = workloads.make_inputs(workloads.WORKLOAD_BY_NAME[name])
    dev = DeviceWorkload(inp)
    ok = torch.full_like(dev.beam_k, 0x7FC0)
    ov = torch.full_like(dev.beam_v, 0x7FC0)
    op = torch.full_like(dev.beam_path, -1)
    gr.gr_beam_reorder(dev.shape, dev.beam_k, dev.beam_v, dev.beam_path, dev.widths, step, ok, ov, op)
    torch.cuda.synchronize()
    want_k, want_v, want_p = oracle_gather(inp, step)
    assert np.array_equal(_bits(ok), want_k)
    assert np.array_equal(_bits(ov), want_v)
    assert np.array_equal(_bits(op), want_p)
    assert gr.gr_get_device_error() == 0


@pytest.mark.parametrize("splits", [1, 2])
def test_attention_on_reordered_cache_meets_the_oracle(splits):
    inp = workloads.make_custom(2, 16, 8, 128, [300, 1000], [5, 70, 133], seed=50 + splits)
    dev = DeviceWorkload(inp)
    os.environ["GR_ATTN_FORCE_SPLITS"] = str(splits)
    try:
        for step in (1, 2):
            ok, ov, op = torch.empty_like(dev.beam_k), torch.empty_like(dev.beam_v), torch.empty_like(dev.beam_path)
            gr.gr_beam_reorder(dev.shape, dev.beam_k, dev.beam_v, dev.beam_path, dev.widths, step, ok, ov, op)
            flat = [dev.widths[step]] * len(dev.widths)
            out, lse = dev.outputs(step)
            ws = torch.empty(max(16, gr.gr_decode_attn_workspace_size(dev.shape, flat, step)),
                             dtype=torch.uint8, device="cuda")
            gr.gr_decode_attn(dev.shape, dev.q[step], dev.ctx_k, dev.ctx_v, dev.ctx_len, ok, ov, op, flat, step,
                              out, lse, ws)
            torch.cuda.synchronize()
            ref_out, ref_lse, _ = ORC.decode_attn(inp, step)      # the original cache, through BeamPath
            got = (out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
            compare(got.reshape(ref_out.shape), lse.cpu().numpy().reshape(ref_lse.shape), ref_out, ref_lse)
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)


@pytest.mark.parametrize("splits", [1, 2])
def test_reordered_cache_gives_the_same_rows(splits):
    inp = workloads.make_custom(2, 16, 8, 128, [300, 1000], [5, 70, 133], seed=40 + splits)
    dev = DeviceWorkload(inp)
    os.environ["GR_ATTN_FORCE_SPLITS"] = str(splits)
    try:
        for step in (1, 2):
            ref_out, ref_lse = dev.run(step)
            ok = torch.full_like(dev.beam_k, 0x7FC0)      # NaN: any row not written would show
            ov = torch.full_like(dev.beam_v, 0x7FC0)
            op = torch.full_like(dev.beam_path, -1)
            gr.gr_beam_reorder(dev.shape, dev.beam_k, dev.beam_v, dev.beam_path, dev.widths, step, ok, ov, op)
            flat = [dev.widths[step]] * len(dev.widths)
            out, lse = dev.outputs(step)
            ws = torch.empty(max(16, gr.gr_decode_attn_workspace_size(dev.shape, flat, step)),
                             dtype=torch.uint8, device="cuda")
            gr.gr_decode_attn(dev.shape, dev.q[step], dev.ctx_k, dev.ctx_v, dev.ctx_len, ok, ov, op, flat, step,
                              out, lse, ws)
            torch.cuda.synchronize()
            got = (out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
            assert np.array_equal(got.reshape(ref_out.shape), ref_out)
            assert np.array_equal(lse.cpu().numpy().reshape(ref_lse.shape), ref_lse)
            assert gr.gr_get_device_error() == 0
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)


def test_reorder_refuses_in_place():
    inp = workloads.make_custom(1, 4, 2, 64, [100], [2, 3], seed=2)
    dev = DeviceWorkload(inp)
    op = torch.empty_like(dev.beam_path)
    with pytest.raises(gr.GRError) as e:
        gr.gr_beam_reorder(dev.shape, dev.beam_k, dev.beam_v, dev.beam_path, dev.widths, 1, dev.beam_k,
                           torch.empty_like(dev.beam_v), op)
    assert e.value.status == -2


def oracle_inplace(inp, step, broken=()):
    """The cache and path after an in-place reorder at `step`, from the
    oracle's ancestor table: levels t < step get row b = old row a_t(b) for
    b < W_step, levels 1..step get the identity path there, and everything
    else keeps its old contents.  `broken` lists (r, b, t_break) beams whose
    chain breaks at level t_break: their rows below it stay as they were."""
    anc = ORC.ancestors(inp, step)
    W_s = int(inp["widths"][step])
    k, v, p = inp["beam_k"].copy(), inp["beam_v"].copy(), inp["beam_path"].copy()
    for r in range(inp["num_requests"]):
        for t in range(step):
            k[r, t, :W_s] = inp["beam_k"][r, t, anc[r, :, t]]
            v[r, t, :W_s] = inp["beam_v"][r, t, anc[r, :, t]]
        for t in range(1, step + 1):
            p[r, t, :W_s] = np.arange(W_s)
    for r, b, tb in broken:
        k[r, :tb, b] = inp["beam_k"][r, :tb, b]
        v[r, :tb, b] = inp["beam_v"][r, :tb, b]
    return k, v, p


@pytest.mark.parametrize("name", ["qwen3_0.6b_r8_lc1024_w128", "qwen3_0.6b_r4_lc2048_w900",
                                  "qwen3_1.7b_r16_lc512-4096_w20-300-900"])
@pytest.mark.parametrize("step", [0, 1, 2])
def test_inplace_reorder_equals_the_oracle_gather(name, step):
    inp = workloads.make_inputs(workloads.WORKLOAD_BY_NAME[name])
    dev = DeviceWorkload(inp)
    gr.gr_beam_reorder_inplace(dev.shape, dev.beam_k, dev.beam_v, dev.beam_path, dev.widths, step)
    torch.cuda.synchronize()
    want_k, want_v, want_p = oracle_inplace(inp, step)
    assert np.array_equal(_bits(dev.beam_k), want_k)
    assert np.array_equal(_bits(dev.beam_v), want_v)
    assert np.array_equal(_bits(dev.beam_path), want_p)
    assert gr.gr_get_device_error() == 0


@pytest.mark.parametrize("splits", [1, 2])
def test_attention_after_inplace_reorder_gives_the_same_rows(splits):
    inp = workloads.make_custom(2, 16, 8, 128, [300, 1000], [5, 70, 133], seed=60 + splits)
    os.environ["GR_ATTN_FORCE_SPLITS"] = str(splits)
    try:
        for step in (1, 2):
            dev = DeviceWorkload(inp)
            ref_out, ref_lse = dev.run(step)
            gr.gr_beam_reorder_inplace(dev.shape, dev.beam_k, dev.beam_v, dev.beam_path, dev.widths, step)
            dev.widths = [dev.widths[step]] * (step + 1) + dev.widths[step + 1:]
            out, lse = dev.run(step)
            assert np.array_equal(out, ref_out)
            assert np.array_equal(lse, ref_lse)
            assert gr.gr_get_device_error() == 0
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)


def test_inplace_reorder_stops_at_a_broken_chain():
    inp = workloads.make_custom(2, 8, 4, 64, [100, 200], [6, 40, 40], seed=71)
    good = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in inp.items()}
    bad = dict(good)
    bad["beam_path"] = good["beam_path"].copy()
    bad["beam_path"][1, 2, 7] = 40 + 3          # outside [0, W_1): the chain of (1, 7) breaks at level 2
    dev = DeviceWorkload(bad)
    gr.gr_beam_reorder_inplace(dev.shape, dev.beam_k, dev.beam_v, dev.beam_path, dev.widths, 2)
    torch.cuda.synchronize()
    assert gr.gr_get_device_error() == -8
    # the other beams follow the intact path; beam (1, 7) keeps its levels 0 and 1
    want_k, want_v, want_p = oracle_inplace(good, 2, broken=[(1, 7, 2)])
    assert np.array_equal(_bits(dev.beam_k), want_k)
    assert np.array_equal(_bits(dev.beam_v), want_v)
    assert np.array_equal(_bits(dev.beam_path), want_p)


def test_inplace_reorder_refuses_shared_buffers():
    inp = workloads.make_custom(1, 4, 2, 64, [100], [2, 3], seed=2)
    dev = DeviceWorkload(inp)
    with pytest.raises(gr.GRError) as e:
        gr.gr_beam_reorder_inplace(dev.shape, dev.beam_k, dev.beam_k, dev.beam_path, dev.widths, 1)
    assert e.value.status == -2
