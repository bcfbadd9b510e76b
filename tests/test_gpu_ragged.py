"""gr_decode_attn_ragged: a beam width per request in one batch (SID-GR
README, section 10 "TODO and Roadmap", per-request beam widths).

Each request's rows b < W[r][s] are checked against the oracle on the padded
workload (the tensors keep each step's largest width), and bit-for-bit
against gr_decode_attn on the same padded tensors, whose plan is the same;
parents are checked against the request's own previous width."""

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
from gpu_util import DeviceWorkload, compare, to_dev  # noqa: E402

ORC = oracle.Oracle()

# request widths per step; the padded layout takes each step's largest
WIDTHS = [[5, 70, 133], [3, 9, 20], [5, 40, 300]]


def ragged_inputs(widths, seed):
    W = np.asarray(widths, np.int32)
    wpad = W.max(axis=0)
    inp = workloads.make_custom(len(widths), 16, 8, 128, [700, 0, 1000], [int(w) for w in wpad], seed=seed, lc_max=1000)
    bp = inp["beam_path"]
    for r in range(W.shape[0]):
        for t in range(1, W.shape[1]):
            bp[r, t, :wpad[t]] %= W[r, t - 1]   # parents inside the request's own width
    return inp, W


def run_ragged(dev, W, step):
    out, lse = dev.outputs(step)
    ws = torch.empty(max(16, gr.gr_decode_attn_workspace_size(dev.shape, dev.widths, step)),
                     dtype=torch.uint8, device="cuda")
    S_max = dev.inp["step_capacity"]
    wdev = np.zeros((W.shape[0], S_max), np.int32)
    wdev[:, :W.shape[1]] = W
    gr.gr_decode_attn_ragged(dev.shape, dev.q[step], dev.ctx_k, dev.ctx_v, dev.ctx_len, dev.beam_k, dev.beam_v,
                             dev.beam_path, W.tolist(), to_dev(wdev), step, out, lse, ws)
    torch.cuda.synchronize()
    R, Hq, D = dev.inp["num_requests"], dev.inp["num_q_heads"], dev.inp["head_dim"]
    Wp = dev.widths[step]
    o = (out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).reshape(R, Wp, Hq, D)
    return o, lse.cpu().numpy().reshape(R, Wp, Hq)


@pytest.mark.parametrize("splits,path", [(1, "pair"), (1, "persistent"), (2, "pair")])
def test_ragged_rows_match_oracle_and_padded_call(splits, path):
    inp, W = ragged_inputs(WIDTHS, seed=91 + splits)
    dev = DeviceWorkload(inp)
    os.environ["GR_ATTN_FORCE_SPLITS"] = str(splits)
    if path == "persistent":
        os.environ["GR_ATTN_FORCE_PATH"] = "persistent"
    try:
        for step in range(3):
            assert gr.gr_get_device_error() == 0
            out, lse = run_ragged(dev, W, step)
            assert gr.gr_get_device_error() == 0
            dense_out, dense_lse = dev.run(step)
            ref_out, ref_lse, _ = ORC.decode_attn(inp, step)
            for r in range(W.shape[0]):
                w = int(W[r, step])
                compare(out[r, :w], lse[r, :w], ref_out[r, :w], ref_lse[r, :w])
                assert np.array_equal(out[r, :w], dense_out[r, :w], equal_nan=True)
                assert np.array_equal(lse[r, :w], dense_lse[r, :w], equal_nan=True)
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)
        os.environ.pop("GR_ATTN_FORCE_PATH", None)


def test_ragged_parent_checked_against_request_width():
    """A parent inside the padded width but at or past the request's own
    previous width is a bad parent for that request alone."""
    inp, W = ragged_inputs(WIDTHS, seed=97)
    inp["beam_path"][1, 2, 2] = int(W[1, 1])      # request 1 had 9 beams at step 1
    dev = DeviceWorkload(inp)
    assert gr.gr_get_device_error() == 0
    out, lse = run_ragged(dev, W, 2)
    assert gr.gr_get_device_error() == -8          # GR_ERR_BAD_BEAM_PATH
    assert np.isnan(lse[1, 2]).all() and np.isnan(out[1, 2]).all()
    ref_out, ref_lse, _ = ORC.decode_attn(inp, 2)   # the padded workload: every parent in range
    good = [b for b in range(int(W[1, 2])) if b != 2]
    compare(out[1, good], lse[1, good], ref_out[1, good], ref_lse[1, good])
    for r in (0, 2):
        w = int(W[r, 2])
        compare(out[r, :w], lse[r, :w], ref_out[r, :w], ref_lse[r, :w])


def test_ragged_rejects_bad_widths_and_simt_path():
    inp, W = ragged_inputs(WIDTHS, seed=5)
    dev = DeviceWorkload(inp)
    out, lse = dev.outputs(2)
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    wdev = to_dev(np.zeros((3, inp["step_capacity"]), np.int32))
    for bad in ([[0, 1, 1]] + W.tolist()[1:], [[5, 70, 301]] + W.tolist()[1:]):
        with pytest.raises(gr.GRError) as e:
            gr.gr_decode_attn_ragged(dev.shape, dev.q[2], dev.ctx_k, dev.ctx_v, dev.ctx_len, dev.beam_k,
                                     dev.beam_v, dev.beam_path, bad, wdev, 2, out, lse, ws)
        assert e.value.status == -2
    os.environ["GR_ATTN_FORCE_PATH"] = "simt"
    try:
        with pytest.raises(gr.GRError) as e:
            gr.gr_decode_attn_ragged(dev.shape, dev.q[2], dev.ctx_k, dev.ctx_v, dev.ctx_len, dev.beam_k,
                                     dev.beam_v, dev.beam_path, W.tolist(), wdev, 2, out, lse, ws)
        assert e.value.status == -3   # GR_ERR_UNSUPPORTED
    finally:
        os.environ.pop("GR_ATTN_FORCE_PATH", None)
