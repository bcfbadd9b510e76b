"""gr_beam_reorder: decode attention over the reordered per-beam cache (the
identity path, every level W_s wide) equals attention over the original
cache through BeamPath, bit for bit, in the fused and the split path."""

import os

import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():   # pragma: no cover - CPU-only machines
    pytest.skip("needs a GPU", allow_module_level=True)

import beam_decode_attention_gb300 as gr  # noqa: E402
from gpu_util import DeviceWorkload  # noqa: E402


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
