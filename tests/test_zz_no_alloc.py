"""gr_decode_attn_noalloc against gr_decode_attn, through the C ABI, on the GPU.

gr_decode_attn_noalloc is for callers that cannot allocate device memory
(engines whose memory pool already holds the device memory, paths that
cannot afford cudaMalloc's synchronisation): it keeps the context stage's
partial results in a static array inside the library instead of a caller
workspace.  Both entry points run the same kernels on the same plan, so two
calls in a row must give bit-identical outputs to the workspace entry point
(a tolerance could hide a race on the reused scratch).  A call needing more
scratch than the array holds is refused without touching its outputs.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""

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

def _noalloc(dev, step):
    R, Hq, D = dev.inp["num_requests"], dev.inp["num_q_heads"], dev.inp["head_dim"]
    W_s = dev.widths[step]
    out, lse = dev.outputs(step)
    gr.gr_decode_attn_noalloc(dev.shape, dev.q[step], dev.ctx_k, dev.ctx_v, dev.ctx_len,
                              dev.beam_k, dev.beam_v, dev.beam_path, dev.widths, step, out, lse)
    torch.cuda.synchronize()
    o = (out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    return o.reshape(R, W_s, Hq, D), lse.cpu().numpy().reshape(R, W_s, Hq)


@pytest.mark.parametrize("splits", [None, 2, 3])
def test_noalloc_matches_workspace_entry_point_on_two_calls(splits):
    """Two calls in a row (the second on another step, so its partials land
    over the first call's), each bit-identical to gr_decode_attn; forced key
    splits make the plan keep partials in the scratch."""
    inp = workloads.make_inputs(workloads.WORKLOAD_BY_NAME["qwen3_0.6b_r8_lc1024_w128"])
    dev = DeviceWorkload(inp)
    if splits is not None:
        os.environ["GR_ATTN_FORCE_SPLITS"] = str(splits)
    try:
        if splits is not None:
            assert gr.gr_decode_attn_workspace_size(dev.shape, dev.widths, 2) > 0
        for step in (2, 1):
            ref_out, ref_lse = dev.run(step)
            out, lse = _noalloc(dev, step)
            assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
            assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)
    assert gr.gr_get_device_error() == 0


def test_noalloc_refuses_a_call_beyond_its_scratch():
    # 57600 rows x (128 + 1) fp32 per key split: three splits need ~89 MB,
    # more than the 64 MiB static scratch
    inp = workloads.make_custom(4, 16, 8, 128, [1024] * 4, [900], seed=5)
    dev = DeviceWorkload(inp)
    out, lse = dev.outputs(0)
    os.environ["GR_ATTN_FORCE_SPLITS"] = "3"
    try:
        need = gr.gr_decode_attn_workspace_size(dev.shape, dev.widths, 0)
        assert need > gr.NOALLOC_SCRATCH_BYTES
        with pytest.raises(gr.GRError) as e:
            gr.gr_decode_attn_noalloc(dev.shape, dev.q[0], dev.ctx_k, dev.ctx_v, dev.ctx_len,
                                      dev.beam_k, dev.beam_v, dev.beam_path, dev.widths, 0, out, lse)
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)
    assert e.value.status == -5      # GR_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.all(out == 0x5A5A) and torch.all(lse == 7.25)   # nothing was enqueued
