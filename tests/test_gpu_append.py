"""gr_beam_append: the step's new K/V rows land in their own slots of the
step plane, byte for byte, from a dense [R, W_s, Hkv, D] source or from rows
of a wider (fused-QKV-like) buffer; nothing else in BeamKV changes."""

import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():   # pragma: no cover - CPU-only machines
    pytest.skip("needs a GPU", allow_module_level=True)

import beam_decode_attention_gb300 as gr  # noqa: E402
from gpu_util import to_dev  # noqa: E402


@pytest.mark.parametrize("R,Hkv,D,widths,step", [(1, 2, 64, (4, 4, 4), 1), (4, 8, 128, (900, 900, 900), 2),
                                                   (16, 8, 128, (20, 300, 900), 0), (3, 1, 64, (5, 7), 1),
                                                   (16, 8, 128, (20, 300, 900), 1)])
@pytest.mark.parametrize("extra", [0, 2])
def test_append_writes_the_step_plane(R, Hkv, D, widths, step, extra):
    S, W_max, W_s = len(widths), max(widths), widths[step]
    row = Hkv * D
    stride = row * (1 + extra)      # extra > 0: each beam's row sits inside a wider row
    rng = np.random.Generator(np.random.PCG64(R * 100 + step * 10 + extra))
    k_src = workloads.f32_to_bf16_bits(rng.standard_normal((R * W_s, stride), dtype=np.float32))
    v_src = workloads.f32_to_bf16_bits(rng.standard_normal((R * W_s, stride), dtype=np.float32))
    poison = np.full((R, S, W_max, Hkv, D), workloads.BF16_NAN, np.uint16)
    bk, bv = to_dev(poison), to_dev(poison)
    shape = gr.Shape(R, 2 * Hkv, Hkv, D, 0, S, W_max, float(D) ** -0.5)
    gr.gr_beam_append(shape, list(widths), step, to_dev(k_src), to_dev(v_src), bk, bv, src_stride=stride)
    torch.cuda.synchronize()
    want_k, want_v = poison.copy(), poison.copy()
    want_k[:, step, :W_s] = k_src[:, :row].reshape(R, W_s, Hkv, D)
    want_v[:, step, :W_s] = v_src[:, :row].reshape(R, W_s, Hkv, D)
    assert np.array_equal(bk.cpu().numpy().view(np.uint16), want_k)
    assert np.array_equal(bv.cpu().numpy().view(np.uint16), want_v)


def test_append_refuses_a_source_inside_beamkv():
    shape = gr.Shape(1, 4, 2, 64, 0, 2, 4, 0.125)
    bk = torch.zeros(1 * 2 * 4 * 2 * 64, dtype=torch.int16, device="cuda")
    bv = torch.zeros_like(bk)
    with pytest.raises(gr.GRError) as e:
        gr.gr_beam_append(shape, [4, 4], 1, bk[:512], bv[:512], bk, bv)
    assert e.value.status == -2
