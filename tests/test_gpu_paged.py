"""gr_decode_attn_paged (ContextKV in pages of a shared pool, through a block
table) against the CPU oracle on the dense copy of the same context, within
the parity gate; and against gr_decode_attn on the dense layout, where the
context kernel reads the same values in the same order, so the outputs must
be bit-identical, in the fused single-split path and the split path."""

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


def paged_pool(ctx, page_size, extra_pages, seed):
    """The dense [R, Hkv, Lc_max, D] context as pages of a shuffled pool
    [P, Hkv, page_size, D] plus the block table; padding past Lc_max is NaN."""
    R, Hkv, Lc, D = ctx.shape
    ppr = max(1, -(-Lc // page_size))
    P = R * ppr + extra_pages
    rng = np.random.default_rng(seed)
    order = rng.permutation(P)
    pool = np.full((P, Hkv, page_size, D), workloads.BF16_NAN, np.uint16)
    table = np.empty((R, ppr), np.int32)
    for r in range(R):
        for i in range(ppr):
            page = int(order[r * ppr + i])
            table[r, i] = page
            seg = ctx[r, :, i * page_size:(i + 1) * page_size]
            pool[page, :, :seg.shape[1]] = seg
    return pool, table, ppr, P


@pytest.mark.parametrize("page_size,splits", [(128, 1), (256, 1), (128, 2), (256, 3)])
def test_paged_matches_dense_bit_for_bit(page_size, splits):
    inp = workloads.make_custom(3, 16, 8, 128, [700, 0, 1000], [5, 70, 133], seed=page_size + splits, lc_max=1000)
    dev = DeviceWorkload(inp)
    kp, table, ppr, P = paged_pool(inp["ctx_k"], page_size, 5, seed=1)
    vp, _, _, _ = paged_pool(inp["ctx_v"], page_size, 5, seed=1)
    pages = gr.CtxPages(page_size, P, ppr)
    kp_d, vp_d, tb_d = to_dev(kp), to_dev(vp), to_dev(table)
    os.environ["GR_ATTN_FORCE_SPLITS"] = str(splits)
    try:
        for step in range(3):
            dense_out, dense_lse = dev.run(step)
            out, lse = dev.outputs(step)
            ws = torch.empty(max(16, gr.gr_decode_attn_workspace_size(dev.shape, dev.widths, step)),
                             dtype=torch.uint8, device="cuda")
            gr.gr_decode_attn_paged(dev.shape, pages, dev.q[step], kp_d, vp_d, dev.ctx_len, tb_d, dev.beam_k,
                                    dev.beam_v, dev.beam_path, dev.widths, step, out, lse, ws)
            torch.cuda.synchronize()
            got = (out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
            assert np.array_equal(got.reshape(dense_out.shape), dense_out, equal_nan=True)
            assert np.array_equal(lse.cpu().numpy().reshape(dense_lse.shape), dense_lse, equal_nan=True)
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)


@pytest.mark.parametrize("page_size,splits", [(128, 1), (256, 1), (128, 2), (256, 2), (128, 3), (256, 3)])
def test_paged_meets_the_oracle(page_size, splits):
    """Every row of every step against the fp64 oracle on the dense context;
    one request has no context, one a context that ends inside a page."""
    inp = workloads.make_custom(3, 16, 8, 128, [900, 0, 1000], [7, 60, 129], seed=7 * page_size + splits,
                                lc_max=1000)
    dev = DeviceWorkload(inp)
    kp, table, ppr, P = paged_pool(inp["ctx_k"], page_size, 3, seed=page_size)
    vp, _, _, _ = paged_pool(inp["ctx_v"], page_size, 3, seed=page_size)
    pages = gr.CtxPages(page_size, P, ppr)
    kp_d, vp_d, tb_d = to_dev(kp), to_dev(vp), to_dev(table)
    os.environ["GR_ATTN_FORCE_SPLITS"] = str(splits)
    try:
        for step in range(3):
            out, lse = dev.outputs(step)
            ws = torch.empty(max(16, gr.gr_decode_attn_workspace_size(dev.shape, dev.widths, step)),
                             dtype=torch.uint8, device="cuda")
            gr.gr_decode_attn_paged(dev.shape, pages, dev.q[step], kp_d, vp_d, dev.ctx_len, tb_d, dev.beam_k,
                                    dev.beam_v, dev.beam_path, dev.widths, step, out, lse, ws)
            torch.cuda.synchronize()
            ref_out, ref_lse, _ = ORC.decode_attn(inp, step)
            got = (out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
            compare(got.reshape(ref_out.shape), lse.cpu().numpy().reshape(ref_lse.shape), ref_out, ref_lse)
    finally:
        os.environ.pop("GR_ATTN_FORCE_SPLITS", None)
    assert gr.gr_get_device_error() == 0


def test_paged_rejects_bad_descriptors():
    inp = workloads.make_custom(1, 4, 2, 64, [200], [2, 2], seed=3)
    dev = DeviceWorkload(inp)
    out, lse = dev.outputs(1)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    table = to_dev(np.zeros((1, 2), np.int32))
    for bad in (gr.CtxPages(100, 4, 2), gr.CtxPages(128, 0, 2), gr.CtxPages(128, 4, 1)):
        with pytest.raises(gr.GRError) as e:
            gr.gr_decode_attn_paged(dev.shape, bad, dev.q[1], dev.ctx_k, dev.ctx_v, dev.ctx_len, table,
                                    dev.beam_k, dev.beam_v, dev.beam_path, dev.widths, 1, out, lse, ws)
        assert e.value.status == -2
