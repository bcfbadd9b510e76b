"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/gr_attn.h declares, and rejects bad arguments before
touching a device."""

import ctypes
import os
import re

import pytest

import beam_decode_attention_gb300 as gr
from beam_decode_attention_gb300 import build as gr_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gr_build.build()
    return gr.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gr_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gr_[a-z_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert "gr_decode_attn" in names and "gr_resolve_ancestors" in names
    assert set(names) == set(gr.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    assert gr.gr_status_string(0) == "ok"
    for code in range(-8, 0):
        assert gr.gr_status_string(code) != "unknown status"
    assert gr.gr_status_string(-99) == "unknown status"
    assert gr.gr_version() >= 100


def _shape(**kw):
    d = dict(num_requests=2, num_q_heads=16, num_kv_heads=8, head_dim=128, ctx_capacity=64,
             step_capacity=3, beam_capacity=8, softmax_scale=0.088388)
    d.update(kw)
    return gr.Shape.of(d)


FAKE = 1 << 20   # a 16-byte-aligned address that is never dereferenced


def _call(shape, widths=(4, 4, 4), step=2, **ptrs):
    lib = gr.load()
    p = dict(q=FAKE, ck=FAKE, cv=FAKE, cl=FAKE, bk=FAKE, bv=FAKE, bp=FAKE, out=FAKE, lse=FAKE, ws=FAKE)
    p.update(ptrs)
    w = (ctypes.c_int32 * len(widths))(*widths)
    return lib.gr_decode_attn(ctypes.byref(shape), p["q"], p["ck"], p["cv"], p["cl"], p["bk"],
                              p["bv"], p["bp"], w, step, p["out"], p["lse"], p["ws"], 1 << 30, 0)


@pytest.mark.parametrize("kw,code", [
    (dict(num_requests=0), -2),
    (dict(num_q_heads=12, num_kv_heads=8), -2),
    (dict(head_dim=96), -3),
    (dict(num_q_heads=256, num_kv_heads=1), -3),
    (dict(step_capacity=0), -2),
    (dict(beam_capacity=0), -2),
    (dict(ctx_capacity=-1), -2),
    (dict(softmax_scale=float("nan")), -2),
])
def test_bad_shapes_rejected(lib, kw, code):
    assert _call(_shape(**kw)) == code


def test_bad_step_and_widths_rejected(lib):
    assert _call(_shape(), step=3) == -2
    assert _call(_shape(), step=-1) == -2
    assert _call(_shape(), widths=(4, 9, 4)) == -2       # > beam_capacity
    assert _call(_shape(), widths=(4, 0, 4)) == -2


def test_null_and_misaligned_pointers_rejected(lib):
    assert _call(_shape(), q=None) == -1
    assert _call(_shape(), out=None) == -1
    assert _call(_shape(), bp=None) == -1
    assert _call(_shape(), ck=None) == -1
    assert _call(_shape(), q=FAKE + 8) == -4
    assert _call(_shape(), lse=FAKE + 4) == -4
    assert _call(_shape(), ws=FAKE + 2) == -4


def test_workspace_size_zero_on_bad_args(lib):
    w = (ctypes.c_int32 * 3)(4, 4, 4)
    assert lib.gr_decode_attn_workspace_size(ctypes.byref(_shape(head_dim=80)), w, 2) == 0
    assert lib.gr_decode_attn_workspace_size(None, w, 2) == 0
    assert lib.gr_decode_attn_workspace_size(ctypes.byref(_shape()), w, 5) == 0


def test_utilities_reject_bad_args(lib):
    w = (ctypes.c_int32 * 3)(4, 4, 4)
    assert lib.gr_resolve_ancestors(ctypes.byref(_shape()), None, w, 2, FAKE, 0) == -1
    assert lib.gr_resolve_ancestors(ctypes.byref(_shape()), FAKE, w, 7, FAKE, 0) == -2
    assert lib.gr_validate_beam_path(ctypes.byref(_shape()), FAKE, w, 2, None, FAKE, 0) == -1


def _sel(**kw):
    d = dict(num_requests=2, width=4, vocab=100, next_width=8)
    d.update(kw)
    return gr.SelectShape(d["num_requests"], d["width"], d["vocab"], d["next_width"])


def _sel_bytes(R, W, V, n):
    # per beam row a sorted list of min(n, V) 8-byte entries and its length;
    # per request a 4-byte bound and 32 4-byte bound slots (padded to 16 bytes)
    return R * W * min(n, V) * 8 + (R * 33 * 4 + 15) // 16 * 16 + R * W * 4


def test_beam_select_workspace_size(lib):
    assert lib.gr_beam_select_workspace_size(ctypes.byref(_sel())) == _sel_bytes(2, 4, 100, 8)
    assert lib.gr_beam_select_workspace_size(ctypes.byref(_sel(vocab=3, next_width=10))) == _sel_bytes(2, 4, 3, 10)
    for bad in (dict(num_requests=0), dict(width=0), dict(vocab=0), dict(next_width=0),
                dict(next_width=1025, vocab=1000), dict(width=2, vocab=3, next_width=7),
                dict(width=1 << 16, vocab=1 << 15), dict(width=4097, vocab=10)):
        assert lib.gr_beam_select_workspace_size(ctypes.byref(_sel(**bad))) == 0, bad
    assert lib.gr_beam_select_workspace_size(None) == 0


def test_beam_select_rejects_bad_args(lib):
    ok = ctypes.byref(_sel())

    def call(shape=ok, logits=FAKE, scores=FAKE, parent=FAKE, stride=8, token=FAKE, score=FAKE,
             ws=FAKE, ws_bytes=1 << 20):
        return lib.gr_beam_select(shape, logits, scores, parent, stride, token, score, ws, ws_bytes, None)

    assert call(shape=None) == -1
    assert call(logits=None) == -1
    assert call(parent=None) == -1
    assert call(ws=None) == -1
    assert call(shape=ctypes.byref(_sel(next_width=0))) == -2
    assert call(stride=7) == -2
    assert call(logits=FAKE + 4) == -4
    assert call(token=FAKE + 8) == -4
    assert call(ws_bytes=_sel_bytes(2, 4, 100, 8) - 1) == -5


def _tsel(**kw):
    d = dict(num_requests=2, width=4, vocab=100, next_width=8, num_nodes=10, num_edges=9)
    d.update(kw)
    return gr.TrieSelectShape(*[d[k] for k in ("num_requests", "width", "vocab", "next_width",
                                                  "num_nodes", "num_edges")])


def test_trie_select_workspace_and_bad_args(lib):
    # per beam row a list of next_width 8-byte entries, its length and a slot in the list of
    # rows too wide for one warp; a bound per request and that list's count (16-byte padded)
    assert lib.gr_trie_select_workspace_size(ctypes.byref(_tsel())) == 2 * 4 * 8 * 8 + 16 + 2 * (2 * 4 * 4)
    for bad in (dict(num_nodes=0), dict(num_edges=-1), dict(next_width=1025), dict(width=4097)):
        assert lib.gr_trie_select_workspace_size(ctypes.byref(_tsel(**bad))) == 0, bad

    def call(shape=ctypes.byref(_tsel()), toks=FAKE, node_out=FAKE, stride=8, ws_bytes=1 << 20, logits=FAKE):
        return lib.gr_trie_select(shape, logits, FAKE, FAKE, FAKE, toks, FAKE, FAKE, stride, FAKE, FAKE,
                                  node_out, FAKE, ws_bytes, None)

    assert call(shape=None) == -1
    assert call(toks=None) == -1
    assert call(node_out=None) == -1
    assert call(stride=7) == -2
    assert call(logits=FAKE + 4) == -4
    assert call(ws_bytes=10) == -5


def test_paged_and_reorder_reject_bad_args(lib):
    w = (ctypes.c_int32 * 3)(4, 4, 4)
    sh = ctypes.byref(_shape())

    def paged(pages, table=FAKE):
        return lib.gr_decode_attn_paged(sh, pages, FAKE, FAKE, FAKE, FAKE, table, FAKE, FAKE, FAKE, w, 2,
                                        FAKE, FAKE, FAKE, 1 << 20, None)

    assert paged(None) == -1
    assert paged(ctypes.byref(gr.CtxPages(100, 4, 1))) == -2      # not a multiple of 128
    assert paged(ctypes.byref(gr.CtxPages(128, 0, 1))) == -2      # no pages
    assert paged(ctypes.byref(gr.CtxPages(128, 4, 0))) == -2      # empty block-table rows
    assert paged(ctypes.byref(gr.CtxPages(128, 4, 1)), table=None) == -1
    assert paged(ctypes.byref(gr.CtxPages(128, 4, 1)), table=FAKE + 4) == -4

    # beam_k/beam_v of this shape are 2*3*8*8*128*2 = 98,304 bytes, beam_path 192 bytes:
    # the fake buffers below sit 1 MiB apart, so only the ones a case moves overlap
    MB = 1 << 20
    bk0, bv0, bp0, ok0, ov0, op0 = (FAKE + i * MB for i in range(6))

    def reorder(bk=bk0, out_k=ok0, out_v=ov0, out_path=op0):
        return lib.gr_beam_reorder(sh, bk, bv0, bp0, w, 2, out_k, out_v, out_path, None)

    assert reorder(bk=None) == -1
    assert reorder(out_path=op0 + 8) == -4
    assert reorder(out_k=bk0) == -2                               # in place
    assert reorder(out_path=bp0) == -2                            # the path in place
    assert reorder(out_v=bk0 + 98304 - 16) == -2                  # overlaps the end of beam_k
    assert reorder(out_k=bv0 - 98304 + 16) == -2                  # overlaps the start of beam_v
    assert reorder(out_path=bk0 + 4096) == -2                     # inside beam_k
    assert reorder(out_v=bk0 + 98304) not in (-1, -2, -4)         # adjacent, not overlapping: passes the checks


def test_inplace_reorder_and_append_reject_bad_args(lib):
    w = (ctypes.c_int32 * 3)(4, 4, 4)
    sh = ctypes.byref(_shape())
    MB = 1 << 20
    kv = 98304                                  # bytes of beam_k / beam_v for this shape
    bk0, bv0, bp0, kn0, vn0 = (FAKE + i * MB for i in range(5))

    def inplace(bk=bk0, bv=bv0, bp=bp0, step=2, shape=sh, widths=w):
        return lib.gr_beam_reorder_inplace(shape, bk, bv, bp, widths, step, None)

    assert inplace(bp=None) == -1
    assert inplace(bv=bv0 + 8) == -4
    assert inplace(step=3) == -2                                  # step outside [0, S_max)
    assert inplace(bv=bk0) == -2                                  # K and V the same buffer
    assert inplace(bv=bk0 + kv - 16) == -2                        # V overlaps the end of K
    assert inplace(bp=bv0 + 4096) == -2                           # the path inside V
    assert inplace(bv=bk0 + kv) not in (-1, -2, -3, -4)           # adjacent: passes the checks
    wide = (ctypes.c_int32 * 3)(15000, 15000, 15000)
    big = ctypes.byref(_shape(beam_capacity=15000))
    assert inplace(shape=big, widths=wide, bv=bk0 + 512 * MB, bp=bk0 + 1024 * MB) == -3   # a 15,000-slot
    # level cannot be staged

    row = 8 * 128                               # Hkv * D

    def append(kn=kn0, vn=vn0, stride=row, bk=bk0, bv=bv0, step=1):
        return lib.gr_beam_append(sh, w, step, kn, vn, stride, bk, bv, None)

    assert append(kn=None) == -1
    assert append(bv=None) == -1
    assert append(stride=row - 8) == -2                           # rows overlap each other
    assert append(stride=row + 4) == -4                           # rows not on 16-byte boundaries
    assert append(vn=vn0 + 2) == -4
    assert append(step=-1) == -2
    assert append(kn=bk0 + 16) == -2                              # source inside the destination
    assert append(vn=bv0 - 2 * 4 * row * 2 + 16) == -2            # source running into beam_v
    assert append(bv=bk0) == -2
    assert append(stride=3 * row) not in (-1, -2, -3, -4)         # a fused-QKV row stride passes


def test_ragged_rejects_bad_args(lib):
    sh = ctypes.byref(_shape())

    def ragged(host_w, dev_w=FAKE, step=2):
        arr = None if host_w is None else (ctypes.c_int32 * len(host_w))(*host_w)
        return lib.gr_decode_attn_ragged(sh, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, arr, dev_w, step,
                                         FAKE, FAKE, FAKE, 1 << 20, None)

    assert ragged(None) == -1
    assert ragged([4, 4, 4, 2, 2, 2], dev_w=None) == -1
    assert ragged([4, 4, 4, 2, 0, 2]) == -2                       # a width below 1
    assert ragged([4, 4, 9, 2, 2, 2]) == -2                       # a width above beam_capacity
    assert ragged([4, 4, 4, 2, 2, 2], step=3) == -2               # step past step_capacity
    assert ragged([4, 4, 4, 2, 2, 2], dev_w=FAKE + 2) == -4       # misaligned device widths


def test_ragged_binding_checks_host_widths(lib):
    # the binding refuses host widths that do not cover every request and step,
    # and a device width array smaller than [R, S_max] int32
    import torch
    sh = _shape()
    for bad in ([[4, 4, 4]], [[4, 4], [2, 2]]):
        with pytest.raises(ValueError):
            gr.gr_decode_attn_ragged(sh, None, None, None, None, None, None, None, bad, None, 2, None, None)
    for dev in (torch.zeros(2 * 2, dtype=torch.int32), torch.zeros(2 * 3, dtype=torch.int16),
                torch.zeros(2 * 3, dtype=torch.float32), torch.zeros(2 * 3, dtype=torch.int32),
                torch.zeros(2 * 6, dtype=torch.int32)[::2]):
        # too small, int16, float32, on the host, not contiguous
        with pytest.raises(ValueError):
            gr.gr_decode_attn_ragged(sh, None, None, None, None, None, None, None, [[4, 4, 4], [2, 2, 2]], dev, 2,
                                     None, None)


def test_binding_checks_widths_cover_the_step(lib):
    with pytest.raises(ValueError):
        gr.gr_decode_attn_workspace_size(_shape(), [4, 4], 2)    # widths for steps 0 and 1 only
    with pytest.raises(ValueError):
        gr.gr_decode_attn_plan(_shape(), [4], 1)


def _noalloc(shape, widths=(4, 4, 4), step=2, **ptrs):
    lib = gr.load()
    p = dict(q=FAKE, ck=FAKE, cv=FAKE, cl=FAKE, bk=FAKE, bv=FAKE, bp=FAKE, out=FAKE, lse=FAKE)
    p.update(ptrs)
    w = (ctypes.c_int32 * len(widths))(*widths)
    return lib.gr_decode_attn_noalloc(ctypes.byref(shape), p["q"], p["ck"], p["cv"], p["cl"], p["bk"],
                                      p["bv"], p["bp"], w, step, p["out"], p["lse"], 0)


def test_noalloc_reports_the_same_errors_in_the_same_order(lib):
    """gr_decode_attn_noalloc runs gr_decode_attn's checks, in its order,
    before it looks up its static scratch: shape, NULL and alignment errors
    come back as gr_decode_attn reports them, and with every argument valid
    the first failure is the device check (no GPU here), as for
    gr_decode_attn."""
    cases = [
        (dict(), dict()),
        (dict(), dict(q=None)),
        (dict(), dict(lse=None)),
        (dict(), dict(out=FAKE + 2)),
        (dict(), dict(bp=FAKE + 4)),
        (dict(), dict(q=None, out=FAKE + 2)),
        (dict(head_dim=96), dict()),
        (dict(head_dim=96), dict(q=None)),
        (dict(num_q_heads=12), dict(q=None)),
        (dict(step=5), dict()),
    ]
    for shape_kw, ptrs in cases:
        step = shape_kw.pop("step", 2)
        sh = _shape(**shape_kw)
        want = _call(sh, step=step, **dict(ptrs, ws=FAKE))
        got = _noalloc(sh, step=step, **ptrs)
        assert got == want, (shape_kw, ptrs, got, want)
    assert _noalloc(_shape(), q=None) == -1
    assert _noalloc(_shape(), out=FAKE + 2) == -4
    assert _noalloc(_shape(), widths=(4, 0, 4)) == -2
