"""Python binding of libgrattn.so: large-beam decode attention on GB300.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/gr_attn.h``.  PyTorch provides
device memory and streams.  There is no CPU fallback: if the library is
missing or the device is not an sm_103 GPU, the calls raise.

The functions mirror the C entry points:

* :func:`gr_decode_attn` -- the whole decode attention (shared context stage
  on tensor cores, per-beam stage along BeamPath, log-sum-exp merge);
* :func:`gr_decode_attn_workspace_size`;
* :func:`gr_resolve_ancestors` / :func:`gr_validate_beam_path` -- BeamPath
  utilities;
* :func:`gr_beam_select` / :func:`gr_beam_select_workspace_size` -- beam
  selection after a decode forward (log_softmax + top-W over every beam's
  logits, giving the next BeamPath row);
* :func:`gr_get_device_error`, :func:`gr_status_string`.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from . import build as _build

__all__ = [
    "GRError", "Shape", "load", "lib_path", "gr_decode_attn", "gr_decode_attn_workspace_size",
    "gr_resolve_ancestors", "gr_validate_beam_path", "gr_get_device_error", "gr_status_string",
    "gr_version", "EXPORTED_SYMBOLS", "gr_decode_attn_timed", "gr_decode_attn_plan", "PlanInfo",
    "gr_decode_attn_noalloc", "NOALLOC_SCRATCH_BYTES", "SelectShape", "gr_beam_select",
    "gr_beam_select_workspace_size", "SELECT_MAX_WIDTH", "gr_beam_select_timed",
    "TrieSelectShape", "gr_trie_select", "gr_trie_select_workspace_size", "CtxPages",
    "gr_decode_attn_paged", "gr_beam_reorder", "gr_decode_attn_ragged",
    "gr_beam_reorder_inplace", "gr_beam_append",
]

EXPORTED_SYMBOLS = (
    "gr_decode_attn_workspace_size", "gr_decode_attn", "gr_decode_attn_timed",
    "gr_decode_attn_plan", "gr_resolve_ancestors", "gr_validate_beam_path",
    "gr_get_device_error", "gr_status_string", "gr_version", "gr_decode_attn_noalloc",
    "gr_beam_select_workspace_size", "gr_beam_select", "gr_beam_select_timed",
    "gr_trie_select_workspace_size", "gr_trie_select", "gr_decode_attn_paged", "gr_beam_reorder",
    "gr_decode_attn_ragged", "gr_beam_reorder_inplace", "gr_beam_append",
)

# GR_SELECT_MAX_WIDTH: the largest next_width gr_beam_select takes
SELECT_MAX_WIDTH = 1024

# bytes of the library's static scratch used by gr_decode_attn_noalloc
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024

GR_OK = 0
STATUS_NAMES = {
    0: "GR_OK", -1: "GR_ERR_NULL_ARG", -2: "GR_ERR_BAD_SHAPE", -3: "GR_ERR_UNSUPPORTED",
    -4: "GR_ERR_MISALIGNED", -5: "GR_ERR_WORKSPACE_TOO_SMALL", -6: "GR_ERR_CUDA",
    -7: "GR_ERR_DEVICE_TIMEOUT", -8: "GR_ERR_BAD_BEAM_PATH",
}


class GRError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({gr_status_string(status)})")


class Shape(ctypes.Structure):
    """``gr_attn_shape``."""
    _fields_ = [
        ("num_requests", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("ctx_capacity", ctypes.c_int32),
        ("step_capacity", ctypes.c_int32),
        ("beam_capacity", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
    ]

    @classmethod
    def of(cls, d) -> "Shape":
        return cls(int(d["num_requests"]), int(d["num_q_heads"]), int(d["num_kv_heads"]),
                   int(d["head_dim"]), int(d["ctx_capacity"]), int(d["step_capacity"]),
                   int(d["beam_capacity"]), float(d["softmax_scale"]))


class SelectShape(ctypes.Structure):
    """``gr_select_shape``."""
    _fields_ = [
        ("num_requests", ctypes.c_int32),
        ("width", ctypes.c_int32),
        ("vocab", ctypes.c_int32),
        ("next_width", ctypes.c_int32),
    ]


class TrieSelectShape(ctypes.Structure):
    """``gr_trie_select_shape``."""
    _fields_ = [
        ("num_requests", ctypes.c_int32),
        ("width", ctypes.c_int32),
        ("vocab", ctypes.c_int32),
        ("next_width", ctypes.c_int32),
        ("num_nodes", ctypes.c_int32),
        ("num_edges", ctypes.c_int32),
    ]


class CtxPages(ctypes.Structure):
    """``gr_ctx_pages``."""
    _fields_ = [
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("pages_per_request", ctypes.c_int32),
    ]


class PlanInfo(ctypes.Structure):
    """``gr_plan_info``."""
    _fields_ = [
        ("path", ctypes.c_int32),
        ("n_splits", ctypes.c_int32),
        ("split_len", ctypes.c_int32),
        ("context_ctas", ctypes.c_int32),
        ("kernels", ctypes.c_int32),
        ("fused_merge", ctypes.c_int32),
        ("persistent", ctypes.c_int32),
    ]

    def as_dict(self):
        return {f: int(getattr(self, f)) for f, _ in self._fields_}


_LIB: Optional[ctypes.CDLL] = None


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libgrattn.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    sp = ctypes.POINTER(Shape)
    lib.gr_decode_attn_workspace_size.argtypes = [sp, vp, i32]
    lib.gr_decode_attn_workspace_size.restype = sz
    lib.gr_decode_attn.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
    lib.gr_decode_attn.restype = ctypes.c_int
    lib.gr_decode_attn_timed.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz,
                                         vp, vp]
    lib.gr_decode_attn_timed.restype = ctypes.c_int
    lib.gr_decode_attn_paged.argtypes = [sp, ctypes.POINTER(CtxPages), vp, vp, vp, vp, vp, vp, vp, vp,
                                         vp, i32, vp, vp, vp, sz, vp]
    lib.gr_decode_attn_paged.restype = ctypes.c_int
    lib.gr_decode_attn_plan.argtypes = [sp, vp, i32, ctypes.POINTER(PlanInfo)]
    lib.gr_decode_attn_plan.restype = ctypes.c_int
    lib.gr_decode_attn_noalloc.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp]
    lib.gr_decode_attn_noalloc.restype = ctypes.c_int
    lib.gr_resolve_ancestors.argtypes = [sp, vp, vp, i32, vp, vp]
    lib.gr_resolve_ancestors.restype = ctypes.c_int
    lib.gr_validate_beam_path.argtypes = [sp, vp, vp, i32, vp, vp, vp]
    lib.gr_validate_beam_path.restype = ctypes.c_int
    ssp = ctypes.POINTER(SelectShape)
    lib.gr_beam_select_workspace_size.argtypes = [ssp]
    lib.gr_beam_select_workspace_size.restype = sz
    lib.gr_beam_select.argtypes = [ssp, vp, vp, vp, ctypes.c_int64, vp, vp, vp, sz, vp]
    lib.gr_beam_select.restype = ctypes.c_int
    lib.gr_beam_select_timed.argtypes = [ssp, vp, vp, vp, ctypes.c_int64, vp, vp, vp, sz, vp, vp]
    lib.gr_beam_select_timed.restype = ctypes.c_int
    tsp = ctypes.POINTER(TrieSelectShape)
    lib.gr_trie_select_workspace_size.argtypes = [tsp]
    lib.gr_trie_select_workspace_size.restype = sz
    lib.gr_trie_select.argtypes = [tsp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int64, vp, vp, vp, vp, sz, vp]
    lib.gr_trie_select.restype = ctypes.c_int
    lib.gr_decode_attn_ragged.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
    lib.gr_decode_attn_ragged.restype = ctypes.c_int
    lib.gr_beam_reorder.argtypes = [sp, vp, vp, vp, vp, i32, vp, vp, vp, vp]
    lib.gr_beam_reorder.restype = ctypes.c_int
    lib.gr_beam_reorder_inplace.argtypes = [sp, vp, vp, vp, vp, i32, vp]
    lib.gr_beam_reorder_inplace.restype = ctypes.c_int
    lib.gr_beam_append.argtypes = [sp, vp, i32, vp, vp, ctypes.c_int64, vp, vp, vp]
    lib.gr_beam_append.restype = ctypes.c_int
    lib.gr_get_device_error.argtypes = []
    lib.gr_get_device_error.restype = ctypes.c_int
    lib.gr_status_string.argtypes = [ctypes.c_int]
    lib.gr_status_string.restype = ctypes.c_char_p
    lib.gr_version.argtypes = []
    lib.gr_version.restype = ctypes.c_int
    _LIB = lib
    return lib


def _widths_arr(widths: Sequence[int], step: int):
    """The per-step widths as a C array; the library reads widths[0..step]."""
    if int(step) >= 0 and len(widths) < int(step) + 1:
        raise ValueError("widths needs an entry for every step 0..step")
    arr = (ctypes.c_int32 * max(1, len(widths)))(*[int(w) for w in widths])
    return arr


def _ptr(t) -> Optional[int]:
    """Device/host address of a tensor (None stays NULL)."""
    if t is None:
        return None
    return int(t.data_ptr())


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(rc: int, where: str):
    if rc != GR_OK:
        raise GRError(rc, where)


def gr_status_string(status: int) -> str:
    return load().gr_status_string(int(status)).decode()


def gr_version() -> int:
    return int(load().gr_version())


def gr_decode_attn_workspace_size(shape: Shape, widths: Sequence[int], step: int) -> int:
    w = _widths_arr(widths, step)
    return int(load().gr_decode_attn_workspace_size(ctypes.byref(shape), w, int(step)))


def gr_decode_attn(shape: Shape, q, ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path,
                   widths: Sequence[int], step: int, out, lse, workspace=None,
                   workspace_bytes: Optional[int] = None, stream=None) -> None:
    """Enqueue gr_decode_attn on ``stream`` (default: torch's current stream).

    Tensors are torch CUDA tensors laid out as ``include/gr_attn.h`` states
    (bf16 tensors may be ``torch.bfloat16`` or ``int16`` bit patterns).
    Raises :class:`GRError` on a non-zero status.
    """
    w = _widths_arr(widths, step)
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().gr_decode_attn(ctypes.byref(shape), _ptr(q), _ptr(ctx_k), _ptr(ctx_v),
                               _ptr(ctx_len), _ptr(beam_k), _ptr(beam_v), _ptr(beam_path), w,
                               int(step), _ptr(out), _ptr(lse), _ptr(workspace),
                               int(workspace_bytes), _stream_handle(stream))
    _check(rc, "gr_decode_attn")


def gr_decode_attn_paged(shape: Shape, pages: CtxPages, q, ctx_k_pool, ctx_v_pool, ctx_len, block_table,
                         beam_k, beam_v, beam_path, widths: Sequence[int], step: int, out, lse,
                         workspace=None, workspace_bytes: Optional[int] = None, stream=None) -> None:
    """gr_decode_attn over a paged ContextKV pool (see ``include/gr_attn.h``)."""
    w = _widths_arr(widths, step)
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().gr_decode_attn_paged(ctypes.byref(shape), ctypes.byref(pages), _ptr(q), _ptr(ctx_k_pool),
                                     _ptr(ctx_v_pool), _ptr(ctx_len), _ptr(block_table), _ptr(beam_k),
                                     _ptr(beam_v), _ptr(beam_path), w, int(step), _ptr(out), _ptr(lse),
                                     _ptr(workspace), int(workspace_bytes), _stream_handle(stream))
    _check(rc, "gr_decode_attn_paged")


def gr_decode_attn_timed(shape: Shape, q, ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path,
                         widths: Sequence[int], step: int, out, lse, workspace, events,
                         workspace_bytes: Optional[int] = None, stream=None) -> None:
    """gr_decode_attn recording ``events`` (3 ``torch.cuda.Event(enable_timing=True)``;
    the middle one may be None, and is then not recorded) before the context
    kernel, after it, and after the last kernel."""
    w = _widths_arr(widths, step)
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if len(events) != 3:
        raise ValueError("events: three torch.cuda.Event or None")
    for e in events:
        if e is not None and e.cuda_event == 0:      # torch creates the event lazily on first record
            e.record()
    ev = (ctypes.c_void_p * 3)(*[0 if e is None else int(e.cuda_event) for e in events])
    rc = load().gr_decode_attn_timed(ctypes.byref(shape), _ptr(q), _ptr(ctx_k), _ptr(ctx_v),
                                     _ptr(ctx_len), _ptr(beam_k), _ptr(beam_v), _ptr(beam_path), w,
                                     int(step), _ptr(out), _ptr(lse), _ptr(workspace),
                                     int(workspace_bytes), _stream_handle(stream), ev)
    _check(rc, "gr_decode_attn_timed")


def gr_decode_attn_noalloc(shape: Shape, q, ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path,
                           widths: Sequence[int], step: int, out, lse, stream=None) -> None:
    """gr_decode_attn without a caller-supplied workspace: for callers that
    cannot allocate device memory, the library uses its own static 64 MiB
    device scratch (shared by all calls; calls that overlap on the GPU race).
    Raises :class:`GRError` (GR_ERR_WORKSPACE_TOO_SMALL) when the call needs
    more scratch than that."""
    rc = load().gr_decode_attn_noalloc(ctypes.byref(shape), _ptr(q), _ptr(ctx_k), _ptr(ctx_v),
                                       _ptr(ctx_len), _ptr(beam_k), _ptr(beam_v), _ptr(beam_path),
                                       _widths_arr(widths, step), int(step), _ptr(out), _ptr(lse),
                                       _stream_handle(stream))
    _check(rc, "gr_decode_attn_noalloc")


def gr_decode_attn_plan(shape: Shape, widths: Sequence[int], step: int) -> dict:
    info = PlanInfo()
    rc = load().gr_decode_attn_plan(ctypes.byref(shape), _widths_arr(widths, step), int(step),
                                    ctypes.byref(info))
    _check(rc, "gr_decode_attn_plan")
    return info.as_dict()


def gr_resolve_ancestors(shape: Shape, beam_path, widths: Sequence[int], step: int, anc,
                         stream=None) -> None:
    rc = load().gr_resolve_ancestors(ctypes.byref(shape), _ptr(beam_path), _widths_arr(widths, step),
                                     int(step), _ptr(anc), _stream_handle(stream))
    _check(rc, "gr_resolve_ancestors")


def gr_validate_beam_path(shape: Shape, beam_path, widths: Sequence[int], step: int, ctx_len,
                          bad_count, stream=None) -> None:
    rc = load().gr_validate_beam_path(ctypes.byref(shape), _ptr(beam_path), _widths_arr(widths, step),
                                      int(step), _ptr(ctx_len), _ptr(bad_count),
                                      _stream_handle(stream))
    _check(rc, "gr_validate_beam_path")


def gr_beam_select_workspace_size(shape: SelectShape) -> int:
    return int(load().gr_beam_select_workspace_size(ctypes.byref(shape)))


def gr_beam_select(shape: SelectShape, logits, beam_scores, next_parent, next_token, next_score,
                   workspace, parent_stride: Optional[int] = None,
                   workspace_bytes: Optional[int] = None, stream=None) -> None:
    """Enqueue gr_beam_select on ``stream`` (default: torch's current stream).

    ``logits`` fp32 [R, W_s, V], ``beam_scores`` fp32 [R, W_s]; writes
    ``next_parent`` (row r at r * parent_stride, default next_width),
    ``next_token`` and ``next_score`` ([R, next_width]).  Raises
    :class:`GRError` on a non-zero status.
    """
    if parent_stride is None:
        parent_stride = shape.next_width
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().gr_beam_select(ctypes.byref(shape), _ptr(logits), _ptr(beam_scores),
                               _ptr(next_parent), int(parent_stride), _ptr(next_token),
                               _ptr(next_score), _ptr(workspace), int(workspace_bytes),
                               _stream_handle(stream))
    _check(rc, "gr_beam_select")


def gr_beam_select_timed(shape: SelectShape, logits, beam_scores, next_parent, next_token,
                         next_score, workspace, events, parent_stride: Optional[int] = None,
                         workspace_bytes: Optional[int] = None, stream=None) -> None:
    """gr_beam_select recording ``events`` (3 ``torch.cuda.Event(enable_timing=True)``)
    before the per-row kernel, between the two kernels, and after the merge."""
    if parent_stride is None:
        parent_stride = shape.next_width
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    for e in events:
        if e.cuda_event == 0:      # torch creates the event lazily on first record
            e.record()
    ev = (ctypes.c_void_p * 3)(*[int(e.cuda_event) for e in events])
    rc = load().gr_beam_select_timed(ctypes.byref(shape), _ptr(logits), _ptr(beam_scores),
                                     _ptr(next_parent), int(parent_stride), _ptr(next_token),
                                     _ptr(next_score), _ptr(workspace), int(workspace_bytes),
                                     _stream_handle(stream), ev)
    _check(rc, "gr_beam_select_timed")


def gr_trie_select_workspace_size(shape: TrieSelectShape) -> int:
    return int(load().gr_trie_select_workspace_size(ctypes.byref(shape)))


def gr_trie_select(shape: TrieSelectShape, logits, beam_scores, beam_node, trie_offsets, trie_tokens,
                   trie_children, next_parent, next_token, next_score, next_node, workspace,
                   parent_stride: Optional[int] = None, workspace_bytes: Optional[int] = None,
                   stream=None) -> None:
    """Enqueue gr_trie_select (item-constrained beam selection) on ``stream``."""
    if parent_stride is None:
        parent_stride = shape.next_width
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().gr_trie_select(ctypes.byref(shape), _ptr(logits), _ptr(beam_scores), _ptr(beam_node),
                               _ptr(trie_offsets), _ptr(trie_tokens), _ptr(trie_children),
                               _ptr(next_parent), int(parent_stride), _ptr(next_token),
                               _ptr(next_score), _ptr(next_node), _ptr(workspace), int(workspace_bytes),
                               _stream_handle(stream))
    _check(rc, "gr_trie_select")


def gr_decode_attn_ragged(shape: Shape, q, ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path,
                          req_widths_host, req_widths, step: int, out, lse, workspace=None,
                          workspace_bytes: Optional[int] = None, stream=None) -> None:
    """gr_decode_attn with a width per request: ``req_widths_host`` is a
    [R][step+1] sequence, ``req_widths`` the device int32 [R, S_max] copy."""
    rows = [list(row) for row in req_widths_host]
    if len(rows) != shape.num_requests or any(len(row) < int(step) + 1 for row in rows):
        raise ValueError("req_widths_host needs num_requests rows of at least step + 1 widths")
    if req_widths is not None and hasattr(req_widths, "numel"):
        # the kernels index the device copy as a dense int32 [R, S_max]
        import torch
        if (req_widths.dtype != torch.int32 or not req_widths.is_cuda or not req_widths.is_contiguous()
                or req_widths.numel() < shape.num_requests * shape.step_capacity):
            raise ValueError("req_widths must be a contiguous device int32 tensor of "
                             "num_requests * step_capacity entries")
    flat = [int(w) for row in rows for w in row[:int(step) + 1]]
    arr = (ctypes.c_int32 * max(1, len(flat)))(*flat)
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().gr_decode_attn_ragged(ctypes.byref(shape), _ptr(q), _ptr(ctx_k), _ptr(ctx_v), _ptr(ctx_len),
                                      _ptr(beam_k), _ptr(beam_v), _ptr(beam_path), arr, _ptr(req_widths),
                                      int(step), _ptr(out), _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                      _stream_handle(stream))
    _check(rc, "gr_decode_attn_ragged")


def gr_beam_reorder(shape: Shape, beam_k, beam_v, beam_path, widths: Sequence[int], step: int,
                    out_k, out_v, out_path, stream=None) -> None:
    """The per-beam cache reordered along BeamPath (see ``include/gr_attn.h``)."""
    rc = load().gr_beam_reorder(ctypes.byref(shape), _ptr(beam_k), _ptr(beam_v), _ptr(beam_path),
                                _widths_arr(widths, step), int(step), _ptr(out_k), _ptr(out_v), _ptr(out_path),
                                _stream_handle(stream))
    _check(rc, "gr_beam_reorder")


def gr_beam_reorder_inplace(shape: Shape, beam_k, beam_v, beam_path, widths: Sequence[int], step: int,
                            stream=None) -> None:
    """The per-beam cache reordered along BeamPath in place, and the path set
    to the identity (see ``include/gr_attn.h``)."""
    rc = load().gr_beam_reorder_inplace(ctypes.byref(shape), _ptr(beam_k), _ptr(beam_v), _ptr(beam_path),
                                        _widths_arr(widths, step), int(step), _stream_handle(stream))
    _check(rc, "gr_beam_reorder_inplace")


def gr_beam_append(shape: Shape, widths: Sequence[int], step: int, k_new, v_new, beam_k, beam_v,
                   src_stride: Optional[int] = None, stream=None) -> None:
    """BeamKV append of the step's new K/V rows (see ``include/gr_attn.h``).
    ``src_stride`` (elements between beams' rows) defaults to Hkv * D."""
    stride = shape.num_kv_heads * shape.head_dim if src_stride is None else int(src_stride)
    rc = load().gr_beam_append(ctypes.byref(shape), _widths_arr(widths, step), int(step), _ptr(k_new),
                               _ptr(v_new), stride, _ptr(beam_k), _ptr(beam_v), _stream_handle(stream))
    _check(rc, "gr_beam_append")


def gr_get_device_error() -> int:
    return int(load().gr_get_device_error())
