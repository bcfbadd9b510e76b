"""CPU oracle for large-beam decode attention (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it
and shares no code with it.

Two independent implementations live here:

* ``gr_oracle.c`` -- the fp64 oracle proper (C, OpenMP over rows), built
  with gcc into ``oracle/_build/liboracle*.so`` and called through ctypes.
* :mod:`oracle.brute` -- a short numpy brute force for tiny inputs, written
  separately so the two can pin each other.

Both follow the definition of the three-stage attention (shared context,
per-beam chain reached through BeamPath, log-sum-exp merge) from the
GR-Inference blog ("system design" and "kernel design" sections) and the
xGR review ("xAttention", three-stage computation).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gr_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: Dict[int, ctypes.CDLL] = {}

# planted mistakes (compile-time ORACLE_MUTANT); 0 is the oracle itself
MUTANTS = {
    1: "drops the per-beam stage",
    2: "reads parents from the wrong BeamPath step row",
    3: "interleaved GQA head grouping",
    4: "softmax scale left out",
    5: "ignores BeamPath (keeps the beam's own slot)",
    6: "base-2 log in the LSE",
    7: "unnormalised output weights",
    8: "leaves out the current step's token",
}


def lib_path(mutant: int = 0) -> str:
    return os.path.join(_BUILD, "liboracle.so" if mutant == 0 else f"liboracle_m{mutant}.so")


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2 -fopenmp, no fast-math)."""
    path = lib_path(mutant)
    if not force and os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(_SRC):
        return path
    os.makedirs(_BUILD, exist_ok=True)
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           f"-DORACLE_MUTANT={mutant}", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def _load(mutant: int = 0) -> ctypes.CDLL:
    with _LOCK:
        if mutant in _LIBS:
            return _LIBS[mutant]
        lib = ctypes.CDLL(build(mutant))
        i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        vp = ctypes.c_void_p
        lib.oracle_decode_attn.restype = ctypes.c_int
        lib.oracle_decode_attn.argtypes = [i32, i32, i32, i32, i32, i32, i32, f32,
                                           vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                           vp, vp, i64, i32, i32, i32, vp, vp, vp, i32]
        lib.oracle_ancestors.restype = ctypes.c_int
        lib.oracle_ancestors.argtypes = [i32, i32, i32, vp, vp, i32, vp, vp, i64, vp]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_mutant_id.restype = ctypes.c_int
        _LIBS[mutant] = lib
        return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _selection(inp, step, rows):
    W_s = int(inp["widths"][step])
    if rows is None:
        rr, bb = np.meshgrid(np.arange(inp["num_requests"], dtype=np.int32),
                             np.arange(W_s, dtype=np.int32), indexing="ij")
        return rr.reshape(-1).copy(), bb.reshape(-1).copy()
    rows = np.asarray(rows, dtype=np.int32).reshape(-1, 2)
    return rows[:, 0].copy(), rows[:, 1].copy()


class Oracle:
    """ctypes front end of the C oracle (or of one planted-mistake variant)."""

    def __init__(self, mutant: int = 0):
        self.mutant = mutant
        self._lib = _load(mutant)

    @property
    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())

    def ancestors(self, inp, step: int, rows=None) -> np.ndarray:
        """Ancestor slots a_0..a_s for each selected (r, b): int32 [n, s+1].

        With ``rows=None`` all (r, b < W_s) rows are returned as [R, W_s, s+1].
        """
        sel_r, sel_b = _selection(inp, step, rows)
        bp = _c(inp["beam_path"], np.int32)
        widths = _c(inp["widths"], np.int32)
        anc = np.empty((len(sel_r), step + 1), dtype=np.int32)
        rc = self._lib.oracle_ancestors(inp["num_requests"], inp["step_capacity"],
                                        inp["beam_capacity"], _ptr(bp), _ptr(widths), step,
                                        _ptr(sel_r), _ptr(sel_b), len(sel_r), _ptr(anc))
        if rc != 0:
            raise ValueError(f"oracle_ancestors failed with status {rc}")
        if rows is None:
            return anc.reshape(inp["num_requests"], int(inp["widths"][step]), step + 1)
        return anc

    def decode_attn(self, inp, step: int, rows=None, ctx_range: Tuple[int, int] = (0, -1),
                    include_beam: bool = True, q=None, num_threads: int = 0):
        """fp64 attention for the selected rows.

        Returns ``(out, lse, anc)``: ``out`` f64 [n, Hq, D] (or
        [R, W_s, Hq, D] when ``rows`` is None), ``lse`` f64 [n, Hq], ``anc``
        int32 [n, s+1].  ``ctx_range=(lo, hi)`` restricts the context keys to
        positions [lo, hi) (hi < 0: the full context) and ``include_beam``
        keeps or drops the per-beam chain; both exist to state the merge
        identity in the tests.
        """
        R, Hq, Hkv, D = (inp["num_requests"], inp["num_q_heads"], inp["num_kv_heads"],
                         inp["head_dim"])
        sel_r, sel_b = _selection(inp, step, rows)
        n = len(sel_r)
        qs = _c(inp["q"][step] if q is None else q, np.uint16)
        ck = _c(inp["ctx_k"], np.uint16)
        cv = _c(inp["ctx_v"], np.uint16)
        bk = _c(inp["beam_k"], np.uint16)
        bv = _c(inp["beam_v"], np.uint16)
        bp = _c(inp["beam_path"], np.int32)
        cl = _c(inp["ctx_len"], np.int32)
        widths = _c(inp["widths"], np.int32)
        out = np.empty((n, Hq, D), dtype=np.float64)
        lse = np.empty((n, Hq), dtype=np.float64)
        anc = np.empty((n, step + 1), dtype=np.int32)
        rc = self._lib.oracle_decode_attn(
            R, Hq, Hkv, D, inp["ctx_capacity"], inp["step_capacity"], inp["beam_capacity"],
            ctypes.c_float(inp["softmax_scale"]),
            _ptr(qs), _ptr(ck), _ptr(cv), _ptr(cl), _ptr(bk), _ptr(bv), _ptr(bp), _ptr(widths),
            step, _ptr(sel_r), _ptr(sel_b), n, int(ctx_range[0]), int(ctx_range[1]),
            1 if include_beam else 0, _ptr(out), _ptr(lse), _ptr(anc), int(num_threads))
        if rc != 0:
            raise ValueError(f"oracle_decode_attn failed with status {rc}")
        if rows is None:
            W_s = int(inp["widths"][step])
            return (out.reshape(R, W_s, Hq, D), lse.reshape(R, W_s, Hq),
                    anc.reshape(R, W_s, step + 1))
        return out, lse, anc


def oracle(mutant: int = 0) -> Oracle:
    return Oracle(mutant)
