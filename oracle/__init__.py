"""CPU oracle of the Sparse State Expansion (SSE) layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import or run this package.  The CUDA library never calls it
and shares no code with it.

Contents
--------
* ``forward`` / ``decode_step`` / ``group``: the token-by-token float64
  recurrence of "Scaling Linear Attention with Sparse State Expansion"
  (close-reading notes, section 2.3, eqs. 9-14, plus the always-on shared
  partition of section 2.5) and the token->partition grouping of section 2.6,
  written in plain C (``sse_oracle.c``) and called through ctypes.
* ``closed_form``: the unrolled form of the same layer (section 2.4, the sum
  over s <= t and over partitions shared by t and s of e_t e_s q_t
  (prod of the selected-step decays) k_s^T v_s), brute force in numpy.
* ``dense_gla``: gated linear attention written as its quadratic masked form,
  brute force in numpy (the k = N special case of section 5.3).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against the textbook masked form, the unrolled closed form, the worked decay
example of section 2.4, the k = N special case and routing invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libsse_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``sse_oracle.c`` into ``_build/libsse_oracle.so`` (gcc, OpenMP)."""
    src = os.path.join(_HERE, "sse_oracle.c")
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(src)):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.sse_oracle_forward.restype = ctypes.c_int
    lib.sse_oracle_forward.argtypes = [i64, i32, i32, i32, i32, i32, i32, f64,
                                       P, P, P, P, P, P, P, P, i32, P, P, P, P, P, P, i64]
    lib.sse_oracle_decode_step.restype = ctypes.c_int
    lib.sse_oracle_decode_step.argtypes = [i32, i32, i32, i32, i32, i32, i32, f64,
                                           P, P, P, P, P, P, P, P, P, P, P, P, i64]
    lib.sse_oracle_group.restype = ctypes.c_int
    lib.sse_oracle_group.argtypes = [i64, i32, i32, i32, P, P, i32, P, P]
    lib.sse_oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_SO))
    return _lib


class _library_override:
    """Context manager: route the ctypes calls to another build of the oracle
    source (used only by the mutation tests, which plant mistakes in a copy)."""

    def __init__(self, so_path: str):
        self.so_path = so_path

    def __enter__(self):
        global _lib
        self._saved = _load()
        _lib = _bind(ctypes.CDLL(self.so_path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def max_threads() -> int:
    return int(_load().sse_oracle_max_threads())


def to_f64(x: np.ndarray) -> np.ndarray:
    """Exact upcast of stored values (float32, or bfloat16 bits held in uint16/int16)."""
    x = np.asarray(x)
    if x.dtype in (np.uint16, np.int16):
        return (x.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def forward(q, k, v, g, logits, cu_seqlens, *, top_k: int, use_shared: int = 1,
            scale: float = 1.0, q_shared=None, k_shared=None, initial_state=None,
            pairs=None, want_state: bool = True):
    """fp64 forward.  Arrays are [T, H, .]; returns dict with ``out`` [T,H,d],
    ``final_state`` [S,H,P,c,d] (or None), ``topk_idx`` [T,H,k] int32,
    ``topk_w`` [T,H,k], ``threads``.  ``pairs`` (iterable of b*H+h) limits the
    computed (sequence, head) pairs; other entries of the outputs are NaN /
    -1."""
    lib = _load()
    q64, k64, v64, g64, l64 = (to_f64(a) for a in (q, k, v, g, logits))
    T, H, c = q64.shape
    d = v64.shape[2]
    N = l64.shape[2]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    S = len(cu) - 1
    P = N + (1 if use_shared else 0)
    qs = None if q_shared is None else to_f64(q_shared)
    ks = None if k_shared is None else to_f64(k_shared)
    init = None if initial_state is None else to_f64(initial_state)
    out = np.full((T, H, d), np.nan)
    idx = np.full((T, H, top_k), -1, dtype=np.int32)
    w = np.full((T, H, top_k), np.nan)
    fin = np.full((S, H, P, c, d), np.nan) if want_state else None
    plist = None
    if pairs is not None:
        plist = np.ascontiguousarray(np.asarray(list(pairs), dtype=np.int64))
    nthr = lib.sse_oracle_forward(T, H, c, d, N, top_k, int(bool(use_shared)), float(scale),
                                  _ptr(q64), _ptr(k64), _ptr(v64), _ptr(g64), _ptr(l64),
                                  _ptr(qs), _ptr(ks), _ptr(cu), S, _ptr(init), _ptr(fin),
                                  _ptr(out), _ptr(idx), _ptr(w), _ptr(plist),
                                  0 if plist is None else len(plist))
    if nthr < 0:
        raise ValueError("oracle rejected the arguments")
    return {"out": out, "final_state": fin, "topk_idx": idx, "topk_w": w, "threads": nthr}


def decode_step(state, q, k, v, g, logits, *, top_k: int, use_shared: int = 1,
                scale: float = 1.0, q_shared=None, k_shared=None, pairs=None):
    """One fp64 decode step.  ``state`` [B,H,P,c,d] float64 is updated in place.
    Returns dict with ``out`` [B,H,d], ``topk_idx``, ``topk_w``, ``threads``."""
    lib = _load()
    assert state.dtype == np.float64 and state.flags["C_CONTIGUOUS"]
    q64, k64, v64, g64, l64 = (to_f64(a) for a in (q, k, v, g, logits))
    B, H, c = q64.shape
    d = v64.shape[2]
    N = l64.shape[2]
    qs = None if q_shared is None else to_f64(q_shared)
    ks = None if k_shared is None else to_f64(k_shared)
    out = np.full((B, H, d), np.nan)
    idx = np.full((B, H, top_k), -1, dtype=np.int32)
    w = np.full((B, H, top_k), np.nan)
    plist = None
    if pairs is not None:
        plist = np.ascontiguousarray(np.asarray(list(pairs), dtype=np.int64))
    nthr = lib.sse_oracle_decode_step(B, H, c, d, N, top_k, int(bool(use_shared)), float(scale),
                                      _ptr(q64), _ptr(k64), _ptr(v64), _ptr(g64), _ptr(l64),
                                      _ptr(qs), _ptr(ks), _ptr(state), _ptr(out), _ptr(idx),
                                      _ptr(w), _ptr(plist), 0 if plist is None else len(plist))
    if nthr < 0:
        raise ValueError("oracle rejected the arguments")
    return {"out": out, "topk_idx": idx, "topk_w": w, "threads": nthr}


def group(topk_idx, cu_seqlens, num_partitions: int):
    """Segment offsets and time-ordered token lists per (sequence, head,
    partition).  Returns (seg_off [S*H*N+1] int64, perm [H*k*T] int64)."""
    lib = _load()
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, H, k = idx.shape
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    S = len(cu) - 1
    seg_off = np.zeros(S * H * num_partitions + 1, dtype=np.int64)
    perm = np.full(H * k * T, -1, dtype=np.int64)
    lib.sse_oracle_group(T, H, num_partitions, k, _ptr(idx), _ptr(cu), S, _ptr(seg_off), _ptr(perm))
    return seg_off, perm


from .closed_form import closed_form, dense_gla  # noqa: E402

__all__ = ["build", "forward", "decode_step", "group", "closed_form", "dense_gla",
           "to_f64", "max_threads"]
