"""Float64 CPU oracle for Multi-Segment Attention (MSA).

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python
binding) never imports, links or runs anything in this package; only the
tests, the smoke check and the bench's CPU-baseline leg do.  It shares no
code with the CUDA path.

Contents
  oracle.c     -- dense float64 attention over logical K/V, the segmented
                  (per-segment partials + log-sum-exp merge) float64 oracle
                  that reads the paged pool, the plain segment splitter and
                  the scatter reference.  Built to ``liboracle.so``.
  brute.py     -- tiny explicit-softmax float64 numpy version, for pins.
  segments.py  -- pure-Python brute-force segment splitter, for planner pins.

See ``oracle.c`` for the definition each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain C, -O2, portable)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-shared", "-fPIC", "-pthread",
               _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_dense_attention.argtypes = [i32, i32, i32, i32, f64, p, p, p, p, p, p, p, i64, p, p, i32]
    lib.oracle_dense_attention.restype = ctypes.c_int
    lib.oracle_segmented_attention.argtypes = [i32, i32, i32, i32, i32, f64, i32, p, p, p, p,
                                               p, p, p, p, i64, p, p, i32]
    lib.oracle_segmented_attention.restype = ctypes.c_int
    lib.oracle_segment_runs.argtypes = [i32, p, p, p]
    lib.oracle_segment_runs.restype = ctypes.c_int
    lib.oracle_scatter_rows.argtypes = [i64, i64, p, p, p, i64]
    lib.oracle_scatter_rows.restype = ctypes.c_int
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = f64
    return lib


def _load():
    global _lib
    if _lib is None:
        build_oracle()
        _lib = _bind(_LIB)
    return _lib


def load_variant(path):
    """Bind another build of oracle.c (used by the tests that plant mistakes
    in a copy of the oracle to show the pins catch them)."""
    return _bind(path)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _bits(a):
    """Accept bf16 data as uint16 bit patterns (numpy) or a torch bf16 tensor."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs must be uint16 bit patterns or torch.bfloat16 tensors")
    return np.ascontiguousarray(a)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def dense_attention(kv_indptr, k, v, q_indptr, q_pos, q, num_q_heads, num_kv_heads, scale,
                    rows=None, num_threads=None, lib=None):
    """Dense float64 causal attention over logical K/V (see oracle.c).

    k, v: bf16 [total_tokens, Hkv, D]; q: bf16 [n_q, Hq, D].
    Returns (out float64 [n_out, Hq, D], lse float64 [n_out, Hq]).
    """
    lib = lib or _load()
    kb, vb, qb = _bits(k), _bits(v), _bits(q)
    d = qb.shape[-1]
    kv_indptr = _c(kv_indptr, np.int64)
    q_indptr = _c(q_indptr, np.int64)
    q_pos = _c(q_pos, np.int32)
    rows_a = None if rows is None else _c(rows, np.int64)
    n_out = int(q_indptr[-1]) if rows_a is None else len(rows_a)
    out = np.zeros((n_out, num_q_heads, d), np.float64)
    lse = np.zeros((n_out, num_q_heads), np.float64)
    rc = lib.oracle_dense_attention(len(kv_indptr) - 1, num_q_heads, num_kv_heads, d, float(scale),
                                    _ptr(kv_indptr), _ptr(kb), _ptr(vb), _ptr(q_indptr), _ptr(q_pos),
                                    _ptr(qb), _ptr(rows_a), 0 if rows_a is None else len(rows_a),
                                    _ptr(out), _ptr(lse), num_threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_dense_attention failed: {rc}")
    return out, lse


def segmented_attention(block_table, seq_lens, k_pool, v_pool, q_indptr, q_pos, q, num_q_heads,
                        num_kv_heads, block_size, scale, rows=None, num_threads=None, lib=None):
    """Per-segment float64 attention + log-sum-exp merge, read through the block table."""
    lib = lib or _load()
    kb, vb, qb = _bits(k_pool), _bits(v_pool), _bits(q)
    d = qb.shape[-1]
    table = _c(block_table, np.int32)
    lens = _c(seq_lens, np.int32)
    q_indptr = _c(q_indptr, np.int64)
    q_pos = _c(q_pos, np.int32)
    rows_a = None if rows is None else _c(rows, np.int64)
    n_out = int(q_indptr[-1]) if rows_a is None else len(rows_a)
    out = np.zeros((n_out, num_q_heads, d), np.float64)
    lse = np.zeros((n_out, num_q_heads), np.float64)
    rc = lib.oracle_segmented_attention(table.shape[0], num_q_heads, num_kv_heads, d, block_size,
                                        float(scale), table.shape[1], _ptr(table), _ptr(lens),
                                        _ptr(kb), _ptr(vb), _ptr(q_indptr), _ptr(q_pos), _ptr(qb),
                                        _ptr(rows_a), 0 if rows_a is None else len(rows_a),
                                        _ptr(out), _ptr(lse), num_threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_segmented_attention failed: {rc}")
    return out, lse


def segment_runs(table_row, n_blocks):
    """Segments of one sequence as an int32 array [n_runs, 3] =
    (first logical block, first physical block, number of blocks)."""
    lib = _load()
    t = _c(table_row, np.int32)
    runs = np.zeros((max(n_blocks, 1), 3), np.int32)
    n = ctypes.c_int32(0)
    rc = lib.oracle_segment_runs(int(n_blocks), _ptr(t), _ptr(runs), ctypes.byref(n))
    if rc != 0:
        raise ValueError(f"missing block in table (rc={rc})")
    return runs[: n.value].copy()


def scatter_rows(src_bits, slot, pool_bits):
    """pool[slot[t]] = src[t] (slot < 0 skipped); operates in place on uint16 bits."""
    lib = _load()
    src = _c(src_bits, np.uint16)
    slot = _c(slot, np.int64)
    assert pool_bits.dtype == np.uint16 and pool_bits.flags["C_CONTIGUOUS"]
    row = int(np.prod(src.shape[1:])) if src.ndim > 1 else 1
    rc = lib.oracle_scatter_rows(len(slot), row, _ptr(src), _ptr(slot), _ptr(pool_bits),
                                 pool_bits.shape[0])
    if rc != 0:
        raise ValueError("slot out of range")
    return pool_bits


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))
