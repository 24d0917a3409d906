"""Host oracle for the DeepSeek-Sparse-Attention hot path (test infrastructure).

This package is TEST INFRASTRUCTURE, not product code.  Only ``tests/``, the
smoke check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import it.  The CUDA library never calls it, and it shares no code with it.

The arithmetic lives in ``dsa_oracle.c`` (plain C, double accumulation); this
module compiles it with the host C compiler and wraps it with ``ctypes``.  All
arrays are numpy arrays on the host: float inputs are ``float32`` (bf16 inputs
are widened to float32 exactly by the caller before they reach the oracle),
scores and outputs are ``float64``, indices ``int32``.

Sources are cited in ``dsa_oracle.h`` per function (page title and section).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``dsa_oracle.c`` into ``liboracle.so`` (gcc -O2, OpenMP)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                           os.path.getmtime(os.path.join(_HERE, "dsa_oracle.h"))))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64, i32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            lib.oracle_index_scores.argtypes = [P, P, P, i64, i32, i32, P]
            lib.oracle_topk.argtypes = [P, i64, i64, P, P]
            lib.oracle_kpool_select.argtypes = [P, i64, i64, i32, P, P]
            lib.oracle_sparse_mla.argtypes = [P, P, i64, i32, i32, i32, f64, P, i64, P, P]
            lib.oracle_dense_masked_mla.argtypes = [P, P, i64, i32, i32, i32, f64, P, P, P]
            lib.oracle_decode_step.argtypes = [P, P, P, i32, i32, P, P, i64, i32, i32, i32,
                                               f64, i64, i32, P, P, P, P, P]
            lib.oracle_pool_compress.argtypes = [P, i64, P, i32, i32, P]
            lib.oracle_new_pools.argtypes = [i64, i64, i32, P, P]
            lib.oracle_hadamard.argtypes = [P, i32, P]
            lib.oracle_rope.argtypes = [P, i32, i32, f64, i64, P]
            lib.oracle_index_prepare.argtypes = [P, P, i64, i32, i32, f64, P]
            lib.oracle_absorb_q.argtypes = [P, P, i32, i32, i32, i32, P]
            lib.oracle_up_project.argtypes = [P, P, i32, i32, i32, P]
            lib.oracle_order_desc.argtypes = [P, i64, P, i64, i64, i32, P]
            lib.oracle_order_desc.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [i32]
            lib.oracle_set_threads.restype = ctypes.c_int
            for fn in (lib.oracle_index_scores, lib.oracle_topk, lib.oracle_kpool_select,
                       lib.oracle_sparse_mla, lib.oracle_dense_masked_mla,
                       lib.oracle_decode_step, lib.oracle_pool_compress, lib.oracle_new_pools,
                       lib.oracle_hadamard, lib.oracle_rope, lib.oracle_index_prepare,
                       lib.oracle_absorb_q, lib.oracle_up_project):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, name: str):
    if rc != 0:
        raise ValueError(f"{name} rejected its arguments (rc={rc})")


def threads() -> int:
    """Number of OpenMP threads the oracle's parallel loops use."""
    return int(_load().oracle_set_threads(0))


def set_threads(n: int) -> int:
    """Use n threads from now on (n > 0); returns the number in effect."""
    return int(_load().oracle_set_threads(int(n)))


def index_scores(q, w, keys) -> np.ndarray:
    """s_t = sum_h w_h * relu(q_h . k_t) for every key row (float64)."""
    q, w, keys = _f32(q), _f32(w), _f32(keys)
    heads, dim = q.shape
    assert w.shape == (heads,) and keys.ndim == 2 and keys.shape[1] == dim
    out = np.empty(keys.shape[0], dtype=np.float64)
    _check(_load().oracle_index_scores(_ptr(q), _ptr(w), _ptr(keys), keys.shape[0],
                                       heads, dim, _ptr(out)), "oracle_index_scores")
    return out


def topk(scores, k: int) -> np.ndarray:
    """Ascending indices of the top-k under (score desc, index asc); all if n <= k."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    n = s.shape[0]
    idx = np.empty(max(min(n, k), 1), dtype=np.int32)
    n_sel = ctypes.c_int64(0)
    _check(_load().oracle_topk(_ptr(s), n, k, _ptr(idx), ctypes.byref(n_sel)), "oracle_topk")
    return idx[: n_sel.value].copy()


def kpool_select(pool_scores, L: int, k: int, kpool: int) -> np.ndarray:
    """Token indices selected by the k-pool rule for a query that sees L tokens."""
    s = np.ascontiguousarray(pool_scores, dtype=np.float64)
    assert s.shape[0] == L // kpool
    idx = np.empty(max(k + kpool - 1, L if L // kpool <= k // kpool else 0, 1), dtype=np.int32)
    n_sel = ctypes.c_int64(0)
    _check(_load().oracle_kpool_select(_ptr(s) if s.size else None, L, k, kpool, _ptr(idx),
                                       ctypes.byref(n_sel)), "oracle_kpool_select")
    return idx[: n_sel.value].copy()


def order_desc(unit_scores, sel, L: int, kpool: int) -> np.ndarray:
    """The selection `sel` (ascending, as the select functions emit it) with its
    units sorted by score descending, ties by ascending unit, the tail last."""
    s = np.ascontiguousarray(unit_scores, dtype=np.float64)
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    out = np.empty(max(sel.shape[0], 1), dtype=np.int32)
    _check(_load().oracle_order_desc(_ptr(s) if s.size else None, s.shape[0],
                                     _ptr(sel) if sel.size else None, sel.shape[0], L, kpool,
                                     _ptr(out)), "oracle_order_desc")
    return out[: sel.shape[0]].copy()


def sparse_mla(q_abs, rows, idx, scale: float, dv: int):
    """(out [heads, dv], lse [heads]) of softmax attention over rows[idx]."""
    q_abs, rows = _f32(q_abs), _f32(rows)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    heads, width = q_abs.shape
    assert rows.ndim == 2 and rows.shape[1] == width
    out = np.empty((heads, dv), dtype=np.float64)
    lse = np.empty(heads, dtype=np.float64)
    _check(_load().oracle_sparse_mla(_ptr(q_abs), _ptr(rows), rows.shape[0], heads, width, dv,
                                     float(scale), _ptr(idx), idx.shape[0], _ptr(out), _ptr(lse)),
           "oracle_sparse_mla")
    return out, lse


def dense_masked_mla(q_abs, rows, mask, scale: float, dv: int):
    """(out, lse) of dense attention over all rows with masked-off logits at -inf."""
    q_abs, rows = _f32(q_abs), _f32(rows)
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    heads, width = q_abs.shape
    assert mask.shape == (rows.shape[0],)
    out = np.empty((heads, dv), dtype=np.float64)
    lse = np.empty(heads, dtype=np.float64)
    _check(_load().oracle_dense_masked_mla(_ptr(q_abs), _ptr(rows), rows.shape[0], heads, width,
                                           dv, float(scale), _ptr(mask), _ptr(out), _ptr(lse)),
           "oracle_dense_masked_mla")
    return out, lse


def decode_step(q_idx, w, keys, q_abs, rows, L: int, k: int, kpool: int, scale: float, dv: int):
    """One query through scoring, selection and attention.

    ``keys`` holds L token keys (kpool == 1) or floor(L/kpool) pool keys.
    Returns a dict with ``scores`` (float64), ``idx`` (int32, ascending),
    ``out`` [heads, dv] and ``lse`` [heads] (float64).
    """
    q_idx, w, keys, q_abs, rows = _f32(q_idx), _f32(w), _f32(keys), _f32(q_abs), _f32(rows)
    ih, idim = q_idx.shape
    heads, width = q_abs.shape
    n_keys = L // kpool
    assert keys.shape[0] >= n_keys and rows.shape[0] >= L
    scores = np.empty(max(n_keys, 1), dtype=np.float64)
    idx = np.empty(max(k + kpool - 1, L, 1), dtype=np.int32)
    n_sel = ctypes.c_int64(0)
    out = np.empty((heads, dv), dtype=np.float64)
    lse = np.empty(heads, dtype=np.float64)
    _check(_load().oracle_decode_step(_ptr(q_idx), _ptr(w), _ptr(keys), ih, idim, _ptr(q_abs),
                                      _ptr(rows), L, heads, width, dv, float(scale), k, kpool,
                                      _ptr(scores), _ptr(idx), ctypes.byref(n_sel), _ptr(out),
                                      _ptr(lse)), "oracle_decode_step")
    return {"scores": scores[:n_keys].copy(), "idx": idx[: n_sel.value].copy(),
            "out": out, "lse": lse}


if __name__ == "__main__":  # pragma: no cover - manual build helper
    print(build(force="--force" in sys.argv))


def pool_compress(cells, pos) -> np.ndarray:
    """Compressed keys of complete pools: cells [n_pools, kpool, 2*dim] ([key | gate]
    per cell), pos [kpool, dim] -> [n_pools, dim] float64 (softmax over the slots of
    gate + pos, per channel, weighting the keys)."""
    cells, pos = _f32(cells), _f32(pos)
    n_pools, kpool, w2 = cells.shape
    dim = w2 // 2
    assert w2 == 2 * dim and pos.shape == (kpool, dim)
    out = np.empty((n_pools, dim), dtype=np.float64)
    _check(_load().oracle_pool_compress(_ptr(cells) if n_pools else None, n_pools, _ptr(pos),
                                        kpool, dim, _ptr(out) if n_pools else None),
           "oracle_pool_compress")
    return out


def new_pools(L: int, q_len: int, kpool: int):
    """(j0, j1): the complete pools whose last token is among the last q_len of L."""
    j0, j1 = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(_load().oracle_new_pools(L, q_len, kpool, ctypes.byref(j0), ctypes.byref(j1)),
           "oracle_new_pools")
    return j0.value, j1.value


def hadamard(x) -> np.ndarray:
    """H x with H the orthonormal Sylvester-Hadamard matrix (len(x) a power of two)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    _check(_load().oracle_hadamard(_ptr(x), x.shape[0], _ptr(out)), "oracle_hadamard")
    return out


def rope(x, rope_dims: int, base: float, pos: int) -> np.ndarray:
    """Rotary embedding of adjacent pairs of the first rope_dims dims at position pos."""
    x = _f32(x)
    out = np.empty(x.shape[0], dtype=np.float64)
    _check(_load().oracle_rope(_ptr(x), x.shape[0], rope_dims, float(base), int(pos), _ptr(out)),
           "oracle_rope")
    return out


def index_prepare(x, pos, rope_dims: int, base: float) -> np.ndarray:
    """H rope(x[v], pos[v]) for each row v of x [n, dim] (float64 out)."""
    x = _f32(x)
    p = np.ascontiguousarray(pos, dtype=np.int64)
    n, dim = x.shape
    out = np.empty((n, dim), dtype=np.float64)
    _check(_load().oracle_index_prepare(_ptr(x) if n else None, _ptr(p) if n else None, n, dim,
                                        rope_dims, float(base), _ptr(out) if n else None),
           "oracle_index_prepare")
    return out


def absorb_q(q, w_uk, rope: int) -> np.ndarray:
    """q [heads, nope + rope], w_uk [heads, nope, kv_lora] -> q_abs [heads, kv_lora + rope]."""
    q, w_uk = _f32(q), _f32(w_uk)
    heads, nope, kv_lora = w_uk.shape
    assert q.shape == (heads, nope + rope)
    out = np.empty((heads, kv_lora + rope), dtype=np.float64)
    _check(_load().oracle_absorb_q(_ptr(q), _ptr(w_uk), heads, nope, rope, kv_lora, _ptr(out)),
           "oracle_absorb_q")
    return out


def up_project(o, w_uv) -> np.ndarray:
    """o [heads, kv_lora] (latent), w_uv [heads, v_dim, kv_lora] -> [heads, v_dim]."""
    o = np.ascontiguousarray(o, dtype=np.float64)
    w_uv = _f32(w_uv)
    heads, v_dim, kv_lora = w_uv.shape
    assert o.shape == (heads, kv_lora)
    out = np.empty((heads, v_dim), dtype=np.float64)
    _check(_load().oracle_up_project(_ptr(o), _ptr(w_uv), heads, kv_lora, v_dim, _ptr(out)),
           "oracle_up_project")
    return out
