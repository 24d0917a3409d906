"""Python binding of libdsa, the GB300 DeepSeek-Sparse-Attention hot path.

Argument marshalling only: every step of the path runs in the CUDA kernels of
``libdsa.so`` behind the C ABI declared in ``include/dsa.h``.  The functions
below keep the C names, take torch CUDA tensors (PyTorch supplies device
memory and streams), pass their raw device pointers through ``ctypes`` and
raise :class:`DsaError` on any non-OK status.  There is no fallback: if the
library is missing or fails to load, importing the entry points raises.

Tensor layouts (row-major, contiguous), with ``W = kv_lora + rope_dim``:

* ``q_idx`` [n_q, idx_heads, idx_dim], ``k_idx`` [keys, idx_dim],
  ``q_abs`` [n_q, heads, W], ``cache`` [rows, W]: float32 or bfloat16
  (one dtype for all four, the shape's ``dtype``)
* ``w`` [n_q, idx_heads] float32
* ``scores`` [n_q, ld] float32, ``idx`` [n_q, top_k + kpool - 1] int32,
  ``n_sel`` [n_q] int32, ``out`` [n_q, heads, kv_lora] float32,
  ``lse`` [n_q, heads] float32
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

__all__ = [
    "DsaError", "Shape", "Batch", "load", "make_shape", "make_batch", "workspace_size",
    "alloc_workspace", "dsa_version", "dsa_index_row_width", "dsa_workspace_size",
    "dsa_workspace_init", "dsa_plan", "dsa_index_scores", "dsa_topk_select", "dsa_index_select",
    "dsa_sparse_mla_attn",
    "dsa_decode_step", "dsa_decode_step_host", "dsa_decode_step_noalloc", "dsa_check_device_error", "DecodeStep", "LIB_PATH",
    "OP_INDEX_SCORES", "OP_TOPK_SELECT", "OP_SPARSE_MLA", "OP_DECODE_STEP", "OP_INDEX_SELECT",
    "OP_POOL_COMPRESS", "dsa_pool_compress", "dsa_index_prepare", "dsa_workspace_set_wait_budget",
    "FLAG_TWO_LAUNCH", "FLAG_DESC_ORDER", "FLAG_DENSE", "OP_PROJECT", "dsa_absorb_q",
    "dsa_up_project", "OP_DECODE_STEP_HOST",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdsa.so")

DSA_F32, DSA_BF16 = 0, 1
OP_INDEX_SCORES, OP_TOPK_SELECT, OP_SPARSE_MLA, OP_DECODE_STEP, OP_INDEX_SELECT = 0, 1, 2, 3, 4
OP_POOL_COMPRESS = 5
OP_PROJECT = 6
OP_DECODE_STEP_HOST = 7
FLAG_TWO_LAUNCH, FLAG_DESC_ORDER, FLAG_DENSE = 0x1, 0x2, 0x4
STATUS = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED",
          3: "DSA_ERR_WORKSPACE", 4: "DSA_ERR_CUDA", 5: "DSA_ERR_DEVICE", 6: "DSA_ERR_TIMEOUT"}


class DsaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


class Shape(ctypes.Structure):
    _fields_ = [("idx_heads", ctypes.c_int32), ("idx_dim", ctypes.c_int32),
                ("heads", ctypes.c_int32), ("kv_lora", ctypes.c_int32),
                ("rope_dim", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("kpool", ctypes.c_int32), ("scale", ctypes.c_float), ("dtype", ctypes.c_int32)]


class Batch(ctypes.Structure):
    _fields_ = [("n_seq", ctypes.c_int32), ("n_q", ctypes.c_int32),
                ("max_q_len", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("max_kv_len", ctypes.c_int64), ("total_rows", ctypes.c_int64),
                ("total_keys", ctypes.c_int64), ("row_off", ctypes.c_void_p),
                ("key_off", ctypes.c_void_p), ("q_off", ctypes.c_void_p)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("kernel_launches", ctypes.c_int32), ("attn_splits", ctypes.c_int32),
                ("attn_rows_per_split", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def load() -> ctypes.CDLL:
    """Load libdsa.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdsa.so not found at {LIB_PATH}: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        P, S, i32, i64, sz = (ctypes.c_void_p, ctypes.POINTER(Shape), ctypes.c_int32,
                              ctypes.c_int64, ctypes.c_size_t)
        B = ctypes.POINTER(Batch)
        sigs = {
            "dsa_version": ([], ctypes.c_int),
            "dsa_status_string": ([i32], ctypes.c_char_p),
            "dsa_index_row_width": ([S], i64),
            "dsa_workspace_size": ([S, B, i32, ctypes.POINTER(sz)], ctypes.c_int),
            "dsa_workspace_init": ([P, sz, P], ctypes.c_int),
            "dsa_plan": ([S, B, i32, ctypes.POINTER(PlanInfo)], ctypes.c_int),
            "dsa_index_scores": ([S, B, P, P, P, P, i64, P, sz, P], ctypes.c_int),
            "dsa_topk_select": ([S, B, P, i64, P, P, P, sz, P], ctypes.c_int),
            "dsa_index_select": ([S, B, P, P, P, P, P, P, sz, P], ctypes.c_int),
            "dsa_sparse_mla_attn": ([S, B, P, P, P, P, P, P, P, sz, P], ctypes.c_int),
            "dsa_decode_step": ([S, B, P, P, P, P, P, P, P, P, P, P, sz, P], ctypes.c_int),
            "dsa_decode_step_host": ([S, B, P, P, P, P, P, P, P, P, P, P, sz, P], ctypes.c_int),
            "dsa_check_device_error": ([P, sz, P, ctypes.POINTER(i32)], ctypes.c_int),
            "dsa_decode_step_noalloc": ([S, B, P, P, P, P, P, P, P, P, P, P], ctypes.c_int),
            "dsa_pool_compress": ([S, B, P, P, P, P, sz, P], ctypes.c_int),
            "dsa_index_prepare": ([S, i64, P, P, i32, ctypes.c_double, P, P], ctypes.c_int),
            "dsa_workspace_set_wait_budget": ([P, sz, ctypes.c_uint64, P], ctypes.c_int),
            "dsa_absorb_q": ([S, i32, i32, P, P, P, P, sz, P], ctypes.c_int),
            "dsa_up_project": ([S, i32, i32, P, P, P, P, sz, P], ctypes.c_int),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libdsa takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libdsa takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _call(name: str, *args) -> int:
    rc = getattr(load(), name)(*args)
    if rc != 0:
        raise DsaError(name, rc)
    return rc


def make_shape(idx_heads=32, idx_dim=128, heads=64, kv_lora=512, rope_dim=64, top_k=2048,
               kpool=1, scale=1.0 / 16.0, dtype="bf16") -> Shape:
    d = {"f32": DSA_F32, "bf16": DSA_BF16, torch.float32: DSA_F32, torch.bfloat16: DSA_BF16}[dtype]
    return Shape(idx_heads, idx_dim, heads, kv_lora, rope_dim, top_k, kpool, float(scale), d)


def make_batch(row_off: torch.Tensor, key_off: torch.Tensor, q_off: torch.Tensor, n_q: int,
               max_q_len: int, max_kv_len: int, total_rows: int, total_keys: int,
               flags: int = 0) -> Batch:
    """Batch descriptor over int64 device offset arrays of n_seq+1 entries.

    ``total_rows`` / ``total_keys`` are the row counts of the cache and key
    tensors; ``flags`` the call's ``FLAG_*`` options.  The returned structure
    holds raw pointers: keep the three tensors alive while it is in use.
    """
    for t in (row_off, key_off, q_off):
        if t.dtype != torch.int64:
            raise ValueError("offset arrays are int64")
    n_seq = row_off.numel() - 1
    b = Batch(n_seq, int(n_q), int(max_q_len), int(flags), int(max_kv_len), int(total_rows),
              int(total_keys), _ptr(row_off), _ptr(key_off), _ptr(q_off))
    b._keep = (row_off, key_off, q_off)
    return b


def dsa_version() -> int:
    return load().dsa_version()


def dsa_index_row_width(shape: Shape) -> int:
    return int(load().dsa_index_row_width(ctypes.byref(shape)))


def dsa_workspace_size(shape: Shape, batch: Batch, op: int) -> int:
    n = ctypes.c_size_t(0)
    _call("dsa_workspace_size", ctypes.byref(shape), ctypes.byref(batch), op, ctypes.byref(n))
    return int(n.value)


workspace_size = dsa_workspace_size


def dsa_plan(shape: Shape, batch: Batch, op: int) -> dict:
    info = PlanInfo()
    _call("dsa_plan", ctypes.byref(shape), ctypes.byref(batch), op, ctypes.byref(info))
    return {"kernel_launches": info.kernel_launches, "attn_splits": info.attn_splits,
            "attn_rows_per_split": info.attn_rows_per_split}


def alloc_workspace(shape: Shape, batch: Batch, op: int = OP_DECODE_STEP,
                    device="cuda") -> torch.Tensor:
    """Zero-filled workspace of the size the library asks for (256-byte aligned)."""
    n = dsa_workspace_size(shape, batch, op)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def dsa_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _call("dsa_workspace_init", _ptr(ws), ws.numel(), _stream(stream))


def dsa_index_scores(shape, batch, q_idx, w, k_idx, scores, ld, ws, stream=None) -> None:
    _call("dsa_index_scores", ctypes.byref(shape), ctypes.byref(batch), _ptr(q_idx), _ptr(w),
          _ptr(k_idx), _ptr(scores), int(ld), _ptr(ws), ws.numel(), _stream(stream))


def dsa_topk_select(shape, batch, scores, ld, idx, n_sel, ws, stream=None) -> None:
    _call("dsa_topk_select", ctypes.byref(shape), ctypes.byref(batch), _ptr(scores), int(ld),
          _ptr(idx), _ptr(n_sel), _ptr(ws), ws.numel(), _stream(stream))


def dsa_index_select(shape, batch, q_idx, w, k_idx, idx, n_sel, ws, stream=None) -> None:
    _call("dsa_index_select", ctypes.byref(shape), ctypes.byref(batch), _ptr(q_idx), _ptr(w),
          _ptr(k_idx), _ptr(idx), _ptr(n_sel), _ptr(ws), ws.numel(), _stream(stream))


def dsa_sparse_mla_attn(shape, batch, q_abs, cache, idx, n_sel, out, lse, ws, stream=None) -> None:
    _call("dsa_sparse_mla_attn", ctypes.byref(shape), ctypes.byref(batch), _ptr(q_abs),
          _ptr(cache), _ptr(idx), _ptr(n_sel), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
          _stream(stream))


def dsa_decode_step(shape, batch, q_idx, w, k_idx, q_abs, cache, out, lse=None, idx_out=None,
                    n_sel_out=None, ws=None, stream=None) -> None:
    _call("dsa_decode_step", ctypes.byref(shape), ctypes.byref(batch), _ptr(q_idx), _ptr(w),
          _ptr(k_idx), _ptr(q_abs), _ptr(cache), _ptr(out), _ptr(lse), _ptr(idx_out),
          _ptr(n_sel_out), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream))


def _host_ptr(t: Optional[torch.Tensor]):
    """A pinned host tensor's address (or a CUDA tensor's): the per-step
    buffers of dsa_decode_step_host."""
    if t is None:
        return None
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("dsa_decode_step_host takes pinned host (or CUDA) tensors")
    if not t.is_contiguous():
        raise ValueError("libdsa takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def dsa_decode_step_host(shape, batch, q_idx, w, k_idx, q_abs, cache, out, lse=None,
                         idx_out=None, n_sel_out=None, ws=None, stream=None) -> None:
    """dsa_decode_step with q_idx, w, q_abs, out and lse in page-locked host
    memory (or device memory); the workspace is sized with OP_DECODE_STEP_HOST."""
    _call("dsa_decode_step_host", ctypes.byref(shape), ctypes.byref(batch), _host_ptr(q_idx),
          _host_ptr(w), _ptr(k_idx), _host_ptr(q_abs), _ptr(cache), _host_ptr(out),
          _host_ptr(lse), _ptr(idx_out),
          _ptr(n_sel_out), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream))


def dsa_decode_step_noalloc(shape, batch, q_idx, w, k_idx, q_abs, cache, out, lse=None,
                            idx_out=None, n_sel_out=None, stream=None) -> None:
    """dsa_decode_step without a workspace, for callers that cannot allocate
    device memory: the scratch is a fixed array inside libdsa (see dsa.h)."""
    _call("dsa_decode_step_noalloc", ctypes.byref(shape), ctypes.byref(batch), _ptr(q_idx),
          _ptr(w), _ptr(k_idx), _ptr(q_abs), _ptr(cache), _ptr(out), _ptr(lse), _ptr(idx_out),
          _ptr(n_sel_out), _stream(stream))


def dsa_pool_compress(shape, batch, cells, pos, pool_keys, ws, stream=None) -> None:
    """Compressed keys of the pools completed by each sequence's new tokens (see dsa.h)."""
    _call("dsa_pool_compress", ctypes.byref(shape), ctypes.byref(batch), _ptr(cells), _ptr(pos),
          _ptr(pool_keys), _ptr(ws), ws.numel(), _stream(stream))


def dsa_index_prepare(shape, x, pos, rope_dims, rope_base, out, stream=None) -> None:
    """out = H . rope(x, pos), rounded to the shape's dtype (see dsa.h)."""
    _call("dsa_index_prepare", ctypes.byref(shape), int(x.shape[0]), _ptr(x), _ptr(pos),
          int(rope_dims), float(rope_base), _ptr(out), _stream(stream))


def dsa_check_device_error(ws: Optional[torch.Tensor], stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error code;
    ``ws=None`` reads the no-allocation entry point's scratch array."""
    code = ctypes.c_int32(0)
    rc = load().dsa_check_device_error(_ptr(ws), ws.numel() if ws is not None else 0,
                                       _stream(stream), ctypes.byref(code))
    if rc not in (0, 5, 6):
        raise DsaError("dsa_check_device_error", rc)
    return int(code.value)


def dsa_absorb_q(shape, q, w_uk, q_abs, ws, stream=None) -> None:
    """q [n_q, heads, nope + rope], w_uk [heads, nope, kv_lora] -> q_abs (see dsa.h)."""
    _call("dsa_absorb_q", ctypes.byref(shape), int(q.shape[0]), int(w_uk.shape[1]), _ptr(q),
          _ptr(w_uk), _ptr(q_abs), _ptr(ws), ws.numel(), _stream(stream))


def dsa_up_project(shape, o, w_uv, out, ws, stream=None) -> None:
    """o [n_q, heads, kv_lora] float32, w_uv [heads, v_dim, kv_lora] -> out (see dsa.h)."""
    _call("dsa_up_project", ctypes.byref(shape), int(o.shape[0]), int(w_uv.shape[1]), _ptr(o),
          _ptr(w_uv), _ptr(out), _ptr(ws), ws.numel(), _stream(stream))


def dsa_workspace_set_wait_budget(ws: torch.Tensor, ns: int, stream=None) -> None:
    """Budget of the waits between CTAs of kernels using ``ws`` (0 = default)."""
    _call("dsa_workspace_set_wait_budget", _ptr(ws), ws.numel(), int(ns), _stream(stream))


class DecodeStep:
    """The whole hot path for a fixed batch layout, with its own workspace.

    ``inputs`` is a dict with the tensors of the layout above plus the int64
    offset arrays ``row_off``, ``key_off``, ``q_off`` (all on one CUDA device);
    ``wl`` supplies the geometry (``top_k``, ``kpool``, ``rope``, ``scale``,
    ``dtype``, ``kv_lens``, ``q_lens``).
    """

    def __init__(self, wl, row_off, key_off, q_off, device="cuda"):
        self.shape = make_shape(wl.idx_heads, wl.idx_dim, wl.heads, wl.kv_lora, wl.rope, wl.top_k,
                                wl.kpool, wl.scale, wl.dtype)
        self.batch = make_batch(row_off, key_off, q_off, wl.n_q, max(wl.q_lens), max(wl.kv_lens),
                                sum(wl.kv_lens), sum(wl.key_counts()))
        self.ws = alloc_workspace(self.shape, self.batch, OP_DECODE_STEP, device)
        self.width = dsa_index_row_width(self.shape)
        self.n_q = wl.n_q
        self.heads, self.kv_lora = wl.heads, wl.kv_lora
        dev = self.ws.device
        self.idx = torch.empty((self.n_q, self.width), dtype=torch.int32, device=dev)
        self.n_sel = torch.empty(self.n_q, dtype=torch.int32, device=dev)

    def __call__(self, q_idx, w, k_idx, q_abs, cache, out, lse=None, stream=None):
        dsa_decode_step(self.shape, self.batch, q_idx, w, k_idx, q_abs, cache, out, lse,
                        self.idx, self.n_sel, self.ws, stream)
