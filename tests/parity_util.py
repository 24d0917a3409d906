"""Helpers for the GPU-vs-oracle parity tests.

The GPU side is always called through the C ABI (the Python binding); the
oracle side always receives host copies of exactly the tensors the GPU saw.

Acceptance bars:
* selections: bit-exact against the oracle's, except candidates whose oracle
  score lies within 1e-5 relative of the oracle's k-th score (near-ties the
  GPU's float32 accumulation order may legitimately swap);
* attention outputs, for bf16 inputs with float32 accumulation: both the
  maximum absolute error max|gpu - oracle| <= 2e-3 over every element, and the
  relative error max|gpu - oracle| / max|oracle| <= 1e-2 (the maximum error
  relative to the output's scale: an element-wise ratio is undefined where the
  output crosses zero); float32 inputs 1e-4 and 1e-3.  The log-sum-exp takes
  the same two bounds.  Every check records its achieved errors (printed at the
  end of the run by conftest.py);
* indexer scores: |gpu - oracle| <= 1e-5 * M_t + 1e-6, with M_t = sum_h |w_h|
  sum_i |q_hi k_ti| the magnitude bound of the sum (float32 accumulation of
  128-term dots, then 32 weighted terms, rounds to well under 1e-5 of M_t).
"""
from __future__ import annotations

import os

import numpy as np
import torch

import deepseek_sparse_attention_gb300 as dsa
import oracle

ATT_TOL = {"bf16": (2e-3, 1e-2), "f32": (1e-4, 1e-3)}
NEAR_TIE_REL = 1e-5

# (test id, dtype, max-abs error, relative error) of every attention check
ACHIEVED = []


def host_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def to_device(inp: dict, device="cuda") -> dict:
    out = {}
    for k, v in inp.items():
        if isinstance(v, torch.Tensor):
            out[k] = v.to(device)
        elif isinstance(v, list) and v and isinstance(v[0], torch.Tensor):
            out[k] = [t.to(device) for t in v]
        else:
            out[k] = v
    return out


def gpu_shape(wl):
    return dsa.make_shape(wl.idx_heads, wl.idx_dim, wl.heads, wl.kv_lora, wl.rope, wl.top_k,
                          wl.kpool, wl.scale, wl.dtype)


def gpu_batch(wl, d, flags: int = 0):
    return dsa.make_batch(d["row_off"], d["key_off"], d["q_off"], wl.n_q, max(wl.q_lens),
                          max(wl.kv_lens), sum(wl.kv_lens), sum(wl.key_counts()), flags)


def query_slices(wl, d, q):
    """Host-side coordinates of query q: sequence, L, row/key offsets."""
    seq = int(d["q_seq"][q])
    L = int(d["q_nvis"][q])
    r0 = sum(wl.kv_lens[:seq])
    k0 = sum(wl.key_counts()[:seq])
    return seq, L, r0, k0


def oracle_query(wl, d_host, q):
    """Oracle run of one query on host copies: scores, selection, attention."""
    seq, L, r0, k0 = query_slices(wl, d_host, q)
    n_keys = L // wl.kpool
    keys = host_f32(d_host["k_idx"][k0:k0 + n_keys])
    rows = host_f32(d_host["cache"][r0:r0 + L])
    qi = host_f32(d_host["q_idx"][q])
    w = host_f32(d_host["w"][q])
    qa = host_f32(d_host["q_abs"][q])
    r = oracle.decode_step(qi, w, keys, qa, rows, L, wl.top_k, wl.kpool, wl.scale, wl.kv_lora)
    r.update(L=L, rows=rows, q_abs=qa, keys=keys, q=qi, w=w)
    return r


def score_bound(q, w, keys):
    """M_t = sum_h |w_h| sum_i |q_hi k_ti|, in float64."""
    return np.abs(keys).astype(np.float64) @ np.abs(q).astype(np.float64).T @ np.abs(w).astype(
        np.float64)


def check_scores(gpu_scores: np.ndarray, r: dict):
    ref = r["scores"]
    M = score_bound(r["q"], r["w"], r["keys"])
    err = np.abs(gpu_scores.astype(np.float64) - ref)
    bad = err > 1e-5 * M + 1e-6
    assert not bad.any(), f"{bad.sum()} scores off; worst {err.max():.3e}"


def check_selection(gpu_idx: np.ndarray, r: dict, top_k: int, kpool: int):
    """Exact set match except near-ties at the k-th (pool) score."""
    L = r["L"]
    ref = r["idx"]
    assert len(gpu_idx) == len(ref), f"n_sel {len(gpu_idx)} != oracle {len(ref)}"
    assert np.all(np.diff(gpu_idx) > 0), "selection not strictly ascending"
    assert gpu_idx.min() >= 0 and gpu_idx.max() < L
    if np.array_equal(gpu_idx, ref):
        return 0
    s = r["scores"]
    keep = top_k // kpool
    kth = np.sort(s)[::-1][keep - 1]
    diff = set(gpu_idx.tolist()) ^ set(ref.tolist())
    units = {t // kpool for t in diff}
    for u in units:
        assert u < len(s), f"tail token {u} differs"
        assert abs(s[u] - kth) <= NEAR_TIE_REL * abs(kth), \
            f"unit {u}: score {s[u]!r} vs k-th {kth!r} is not a near-tie"
    return len(units)


def _errors(got: np.ndarray, ref: np.ndarray):
    """(max |got - ref|, that over max |ref|) in float64; -inf == -inf counts as 0."""
    g, r = got.astype(np.float64), np.asarray(ref, dtype=np.float64)
    same = (g == r)                                   # equal infinities included
    err = np.where(same, 0.0, np.abs(g - r))
    scale = np.abs(r[np.isfinite(r)]).max() if np.isfinite(r).any() else 0.0
    mx = float(err.max()) if err.size else 0.0
    return mx, (mx / scale if scale > 0 else (0.0 if mx == 0 else float("inf")))


def check_attention(out: np.ndarray, lse: np.ndarray, ref_out: np.ndarray, ref_lse: np.ndarray,
                    dtype: str, label: str = None):
    """Max-abs and relative error of the output (and lse) within the bars."""
    atol, rtol = ATT_TOL[dtype]
    assert np.all(np.isfinite(out)), "non-finite output"
    abs_e, rel_e = _errors(out, ref_out)
    if label is None:
        label = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    ACHIEVED.append((label, dtype, abs_e, rel_e))
    assert abs_e <= atol, f"max abs err {abs_e:.3e} > {atol}"
    assert rel_e <= rtol, f"relative err {rel_e:.3e} > {rtol} (max abs {abs_e:.3e})"
    if lse is not None:
        l_abs, l_rel = _errors(lse, ref_lse)
        assert l_abs <= atol and l_rel <= rtol, f"lse err {l_abs:.3e} (rel {l_rel:.3e})"
    return abs_e
