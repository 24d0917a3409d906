"""dsa_decode_step_host: the step fed from page-locked host memory.

Its first kernel copies the query-side inputs (q_idx, w, q_abs) from host
memory into the workspace and its last kernel writes out / lse to host memory;
in between run the kernels of dsa_decode_step on the same values, so the
results must equal dsa_decode_step's bit for bit.  One case is also checked
against the oracle, and buffers the device cannot address are refused with
nothing enqueued.
"""
import ctypes

import pytest
import torch

import deepseek_sparse_attention_gb300 as dsa
import oracle
import workloads
from parity_util import (check_attention, check_selection, gpu_batch, gpu_shape, oracle_query,
                         to_device)

pytestmark = pytest.mark.gpu

CASES = [
    (workloads.named("tiny_fp32"), 0),
    (workloads.small("sparse_5000", [5000], top_k=2048, w_std=1 / 32 ** 0.5, cache_scale=0.5), 0),
    (workloads.small("ragged_batch", [300, 2500, 4097, 77], top_k=512), 0),
    (workloads.small("prefill_chunk", [3000], q_lens=[64], top_k=512), 0),
    (workloads.small("kpool_boundary", [2052, 2051, 4099, 9000], top_k=2048, kpool=4, rope=0), 0),
    (workloads.small("mixed_chunks", [3000, 2100, 900, 5000], q_lens=[1, 37, 1, 8], top_k=256), 0),
    (workloads.small("two_launch", [5000, 3000], top_k=2048), dsa.FLAG_TWO_LAUNCH),
    (workloads.small("dense", [700, 1500], top_k=256), dsa.FLAG_DENSE),
    (workloads.small("desc_order", [5000, 2100], top_k=512), dsa.FLAG_DESC_ORDER),
    # one query whose first key tiles the fused launch requests before the
    # batch offsets are read
    (workloads.small("one_query", [40000], top_k=2048, w_std=1 / 32 ** 0.5, cache_scale=0.5), 0),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dsa.load()
    oracle.build()


def _pinned(t: torch.Tensor) -> torch.Tensor:
    return t.cpu().contiguous().pin_memory()


def _run_both(wl, flags):
    d = to_device(workloads.make(wl))
    sh, b = gpu_shape(wl), gpu_batch(wl, d, flags)
    dense = bool(flags & dsa.FLAG_DENSE)
    width = dsa.dsa_index_row_width(sh)
    # the device-fed step
    ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP)
    out = torch.full((wl.n_q, wl.heads, wl.kv_lora), float("nan"), device="cuda")
    lse = torch.full((wl.n_q, wl.heads), float("nan"), device="cuda")
    idx = None if dense else torch.full((wl.n_q, width), -7, dtype=torch.int32, device="cuda")
    n_sel = None if dense else torch.full((wl.n_q,), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_decode_step(sh, b, d["q_idx"], d["w"], d["k_idx"], d["q_abs"], d["cache"], out, lse,
                        idx, n_sel, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    # the host-fed step: inputs and outputs in pinned host memory
    h = {k: _pinned(d[k]) for k in ("q_idx", "w", "q_abs")}
    h_out = torch.full((wl.n_q, wl.heads, wl.kv_lora), float("nan")).pin_memory()
    h_lse = torch.full((wl.n_q, wl.heads), float("nan")).pin_memory()
    ws_h = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP_HOST)
    idx_h = None if dense else torch.full((wl.n_q, width), -7, dtype=torch.int32, device="cuda")
    n_sel_h = None if dense else torch.full((wl.n_q,), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_decode_step_host(sh, b, h["q_idx"], h["w"], d["k_idx"], h["q_abs"], d["cache"], h_out,
                             h_lse, idx_h, n_sel_h, ws_h)
    assert dsa.dsa_check_device_error(ws_h) == 0          # synchronises the stream
    return d, (out, lse, idx, n_sel), (h_out, h_lse, idx_h, n_sel_h)


@pytest.mark.parametrize("wl,flags", CASES, ids=[c[0].name for c in CASES])
def test_host_fed_step_equals_device_step(wl, flags):
    _, dev, host = _run_both(wl, flags)
    for a, c in zip(dev, host):
        if a is None:
            assert c is None
            continue
        assert torch.equal(a.cpu(), c.cpu()), "host-fed step differs from the device-fed one"


def test_host_fed_step_matches_oracle():
    wl = workloads.small("sparse_5000", [5000], top_k=2048, w_std=1 / 32 ** 0.5, cache_scale=0.5)
    _, _, (h_out, h_lse, idx_h, n_sel_h) = _run_both(wl, 0)
    r = oracle_query(wl, workloads.make(wl), 0)
    sel = idx_h[0, : int(n_sel_h[0])].cpu().numpy()
    check_selection(sel, r, wl.top_k, wl.kpool)
    o_ref, l_ref = oracle.sparse_mla(r["q_abs"], r["rows"], sel, wl.scale, wl.kv_lora)
    check_attention(h_out[0].numpy(), h_lse[0].numpy(), o_ref, l_ref, wl.dtype)


def test_host_fed_step_refuses_unaddressable_buffers():
    """Pageable host memory: DSA_ERR_INVALID_ARG, nothing enqueued (the
    outputs keep their fill, the error word stays clear)."""
    wl = workloads.small("sparse_5000", [5000], top_k=2048)
    d = to_device(workloads.make(wl))
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP_HOST)
    pageable = d["q_abs"].cpu().contiguous()                    # not pinned
    h_out = torch.full((wl.n_q, wl.heads, wl.kv_lora), 3.0).pin_memory()
    h_q_idx, h_w = _pinned(d["q_idx"]), _pinned(d["w"])
    P = ctypes.c_void_p
    lib = dsa.load()
    rc = lib.dsa_decode_step_host(ctypes.byref(sh), ctypes.byref(b), P(h_q_idx.data_ptr()),
                                  P(h_w.data_ptr()), P(d["k_idx"].data_ptr()),
                                  P(pageable.data_ptr()), P(d["cache"].data_ptr()),
                                  P(h_out.data_ptr()), None, None, None, P(ws.data_ptr()),
                                  ws.numel(), None)
    assert rc == 1
    # a workspace sized for the device-fed step is too small for the staged inputs
    ws_small = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP)
    rc = lib.dsa_decode_step_host(ctypes.byref(sh), ctypes.byref(b), P(h_q_idx.data_ptr()),
                                  P(h_w.data_ptr()), P(d["k_idx"].data_ptr()),
                                  P(_pinned(d["q_abs"]).data_ptr()), P(d["cache"].data_ptr()),
                                  P(h_out.data_ptr()), None, None, None, P(ws_small.data_ptr()),
                                  ws_small.numel(), None)
    assert rc == 3
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_error(ws) == 0
    assert bool(torch.all(h_out == 3.0))


def test_host_fed_step_takes_device_buffers_too():
    """Device memory for the per-step buffers: the same results."""
    wl = workloads.small("ragged_batch", [300, 2500, 4097, 77], top_k=512)
    d, (out, lse, idx, n_sel), _ = _run_both(wl, 0)
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP_HOST)
    out2 = torch.full_like(out, float("nan"))
    lse2 = torch.full_like(lse, float("nan"))
    dsa.dsa_decode_step_host(sh, b, d["q_idx"], d["w"], d["k_idx"], d["q_abs"], d["cache"], out2,
                             lse2, None, None, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
