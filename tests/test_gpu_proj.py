"""The projections around the attention on the GPU, through the C ABI, against
the oracle ("GLM-5.x (glm-dsa, glm5next)", "The block": attn_k_b folded into
the query, attn_v_b into the output; "GLM 5.2 in one C file", "Attention:
Multi head Latent Attention With a Tiny KV Cache").

Bars, from the arithmetic (M = the sum of |products| of an output element):
* absorb, bf16: the float32 sum of 192 exact bf16 products (within 1e-5 M),
  then rounded to bf16 (half an ulp: 2^-8 of the value); float32: 1e-5 M;
* up-projection, bf16 weights: o carried as two bf16 parts (within 2^-16 of
  o, so 2^-16 M) and a float32 sum of 1024 products (within 3e-5 M): 5e-5 M;
  float32: 1e-5 M.
"""
import numpy as np
import pytest
import torch

import deepseek_sparse_attention_gb300 as dsa
import oracle
import workloads
from parity_util import (check_attention, check_selection, gpu_batch, gpu_shape, host_f32,
                         oracle_query, to_device)

pytestmark = pytest.mark.gpu

NOPE, V_DIM = 192, 256


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dsa.load()
    oracle.build()


def _ws(sh):
    return dsa.alloc_workspace(sh, dsa.make_batch(*(torch.zeros(2, dtype=torch.int64,
                                                                device="cuda"),) * 3,
                                                  0, 0, 0, 1, 1), dsa.OP_PROJECT)


def _absorb(sh, p):
    n_q, heads = p["q_full"].shape[0], p["q_full"].shape[1]
    q_abs = torch.full((n_q, heads, 512 + sh.rope_dim), float("nan"), dtype=p["q_full"].dtype,
                       device="cuda")
    ws = _ws(sh)
    dsa.dsa_absorb_q(sh, p["q_full"], p["w_uk"], q_abs, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    return q_abs


def _up(sh, o, w_uv):
    out = torch.full((o.shape[0], o.shape[1], w_uv.shape[1]), float("nan"), device="cuda")
    ws = _ws(sh)
    dsa.dsa_up_project(sh, o, w_uv, out, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    return out


def check_absorb(got, q, w_uk, rope, dtype):
    ref = oracle.absorb_q(q, w_uk, rope)
    M = np.einsum("hd,hdi->hi", np.abs(q[:, :NOPE]).astype(np.float64),
                  np.abs(w_uk).astype(np.float64))
    err = np.abs(got[:, :512].astype(np.float64) - ref[:, :512])
    bound = (2.0 ** -8 * 1.001 * np.abs(ref[:, :512]) if dtype == "bf16" else 0) + 1e-5 * M + 1e-30
    assert np.all(err <= bound), f"absorb: worst {err.max():.3e}"
    assert np.array_equal(got[:, 512:], q[:, NOPE:])               # the rope part, copied


def check_up(got, o, w_uv, dtype, extra=None):
    ref = oracle.up_project(o, w_uv)
    M = np.einsum("hvi,hi->hv", np.abs(w_uv).astype(np.float64), np.abs(o).astype(np.float64))
    err = np.abs(got.astype(np.float64) - ref)
    bound = (5e-5 if dtype == "bf16" else 1e-5) * M + 1e-30
    if extra is not None:
        bound = bound + extra
    assert np.all(err <= bound), f"up-projection: worst {err.max():.3e}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n_q", [1, 5, 64, 300])
def test_absorb_matches_oracle(n_q, dtype):
    """One query (a decode step), a few, one full query tile, and two tiles of
    which the second is ragged (300 = 256 + 44)."""
    wl = workloads.small("proj", [n_q], q_lens=[n_q], dtype=dtype, seed=n_q)
    p = to_device(workloads.projections(wl, "cpu"))
    sh = gpu_shape(wl)
    got = host_f32(_absorb(sh, p))
    q, w = host_f32(p["q_full"]), host_f32(p["w_uk"])
    for i in sorted({0, n_q // 2, n_q - 1}):
        check_absorb(got[i], q[i], w, wl.rope, dtype)


def test_absorb_nope_rows_without_rope():
    """The NoPE geometry (rope 0): q holds the no-rope part only."""
    wl = workloads.small("proj_nope", [17], q_lens=[17], rope=0, seed=3)
    p = to_device(workloads.projections(wl, "cpu"))
    got = host_f32(_absorb(gpu_shape(wl), p))
    q, w = host_f32(p["q_full"]), host_f32(p["w_uk"])
    for i in (0, 16):
        check_absorb(got[i], q[i], w, 0, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n_q", [1, 5, 64, 300])
def test_up_project_matches_oracle(n_q, dtype):
    wl = workloads.small("proj", [n_q], q_lens=[n_q], dtype=dtype, seed=100 + n_q)
    p = to_device(workloads.projections(wl, "cpu"))
    got = host_f32(_up(gpu_shape(wl), p["o"], p["w_uv"]))
    o, w = host_f32(p["o"]), host_f32(p["w_uv"])
    for i in sorted({0, n_q // 2, n_q - 1}):
        check_up(got[i], o[i], w, dtype)


def test_projections_at_the_prefill_chunk_size():
    """4096 queries (16 query tiles), checked on 64 evenly spaced queries."""
    wl = workloads.named("chunked_prefill_4096")
    p = workloads.projections(wl, "cuda")
    sh = gpu_shape(wl)
    qa = _absorb(sh, p)
    up = _up(sh, p["o"], p["w_uv"])
    w_uk, w_uv = host_f32(p["w_uk"]), host_f32(p["w_uv"])
    for i in sorted({int(round(j * 4095 / 63)) for j in range(64)}):
        check_absorb(host_f32(qa[i]), host_f32(p["q_full"][i]), w_uk, wl.rope, "bf16")
        check_up(host_f32(up[i]), host_f32(p["o"][i]), w_uv, "bf16")


@pytest.mark.parametrize("kv_lens,q_lens", [([9000, 3000], [1, 4]), ([131072], [1])])
def test_chain_absorb_step_up_project(kv_lens, q_lens):
    """absorb -> dsa_decode_step -> up-projection, on one stream, against the
    oracle stage by stage: the GPU's absorbed query against the oracle's
    absorption; the attention over the GPU's selection from that query against
    the oracle's; the final head outputs against the oracle's up-projection of
    the oracle's attention output, the attention's bound carried through the
    weights (|W (o_gpu - o_ref)| <= 2e-3 sum|W|)."""
    wl = workloads.small("chain", kv_lens, q_lens=q_lens, top_k=2048, seed=71,
                         w_std=1 / 32 ** 0.5, cache_scale=0.5)
    host = workloads.make(wl, "cpu")
    d = to_device(host)
    p = to_device(workloads.projections(wl, "cpu"))
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP)
    q_abs = torch.empty_like(d["q_abs"])
    width = dsa.dsa_index_row_width(sh)
    out = torch.empty((wl.n_q, 64, 512), device="cuda")
    lse = torch.empty((wl.n_q, 64), device="cuda")
    idx = torch.empty((wl.n_q, width), dtype=torch.int32, device="cuda")
    n_sel = torch.empty(wl.n_q, dtype=torch.int32, device="cuda")
    heads_out = torch.empty((wl.n_q, 64, V_DIM), device="cuda")
    dsa.dsa_absorb_q(sh, p["q_full"], p["w_uk"], q_abs, ws)
    dsa.dsa_decode_step(sh, b, d["q_idx"], d["w"], d["k_idx"], q_abs, d["cache"], out, lse, idx,
                        n_sel, ws)
    dsa.dsa_up_project(sh, out, p["w_uv"], heads_out, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    qa, o, ho = host_f32(q_abs), out.cpu().numpy(), host_f32(heads_out)
    idx, n_sel = idx.cpu().numpy(), n_sel.cpu().numpy()
    w_uk, w_uv = host_f32(p["w_uk"]), host_f32(p["w_uv"])
    host["q_abs"] = q_abs.cpu()                      # the oracle attends with the GPU's query
    wsum = np.abs(w_uv).astype(np.float64).sum(axis=2)
    for q in range(wl.n_q):
        check_absorb(qa[q], host_f32(p["q_full"][q]), w_uk, wl.rope, "bf16")
        r = oracle_query(wl, host, q)
        sel = idx[q, : n_sel[q]]
        check_selection(sel, r, wl.top_k, wl.kpool)
        o_ref, l_ref = oracle.sparse_mla(r["q_abs"], r["rows"], sel, wl.scale, wl.kv_lora)
        check_attention(o[q], None, o_ref, l_ref, wl.dtype)
        check_up(ho[q], o_ref.astype(np.float32), w_uv, "bf16", extra=2e-3 * wsum)
