"""Variants of the path, each through the C ABI against the oracle:

* cross-layer selection reuse ("GLM-5.x (glm-dsa, glm5next)", "The block", row
  "Indexer layers": the layers without an indexer attend over the selection of
  the last layer that has one) -- one dsa_index_select, then
  dsa_sparse_mla_attn over two layers' caches;
* descending-score emission order (DSA_FLAG_DESC_ORDER; "Add GLM-5.3-Flash
  support", DSA verification);
* the dense A/B switch (DSA_FLAG_DENSE; "GLM-5.x", environment knobs: top-k 0
  attends densely past the indexer's top-k).
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dsa.load()
    oracle.build()


def _outputs(wl, width):
    return (torch.full((wl.n_q, wl.heads, wl.kv_lora), float("nan"), device="cuda"),
            torch.full((wl.n_q, wl.heads), float("nan"), device="cuda"),
            torch.full((wl.n_q, width), -7, dtype=torch.int32, device="cuda"),
            torch.full((wl.n_q,), -7, dtype=torch.int32, device="cuda"))


def _step(wl, d, flags=0):
    sh, b = gpu_shape(wl), gpu_batch(wl, d, flags)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP)
    out, lse, idx, n_sel = _outputs(wl, dsa.dsa_index_row_width(sh))
    dense = bool(flags & dsa.FLAG_DENSE)
    dsa.dsa_decode_step(sh, b, d["q_idx"], d["w"], d["k_idx"], d["q_abs"], d["cache"], out, lse,
                        None if dense else idx, None if dense else n_sel, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    return out.cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy(), n_sel.cpu().numpy()


def _scores(wl, d):
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_INDEX_SCORES)
    ld = max(max(wl.kv_lens) // wl.kpool, 1)
    scores = torch.full((wl.n_q, ld), float("nan"), device="cuda")
    dsa.dsa_index_scores(sh, b, d["q_idx"], d["w"], d["k_idx"], scores, ld, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    return scores.cpu().numpy()


# ------------------------------------------------------------ cross-layer reuse

@pytest.mark.parametrize("kv_lens,kpool", [([9000, 40000, 1500], 1), ([20003, 2052], 4)])
def test_cross_layer_reuse_one_selection_two_caches(kv_lens, kpool):
    """One selection from the indexer layer's inputs, applied to that layer's
    cache and to another layer's (its own absorbed queries and latent rows):
    both attentions match the oracle over the oracle's selection."""
    rope = 64 if kpool == 1 else 0
    wl = workloads.small("reuse_a", kv_lens, top_k=2048, kpool=kpool, rope=rope, seed=31)
    wl_b = workloads.small("reuse_b", kv_lens, top_k=2048, kpool=kpool, rope=rope, seed=32)
    ha, hb = workloads.make(wl, "cpu"), workloads.make(wl_b, "cpu")
    da, db = to_device(ha), to_device(hb)
    sh, b = gpu_shape(wl), gpu_batch(wl, da)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP)
    width = dsa.dsa_index_row_width(sh)
    idx = torch.full((wl.n_q, width), -7, dtype=torch.int32, device="cuda")
    n_sel = torch.full((wl.n_q,), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_index_select(sh, b, da["q_idx"], da["w"], da["k_idx"], idx, n_sel, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    idx_h, n_h = idx.cpu().numpy(), n_sel.cpu().numpy()
    refs = [oracle_query(wl, ha, q) for q in range(wl.n_q)]
    for q in range(wl.n_q):
        check_selection(idx_h[q, : n_h[q]], refs[q], wl.top_k, wl.kpool)
    for layer in (ha, hb):
        dl = da if layer is ha else db
        out = torch.full((wl.n_q, wl.heads, wl.kv_lora), float("nan"), device="cuda")
        lse = torch.full((wl.n_q, wl.heads), float("nan"), device="cuda")
        dsa.dsa_sparse_mla_attn(sh, b, dl["q_abs"], dl["cache"], idx, n_sel, out, lse, ws)
        assert dsa.dsa_check_device_error(ws) == 0
        out, lse = out.cpu().numpy(), lse.cpu().numpy()
        r0 = 0
        for q, L in enumerate(wl.q_nvis()):
            rows = host_f32(layer["cache"][r0:r0 + L])
            o_ref, l_ref = oracle.sparse_mla(host_f32(layer["q_abs"][q]), rows, refs[q]["idx"],
                                             wl.scale, wl.kv_lora)
            check_attention(out[q], lse[q], o_ref, l_ref, wl.dtype)
            r0 += L


# ------------------------------------------------------------ descending order

def _select(scores_np, L_list, top_k, kpool, flags):
    n = len(L_list)
    ld = scores_np.shape[1]
    row_off = torch.tensor(np.concatenate([[0], np.cumsum(L_list)]), dtype=torch.int64).cuda()
    key_off = torch.tensor(np.concatenate([[0], np.cumsum([L // kpool for L in L_list])]),
                           dtype=torch.int64).cuda()
    q_off = torch.arange(n + 1, dtype=torch.int64).cuda()
    sh = dsa.make_shape(top_k=top_k, kpool=kpool, rope_dim=0 if kpool > 1 else 64)
    b = dsa.make_batch(row_off, key_off, q_off, n, 1, max(L_list), sum(L_list),
                       sum(L // kpool for L in L_list), flags)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_TOPK_SELECT)
    width = dsa.dsa_index_row_width(sh)
    idx = torch.full((n, width), -7, dtype=torch.int32, device="cuda")
    n_sel = torch.zeros(n, dtype=torch.int32, device="cuda")
    dsa.dsa_topk_select(sh, b, torch.from_numpy(scores_np).cuda(), ld, idx, n_sel, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    return idx.cpu().numpy(), n_sel.cpu().numpy()


@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("kpool,L_list", [
    (1, [5000, 2048, 2049, 131072, 3, 700]),
    (4, [2050, 2051, 2052, 2053, 2055, 2056, 2100, 16, 40000, 9003]),
], ids=["tokens", "pools"])
def test_desc_order_select_is_exact(kpool, L_list, ties):
    """Given float32 scores, the descending order is bit-exact against the
    oracle's ordering of the oracle's selection: the same set, units by score
    descending and equal scores by ascending index, pools whole, the tail last,
    dense rows included."""
    rng = np.random.default_rng(61 + kpool + 2 * ties)
    top_k = 2048
    ld = max(L // kpool for L in L_list)
    s = np.zeros((len(L_list), ld), np.float32)
    for i, L in enumerate(L_list):
        n = L // kpool
        s[i, :n] = rng.integers(-4, 5, n) if ties else rng.standard_normal(n)
    asc, n_asc = _select(s, L_list, top_k, kpool, 0)
    idx, n_sel = _select(s, L_list, top_k, kpool, dsa.FLAG_DESC_ORDER)
    assert np.array_equal(n_sel, n_asc)
    for i, L in enumerate(L_list):
        u = s[i, : L // kpool].astype(np.float64)
        ref_sel = oracle.topk(u, top_k) if kpool == 1 else oracle.kpool_select(u, L, top_k, kpool)
        assert np.array_equal(asc[i, : n_asc[i]], ref_sel), f"L={L}"
        want = oracle.order_desc(u, ref_sel, L, kpool)
        assert np.array_equal(idx[i, : n_sel[i]], want), f"L={L}"
        assert np.all(idx[i, n_sel[i]:] == -1)


DESC = [
    workloads.small("desc_decode", [40000, 1500, 9000], top_k=2048, seed=41),
    workloads.small("desc_kpool", [9000, 2051, 100003], top_k=2048, kpool=4, rope=0, seed=42),
    workloads.small("desc_prefill", [3000], q_lens=[16], top_k=512, seed=43),
]


@pytest.mark.parametrize("wl", DESC, ids=lambda w: w.name)
def test_desc_order_decode_step(wl):
    """The whole step with descending order: the selection is the ascending
    path's set, ordered as the oracle orders it by the GPU's own float32 scores;
    the attention over it matches the oracle."""
    host = workloads.make(wl, "cpu")
    d = to_device(host)
    _, _, asc, n_asc = _step(wl, d)
    out, lse, idx, n_sel = _step(wl, d, dsa.FLAG_DESC_ORDER)
    sc = _scores(wl, d)
    assert np.array_equal(n_sel, n_asc)
    for q, L in enumerate(wl.q_nvis()):
        sel = idx[q, : n_sel[q]]
        assert np.array_equal(np.sort(sel), asc[q, : n_asc[q]])
        u = sc[q, : L // wl.kpool].astype(np.float64)
        assert np.array_equal(sel, oracle.order_desc(u, asc[q, : n_asc[q]], L, wl.kpool))
        r = oracle_query(wl, host, q)
        check_selection(np.sort(sel), r, wl.top_k, wl.kpool)
        o_ref, l_ref = oracle.sparse_mla(r["q_abs"], r["rows"], sel, wl.scale, wl.kv_lora)
        check_attention(out[q], lse[q], o_ref, l_ref, wl.dtype)


# ------------------------------------------------------------ dense switch

DENSE = [
    workloads.small("dense_rows", [9000, 700, 40000, 3], top_k=2048, seed=51),
    workloads.small("dense_chunk", [3000], q_lens=[8], top_k=512, seed=52),
    workloads.small("dense_nope", [5000, 2051], top_k=2048, kpool=4, rope=0, seed=53),
    workloads.small("dense_f32", [3000, 100], top_k=256, dtype="f32", seed=54),
]


@pytest.mark.parametrize("wl", DENSE, ids=lambda w: w.name)
def test_dense_switch_attends_every_visible_row(wl):
    """With the switch on, each query attends over all of its L rows, past the
    top-k: the oracle's dense attention under an all-ones mask."""
    host = workloads.make(wl, "cpu")
    out, lse, _, _ = _step(wl, to_device(host), dsa.FLAG_DENSE)
    r0 = 0
    seq_q = [s for s, nq in enumerate(wl.q_lens) for _ in range(nq)]
    starts = np.concatenate([[0], np.cumsum(wl.kv_lens)])
    for q, L in enumerate(wl.q_nvis()):
        r0 = int(starts[seq_q[q]])
        rows = host_f32(host["cache"][r0:r0 + L])
        o_ref, l_ref = oracle.dense_masked_mla(host_f32(host["q_abs"][q]), rows,
                                               np.ones(L, np.uint8), wl.scale, wl.kv_lora)
        check_attention(out[q], lse[q], o_ref, l_ref, wl.dtype)


def test_dense_switch_on_the_attention_entry_point():
    """dsa_sparse_mla_attn with the switch ignores idx / n_sel (NULL here)."""
    wl = DENSE[0]
    host = workloads.make(wl, "cpu")
    d = to_device(host)
    sh, b = gpu_shape(wl), gpu_batch(wl, d, dsa.FLAG_DENSE)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_SPARSE_MLA)
    out = torch.full((wl.n_q, wl.heads, wl.kv_lora), float("nan"), device="cuda")
    lse = torch.full((wl.n_q, wl.heads), float("nan"), device="cuda")
    dsa.dsa_sparse_mla_attn(sh, b, d["q_abs"], d["cache"], None, None, out, lse, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    ref_out, ref_lse, _, _ = _step(wl, d, dsa.FLAG_DENSE)
    assert np.array_equal(out.cpu().numpy(), ref_out)
    assert np.array_equal(lse.cpu().numpy(), ref_lse)


def test_dense_switch_full_size_128k():
    """The 128K decode with the switch on: attention over all 131072 rows."""
    wl = workloads.named("glm52_decode_128k")
    d = workloads.make(wl, "cuda")
    out, lse, _, _ = _step(wl, d, dsa.FLAG_DENSE)
    rows = host_f32(d["cache"])
    o_ref, l_ref = oracle.dense_masked_mla(host_f32(d["q_abs"][0]), rows,
                                           np.ones(rows.shape[0], np.uint8), wl.scale, wl.kv_lora)
    check_attention(out[0], lse[0], o_ref, l_ref, wl.dtype, label="dense 128k")
    del d
    torch.cuda.empty_cache()
