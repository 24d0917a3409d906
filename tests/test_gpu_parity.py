"""GPU parity: the CUDA path (through the C ABI) against the host oracle on the
same seeded inputs.  Reduced workloads span several tiles and a ragged tail;
the full-size workloads are checked on sampled queries in the launch
configuration the benchmark times."""
import numpy as np
import pytest
import torch

import deepseek_sparse_attention_gb300 as dsa
import oracle
import workloads
from parity_util import (check_attention, check_scores, check_selection, gpu_batch, gpu_shape,
                         host_f32, oracle_query, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dsa.load()
    oracle.build()


SMALL = [
    workloads.named("tiny_fp32"),
    workloads.small("one_seq_ragged_tail", [933], top_k=256),
    workloads.small("sparse_5000", [5000], top_k=2048, w_std=1 / 32 ** 0.5, cache_scale=0.5),
    workloads.small("dense_below_k", [1500], top_k=2048),
    workloads.small("ragged_batch", [300, 2500, 4097, 77], top_k=512),
    workloads.small("prefill_chunk", [3000], q_lens=[64], top_k=512),
    workloads.small("kpool_boundary", [2052, 2051, 4099, 9000], top_k=2048, kpool=4, rope=0),
    workloads.small("kpool_prefill", [1000], q_lens=[40], top_k=64, kpool=4, rope=0),
    workloads.small("fp32_kpool", [777, 130], top_k=64, kpool=4, rope=0, dtype="f32"),
    workloads.small("mixed_chunks", [3000, 2100, 900, 5000], q_lens=[1, 37, 1, 8], top_k=256),
    workloads.small("small_chunk", [600], q_lens=[5], top_k=128),
    # 24 decode queries with long rows: selection by a pair of CTAs per query
    workloads.small("pair_select_batch", [16384 + 997 * i for i in range(22)] + [1500, 40001],
                    top_k=2048, seed=9),
    # 60 decode queries: two attention splits per query, merged by a CTA pair
    # (an empty second split for L <= 1024, a one-row one for L = 1025)
    workloads.small("pair_merge_batch", [700, 1024, 1025, 30] + [3000 + 97 * i for i in range(56)],
                    top_k=2048, seed=10),
]


def run_step(wl, d):
    """Whole path through dsa_decode_step; returns host copies."""
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP)
    width = dsa.dsa_index_row_width(sh)
    out = torch.full((wl.n_q, wl.heads, wl.kv_lora), float("nan"), device="cuda")
    lse = torch.full((wl.n_q, wl.heads), float("nan"), device="cuda")
    idx = torch.full((wl.n_q, width), -7, dtype=torch.int32, device="cuda")
    n_sel = torch.full((wl.n_q,), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_decode_step(sh, b, d["q_idx"], d["w"], d["k_idx"], d["q_abs"], d["cache"], out, lse,
                        idx, n_sel, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    return out.cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy(), n_sel.cpu().numpy()


def run_scores(wl, d):
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_INDEX_SCORES)
    ld = max(max(wl.kv_lens) // wl.kpool, 1)
    scores = torch.full((wl.n_q, ld), float("nan"), device="cuda")
    dsa.dsa_index_scores(sh, b, d["q_idx"], d["w"], d["k_idx"], scores, ld, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    return scores.cpu().numpy()


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_decode_step_matches_oracle(wl):
    host = workloads.make(wl, "cpu")
    d = to_device(host)
    out, lse, idx, n_sel = run_step(wl, d)
    scores = run_scores(wl, d)
    for q in range(wl.n_q):
        r = oracle_query(wl, host, q)
        n_keys = r["L"] // wl.kpool
        check_scores(scores[q, :n_keys], r)
        sel = idx[q, : n_sel[q]]
        assert np.all(idx[q, n_sel[q]:] == -1), "unused index slots not cleared"
        check_selection(sel, r, wl.top_k, wl.kpool)
        # attention isolated on the GPU's own selection ...
        o_ref, l_ref = oracle.sparse_mla(r["q_abs"], r["rows"], sel, wl.scale, wl.kv_lora)
        check_attention(out[q], lse[q], o_ref, l_ref, wl.dtype)
        # ... and end to end when the sets agree exactly
        if np.array_equal(sel, r["idx"]):
            check_attention(out[q], lse[q], r["out"], r["lse"], wl.dtype)


# Structured indexer keys for the fused decode selection: the selected keys
# concentrated in a few CTAs' ranges, and blocks of equal top scores, resolved
# from the level-1 candidates or -- tie blocks larger than the candidate list --
# by the two further histogram levels and the ranked emission at T.
#   hot:        keys of a 1000-token window scaled by 3 (ReLU is positively
#               homogeneous: those scores triple and fill the top)
#   ties:       the query's best-scoring key vector, scaled by 3, repeated
#               over 3000 tokens: equal top scores, the lowest indices win
#   ties_over:  the same over 12000 tokens (k-pool: 12000 pools), more
#               candidates than the list holds
STRUCTURED = [
    ("hot", [40000, 61000], 1, 2048),
    ("hot", [5000], 1, 2048),                    # fewer key tiles than CTAs
    ("ties", [40000], 1, 2048),
    ("ties_over", [40000, 30000], 1, 2048),
    ("hot", [64000, 9000], 4, 2048),             # k-pool: pool keys
    ("ties_over", [200000], 4, 2048),
]


@pytest.mark.parametrize("kind,kv_lens,kpool,top_k", STRUCTURED,
                         ids=[f"{k}-{'-'.join(map(str, L))}-p{p}" for k, L, p, _ in STRUCTURED])
def test_decode_step_structured_scores(kind, kv_lens, kpool, top_k):
    wl = workloads.small(f"struct_{kind}", kv_lens, top_k=top_k, kpool=kpool,
                         rope=0 if kpool > 1 else 64, seed=21)
    host = workloads.make(wl, "cpu")
    k = host["k_idx"].clone()
    key_off = np.concatenate([[0], np.cumsum([L // kpool for L in kv_lens])])
    for i, L in enumerate(kv_lens):
        n = L // kpool
        k0 = int(key_off[i])
        a = k0 + n // 3
        if kind == "hot":
            m = 1000 // kpool
            k[a:a + m] = (k[a:a + m].float() * 3).to(k.dtype)
        else:
            m = 3000 if kind == "ties" else 12000
            # the best key of the sequence for its query, by its score on the host
            kk = host_f32(k[k0:k0 + n]).astype(np.float64)
            qi = host_f32(host["q_idx"][i]).astype(np.float64)
            wi = host_f32(host["w"][i]).astype(np.float64)
            best = int(np.argmax(np.maximum(kk @ qi.T, 0) @ wi))
            k[a:a + m] = (k[k0 + best].float() * 3).to(k.dtype).unsqueeze(0).expand(m, -1)
    host["k_idx"] = k
    out, lse, idx, n_sel = run_step(wl, to_device(host))
    for q in range(wl.n_q):
        r = oracle_query(wl, host, q)
        sel = idx[q, : n_sel[q]]
        check_selection(sel, r, wl.top_k, wl.kpool)
        if kind != "hot":
            # equal keys are bit-identical on both sides: the tie-break by
            # index is exact
            assert np.array_equal(sel, r["idx"])
        o_ref, l_ref = oracle.sparse_mla(r["q_abs"], r["rows"], sel, wl.scale, wl.kv_lora)
        check_attention(out[q], lse[q], o_ref, l_ref, wl.dtype)


def test_dense_below_k_equals_dense_attention():
    """Below top-k the path is exactly dense attention over every visible row."""
    wl = workloads.small("dense", [700], top_k=2048)
    host = workloads.make(wl, "cpu")
    out, lse, idx, n_sel = run_step(wl, to_device(host))
    assert n_sel[0] == 700 and np.array_equal(idx[0, :700], np.arange(700))
    q_abs, rows = host_f32(host["q_abs"][0]), host_f32(host["cache"])
    o_ref, l_ref = oracle.dense_masked_mla(q_abs, rows, np.ones(700, np.uint8), wl.scale, 512)
    check_attention(out[0], lse[0], o_ref, l_ref, "bf16")


# ------------------------------------------------------------ selection alone

def _select(scores_np, L_list, top_k, kpool):
    """dsa_topk_select on given float32 scores, one decode query per sequence."""
    n = len(L_list)
    ld = scores_np.shape[1]
    row_off = torch.tensor(np.concatenate([[0], np.cumsum(L_list)]), dtype=torch.int64).cuda()
    key_off = torch.tensor(np.concatenate([[0], np.cumsum([L // kpool for L in L_list])]),
                           dtype=torch.int64).cuda()
    q_off = torch.arange(n + 1, dtype=torch.int64).cuda()
    sh = dsa.make_shape(top_k=top_k, kpool=kpool, rope_dim=0 if kpool > 1 else 64)
    b = dsa.make_batch(row_off, key_off, q_off, n, 1, max(L_list), sum(L_list),
                       sum(L // kpool for L in L_list))
    ws = dsa.alloc_workspace(sh, b, dsa.OP_TOPK_SELECT)
    width = dsa.dsa_index_row_width(sh)
    idx = torch.full((n, width), -7, dtype=torch.int32, device="cuda")
    n_sel = torch.zeros(n, dtype=torch.int32, device="cuda")
    dsa.dsa_topk_select(sh, b, torch.from_numpy(scores_np).cuda(), ld, idx, n_sel, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    return idx.cpu().numpy(), n_sel.cpu().numpy()


@pytest.mark.parametrize("kind", ["normal", "int_ties", "all_zero", "signed_zeros", "huge"])
def test_topk_select_bit_exact(kind):
    """Given the same float32 scores, the selection is bit-exact against the
    oracle's (score desc, index asc) order."""
    rng = np.random.default_rng({"normal": 1, "int_ties": 2, "all_zero": 3, "signed_zeros": 4,
                                 "huge": 5}[kind])
    L_list = [5000, 2048, 2049, 131072, 3] if kind != "huge" else [1 << 20]
    top_k = 2048
    ld = max(L_list)
    s = np.zeros((len(L_list), ld), np.float32)
    for i, L in enumerate(L_list):
        if kind == "normal" or kind == "huge":
            s[i, :L] = rng.standard_normal(L)
        elif kind == "int_ties":
            s[i, :L] = rng.integers(-5, 6, L)
        elif kind == "signed_zeros":
            s[i, :L] = np.where(rng.random(L) < 0.5, -0.0, 0.0)
            s[i, :L:97] = 1.0
    idx, n_sel = _select(s, L_list, top_k, 1)
    for i, L in enumerate(L_list):
        ref = oracle.topk(s[i, :L].astype(np.float64), top_k)
        assert np.array_equal(idx[i, : n_sel[i]], ref)


@pytest.mark.parametrize("kind", ["normal", "int_ties", "all_zero", "signed_zeros"])
def test_topk_select_pair_bit_exact(kind):
    """24 queries with long rows take two CTAs per query (each half of the row,
    candidates exchanged): the same bit-exact selection, ties included, with
    odd lengths, a dense row and a row at the split boundary."""
    rng = np.random.default_rng({"normal": 11, "int_ties": 12, "all_zero": 13,
                                 "signed_zeros": 14}[kind])
    L_list = [16384, 16385, 16447, 20001, 2047, 65536, 99999] + [17000 + 3001 * i for i in range(17)]
    top_k = 2048
    ld = max(L_list)
    s = np.zeros((len(L_list), ld), np.float32)
    for i, L in enumerate(L_list):
        if kind == "normal":
            s[i, :L] = rng.standard_normal(L)
        elif kind == "int_ties":
            s[i, :L] = rng.integers(-5, 6, L)
        elif kind == "signed_zeros":
            s[i, :L] = np.where(rng.random(L) < 0.5, -0.0, 0.0)
            s[i, :L:97] = 1.0
    idx, n_sel = _select(s, L_list, top_k, 1)
    for i, L in enumerate(L_list):
        ref = oracle.topk(s[i, :L].astype(np.float64), top_k)
        assert np.array_equal(idx[i, : n_sel[i]], ref), f"L={L}"


@pytest.mark.parametrize("ties", [False, True])
def test_kpool_select_bit_exact(ties):
    rng = np.random.default_rng(7)
    L_list = [2050, 2051, 2052, 2053, 2055, 2056, 2100, 16, 40000]
    top_k, kp = 2048, 4
    ld = max(L // kp for L in L_list)
    s = np.zeros((len(L_list), ld), np.float32)
    for i, L in enumerate(L_list):
        n = L // kp
        s[i, :n] = rng.integers(0, 3, n) if ties else rng.standard_normal(n)
    idx, n_sel = _select(s, L_list, top_k, kp)
    for i, L in enumerate(L_list):
        ref = oracle.kpool_select(s[i, : L // kp].astype(np.float64), L, top_k, kp)
        assert np.array_equal(idx[i, : n_sel[i]], ref), f"L={L}"


# ------------------------------------------------------------ attention alone

@pytest.mark.parametrize("rope,dtype", [(64, "bf16"), (0, "bf16"), (64, "f32")])
def test_sparse_mla_on_given_selection(rope, dtype):
    """Attention over an arbitrary (unsorted) selection, several splits."""
    wl = workloads.small("attn", [6000, 300], top_k=2048, rope=rope, dtype=dtype)
    host = workloads.make(wl, "cpu")
    d = to_device(host)
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    width = dsa.dsa_index_row_width(sh)
    rng = np.random.default_rng(3)
    idx = np.full((2, width), -1, np.int32)
    sels = [rng.permutation(6000)[:2048].astype(np.int32), rng.permutation(300)[:77].astype(np.int32)]
    for i, s in enumerate(sels):
        idx[i, : len(s)] = s
    n_sel = np.array([len(s) for s in sels], np.int32)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_SPARSE_MLA)
    out = torch.empty((2, 64, 512), device="cuda")
    lse = torch.empty((2, 64), device="cuda")
    dsa.dsa_sparse_mla_attn(sh, b, d["q_abs"], d["cache"], torch.from_numpy(idx).cuda(),
                            torch.from_numpy(n_sel).cuda(), out, lse, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    for i, (r0, L) in enumerate([(0, 6000), (6000, 300)]):
        o_ref, l_ref = oracle.sparse_mla(host_f32(host["q_abs"][i]),
                                         host_f32(host["cache"][r0:r0 + L]), sels[i], wl.scale, 512)
        check_attention(out[i].cpu().numpy(), lse[i].cpu().numpy(), o_ref, l_ref, dtype)


def test_bad_index_sets_error_word_without_fault():
    """An index outside [0, L) is reported through the workspace error word and
    skipped; the context stays usable."""
    wl = workloads.small("bad", [100], top_k=64)
    host = workloads.make(wl, "cpu")
    d = to_device(host)
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    idx = torch.full((1, 64), -1, dtype=torch.int32, device="cuda")
    idx[0, :3] = torch.tensor([5, 100, 7], dtype=torch.int32)      # 100 is out of range
    n_sel = torch.tensor([3], dtype=torch.int32, device="cuda")
    ws = dsa.alloc_workspace(sh, b, dsa.OP_SPARSE_MLA)
    out = torch.empty((1, 64, 512), device="cuda")
    dsa.dsa_sparse_mla_attn(sh, b, d["q_abs"], d["cache"], idx, n_sel, out, None, ws)
    assert dsa.dsa_check_device_error(ws) == 1
    assert dsa.dsa_check_device_error(ws) == 0                     # cleared
    o_ref, l_ref = oracle.sparse_mla(host_f32(host["q_abs"][0]), host_f32(host["cache"]),
                                     np.array([5, 7], np.int32), wl.scale, 512)
    check_attention(out[0].cpu().numpy(), None, o_ref, l_ref, "bf16")
    torch.cuda.synchronize()


def test_inputs_written_by_the_previous_kernel_are_used():
    """Each entry point reads its inputs only once the kernel before it in the
    stream has completed: inputs that a kernel enqueued just before the call
    writes (over poisoned buffers) give exactly the results of the same inputs
    written long before."""
    wl = workloads.small("producer", [5000, 3000], top_k=512)
    d = to_device(workloads.make(wl, "cpu"))
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    ref_scores = run_scores(wl, d)
    ref = run_step(wl, d)
    fresh = {k: torch.full_like(d[k], 7.0) for k in ("q_idx", "k_idx", "q_abs", "w")}
    torch.cuda.synchronize()
    # the indexer right after the kernels that write its query, keys and weights
    ld = max(max(wl.kv_lens), 1)
    scores = torch.full((wl.n_q, ld), float("nan"), device="cuda")
    ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP)
    for k in ("q_idx", "k_idx", "w"):
        fresh[k].copy_(d[k])
    dsa.dsa_index_scores(sh, b, fresh["q_idx"], fresh["w"], fresh["k_idx"], scores, ld, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    got = scores.cpu().numpy()
    for q, L in enumerate(wl.q_nvis()):
        assert np.array_equal(got[q, :L], ref_scores[q, :L])
    # the attention right after the kernel that writes its absorbed query
    for t in fresh.values():
        t.fill_(7.0)
    idx = torch.from_numpy(ref[2]).cuda()
    n_sel = torch.from_numpy(ref[3]).cuda()
    out = torch.full((wl.n_q, wl.heads, wl.kv_lora), float("nan"), device="cuda")
    lse = torch.full((wl.n_q, wl.heads), float("nan"), device="cuda")
    torch.cuda.synchronize()
    fresh["q_abs"].copy_(d["q_abs"])
    dsa.dsa_sparse_mla_attn(sh, b, fresh["q_abs"], d["cache"], idx, n_sel, out, lse, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    assert np.array_equal(out.cpu().numpy(), ref[0])
    # the whole step right after the kernels that write every query input
    for t in fresh.values():
        t.fill_(7.0)
    torch.cuda.synchronize()
    for k in fresh:
        fresh[k].copy_(d[k])
    dsa.dsa_decode_step(sh, b, fresh["q_idx"], fresh["w"], fresh["k_idx"], fresh["q_abs"],
                        d["cache"], out, lse, None, None, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    assert np.array_equal(out.cpu().numpy(), ref[0])


def test_repeat_is_bit_identical():
    """Same inputs, same outputs, bit for bit (a race smoke test)."""
    wl = workloads.small("rep", [20000, 9000], top_k=2048)
    d = to_device(workloads.make(wl, "cpu"))
    a = run_step(wl, d)
    b = run_step(wl, d)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ------------------------------------------------------------ full-size workloads

def _full_sample(wl):
    """Queries checked element by element against the oracle at full size:
    every query of the decode batches, 64 evenly spaced queries of the prefill
    chunk (first and last included)."""
    if wl.n_q <= 64:
        return list(range(wl.n_q))
    return sorted({int(round(i * (wl.n_q - 1) / 63)) for i in range(64)})


FULL = ["glm52_decode_128k", "ragged_decode_64", "chunked_prefill_4096", "kpool_nope_1m"]


@pytest.mark.parametrize("name", FULL)
def test_full_size(name):
    """The full-size workloads in the launch configuration the benchmark times:
    for every sampled query the indexer scores (all of them), the selection and
    the attention output against the oracle.  The oracle attends over the rows
    the GPU selected (the same set as the oracle's own, up to near-ties, which
    check_selection allows), gathered on the host."""
    wl = workloads.named(name)
    d = workloads.make(wl, "cuda")
    out, lse, idx, n_sel = run_step(wl, d)
    scores = run_scores(wl, d)
    kv_off = np.concatenate([[0], np.cumsum(wl.kv_lens)])
    key_off = np.concatenate([[0], np.cumsum(wl.key_counts())])
    for q in _full_sample(wl):
        seq, L = int(d["q_seq"][q]), int(d["q_nvis"][q])
        r0, k0 = int(kv_off[seq]), int(key_off[seq])
        nk = L // wl.kpool
        keys = host_f32(d["k_idx"][k0:k0 + nk])
        qi, w = host_f32(d["q_idx"][q]), host_f32(d["w"][q])
        s = oracle.index_scores(qi, w, keys)
        ref = (oracle.topk(s, wl.top_k) if wl.kpool == 1
               else oracle.kpool_select(s, L, wl.top_k, wl.kpool))
        r = {"scores": s, "idx": ref, "L": L, "q": qi, "w": w, "keys": keys}
        check_scores(scores[q, :nk], r)
        sel = idx[q, : n_sel[q]]
        check_selection(sel, r, wl.top_k, wl.kpool)
        rows = host_f32(d["cache"][r0 + torch.from_numpy(sel.astype(np.int64)).to("cuda")])
        o_ref, l_ref = oracle.sparse_mla(host_f32(d["q_abs"][q]), rows,
                                         np.arange(len(sel), dtype=np.int32), wl.scale,
                                         wl.kv_lora)
        check_attention(out[q], lse[q], o_ref, l_ref, wl.dtype, label=f"full size {name}")
    # properties that hold for every query
    assert np.all(n_sel == np.array([min(L, wl.top_k) if wl.kpool == 1 else
                                     (L if L // 4 <= wl.top_k // 4 else wl.top_k + L % 4)
                                     for L in wl.q_nvis()]))
    assert np.all(np.isfinite(out))
    del d
    torch.cuda.empty_cache()
