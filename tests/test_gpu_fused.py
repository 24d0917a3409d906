"""The fused decode kernel (indexer scoring and top-k selection in one
cooperative launch) on the GPU.

Its selection must be bit-exact against the oracle's selection rule applied to
the GPU's own float32 scores (the standalone indexer computes the same bits),
identical to the two-launch path's, and within the parity bars of the oracle's
double-precision path.  Inputs cover one query spread over every CTA, mixed
dense and sparse rows, k-pool rows with tails, 16 queries, exact ties across
CTAs (duplicated keys; all-zero keys, whose candidates overflow the list
and take the histogram levels; signed zeros), and reuse of one workspace
across launches of different batches.
"""
import numpy as np
import pytest
import torch

import deepseek_sparse_attention_gb300 as dsa
import oracle
import workloads
from parity_util import (check_attention, check_selection, gpu_batch, gpu_shape, oracle_query,
                         to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dsa.load()
    oracle.build()


def _lens16():
    rng = np.random.default_rng(16)
    return [int(x) for x in rng.integers(1500, 40000, 16)]


FUSED = [
    workloads.small("one_query_all_ctas", [40000], top_k=2048, w_std=1 / 32 ** 0.5,
                    cache_scale=0.5),
    workloads.small("dense_and_sparse", [3000, 2049, 2048, 70000, 130, 9000], top_k=2048),
    workloads.small("kpool_tails", [100000, 9000, 2051, 8195, 8193], top_k=2048, kpool=4,
                    rope=0),
    workloads.small("batch_16", _lens16(), top_k=2048, seed=3),
    workloads.small("small_k", [20000, 5000, 64], top_k=64),
    # every sequence at the batch's bound
    workloads.small("uniform_4", [20000] * 4, top_k=2048, seed=5),
    workloads.small("uniform_kpool", [30000] * 3, top_k=2048, kpool=4, rope=0, seed=6),
]


def _step(wl, d, ws=None, flags=0):
    """The whole step; flags=dsa.FLAG_TWO_LAUNCH takes the two-launch path."""
    sh, b = gpu_shape(wl), gpu_batch(wl, d, flags)
    if ws is None:
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


TWO = dsa.FLAG_TWO_LAUNCH


def _gpu_scores(wl, d):
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_INDEX_SCORES)
    ld = max(max(wl.kv_lens) // wl.kpool, 1)
    scores = torch.full((wl.n_q, ld), float("nan"), device="cuda")
    dsa.dsa_index_scores(sh, b, d["q_idx"], d["w"], d["k_idx"], scores, ld, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    return scores.cpu().numpy()


def _rule_on(scores_row, L, wl):
    """The oracle's selection rule applied to given (float32) scores."""
    s = scores_row[: L // wl.kpool].astype(np.float64)
    if wl.kpool == 1:
        return oracle.topk(s, wl.top_k)
    return oracle.kpool_select(s, L, wl.top_k, wl.kpool)


def _check_exact(wl, host, d, idx, n_sel):
    sc = _gpu_scores(wl, d)
    width = idx.shape[1]
    for q in range(wl.n_q):
        L = int(host["q_nvis"][q])
        ref = _rule_on(sc[q], L, wl)
        assert n_sel[q] == len(ref), f"q={q} L={L}: n_sel {n_sel[q]} != {len(ref)}"
        assert np.array_equal(idx[q, : n_sel[q]], ref), f"q={q} L={L}"
        assert np.all(idx[q, n_sel[q]: width] == -1), f"q={q}: unused slots not cleared"


def _assert_eligible(wl, d):
    plan = dsa.dsa_plan(gpu_shape(wl), gpu_batch(wl, d), dsa.OP_DECODE_STEP)
    plan2 = dsa.dsa_plan(gpu_shape(wl), gpu_batch(wl, d, TWO), dsa.OP_DECODE_STEP)
    assert plan["kernel_launches"] < plan2["kernel_launches"], "fused path not taken"


@pytest.mark.parametrize("wl", FUSED, ids=lambda w: w.name)
def test_fused_selection_is_exact_and_matches_two_launch_path(wl):
    host = workloads.make(wl, "cpu")
    d = to_device(host)
    _assert_eligible(wl, d)
    out, lse, idx, n_sel = _step(wl, d)
    _check_exact(wl, host, d, idx, n_sel)
    out2, lse2, idx2, n_sel2 = _step(wl, d, flags=TWO)
    assert np.array_equal(idx, idx2) and np.array_equal(n_sel, n_sel2)
    # same selection, same attention kernels: identical outputs
    assert np.array_equal(out, out2, equal_nan=False)
    # against the oracle's own double-precision path, on a sample of queries
    for q in sorted({0, wl.n_q - 1, wl.n_q // 2}):
        r = oracle_query(wl, host, q)
        sel = idx[q, : n_sel[q]]
        check_selection(sel, r, wl.top_k, wl.kpool)
        o_ref, l_ref = oracle.sparse_mla(r["q_abs"], r["rows"], sel, wl.scale, wl.kv_lora)
        check_attention(out[q], lse[q], o_ref, l_ref, wl.dtype)


def test_fused_single_query_shorter_than_its_bounds():
    """One decode query whose sequence is shorter than the batch's bounds
    (max_kv_len, total_keys and total_rows of a cache with spare rows after
    it): the fused launch's CTAs guess their first key tiles from the bounds
    before the offsets are read, and here the guess is wrong for most of them
    -- those loads are drained and the real range issued.  The selection must
    equal the two-launch path's and the oracle rule's on the GPU scores."""
    wl = workloads.small("spare_rows", [5000], top_k=2048, w_std=1 / 32 ** 0.5, cache_scale=0.5)
    big = workloads.small("spare_rows_big", [9000], top_k=2048, w_std=1 / 32 ** 0.5,
                          cache_scale=0.5, seed=7)
    host = workloads.make(wl, "cpu")
    d = to_device(host)
    db = to_device(workloads.make(big, "cpu"))
    k_big = torch.cat([d["k_idx"], db["k_idx"][5000:]]).contiguous()
    c_big = torch.cat([d["cache"], db["cache"][5000:]]).contiguous()
    sh = gpu_shape(wl)
    width = dsa.dsa_index_row_width(sh)
    res = []
    for flags in (0, TWO):
        b = dsa.make_batch(d["row_off"], d["key_off"], d["q_off"], 1, 1, 9000, 9000, 9000, flags)
        ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP)
        out = torch.full((1, wl.heads, wl.kv_lora), float("nan"), device="cuda")
        lse = torch.full((1, wl.heads), float("nan"), device="cuda")
        idx = torch.full((1, width), -7, dtype=torch.int32, device="cuda")
        n_sel = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        for _ in range(2):                 # the workspace as the second launch finds it, too
            dsa.dsa_decode_step(sh, b, d["q_idx"], d["w"], k_big, d["q_abs"], c_big, out, lse,
                                idx, n_sel, ws)
            assert dsa.dsa_check_device_error(ws) == 0
        res.append((out.cpu().numpy(), idx.cpu().numpy(), n_sel.cpu().numpy()))
    b0 = dsa.make_batch(d["row_off"], d["key_off"], d["q_off"], 1, 1, 9000, 9000, 9000)
    assert dsa.dsa_plan(sh, b0, dsa.OP_DECODE_STEP)["kernel_launches"] == 3   # fused
    (out, idx, n_sel), (out2, idx2, n_sel2) = res
    assert np.array_equal(idx, idx2) and np.array_equal(n_sel, n_sel2)
    assert np.array_equal(out, out2)
    _check_exact(wl, host, d, idx, n_sel)
    # the standalone indexer guesses the same way: its scores under the loose
    # bounds equal those under the exact ones, bit for bit
    ws = dsa.alloc_workspace(sh, b0, dsa.OP_INDEX_SCORES)
    sc = torch.full((1, 9000), float("nan"), device="cuda")
    dsa.dsa_index_scores(sh, b0, d["q_idx"], d["w"], k_big, sc, 9000, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    assert np.array_equal(sc.cpu().numpy()[0, :5000], _gpu_scores(wl, d)[0, :5000])
    assert bool(torch.all(torch.isnan(sc[0, 5000:])))          # nothing past the sequence


def _tie_inputs(kind):
    wl = workloads.small(f"ties_{kind}", [30000, 2500, 9000], top_k=2048, seed=11)
    host = workloads.make(wl, "cpu")
    k = host["k_idx"]
    if kind == "duplicate_keys":
        rng = np.random.default_rng(5)
        pick = torch.from_numpy(rng.integers(0, 37, k.shape[0]))
        host["k_idx"] = k[pick].clone()
    elif kind == "zero_keys":
        host["k_idx"] = torch.zeros_like(k)
    elif kind == "signed_zeros":
        # negative weights: every relu'd head that is 0 gives -0.0 terms
        host["w"] = -host["w"].abs()
    return wl, host


@pytest.mark.parametrize("kind", ["duplicate_keys", "zero_keys", "signed_zeros"])
def test_fused_ties_across_ctas(kind):
    wl, host = _tie_inputs(kind)
    d = to_device(host)
    _assert_eligible(wl, d)
    _, _, idx, n_sel = _step(wl, d)
    _check_exact(wl, host, d, idx, n_sel)
    _, _, idx2, n_sel2 = _step(wl, d, flags=TWO)
    assert np.array_equal(idx, idx2) and np.array_equal(n_sel, n_sel2)
    if kind == "zero_keys":
        # every score ties: the lowest indices win
        for q in range(wl.n_q):
            L = int(host["q_nvis"][q])
            assert np.array_equal(idx[q, : n_sel[q]], np.arange(min(L, wl.top_k)))


def test_fused_workspace_reuse_across_batches():
    """Each launch leaves the shared selection state as the next one expects it
    (histograms cleared, the grid barrier at a whole number of rounds, the
    candidates' level-2 copy of the other launch parity cleared): one workspace
    serves consecutive launches of batches with different query counts."""
    wa = workloads.small("reuse_a", [40000, 5000], top_k=2048, seed=21)
    wb = workloads.small("reuse_b", [9000, 70000, 3000], top_k=512, seed=22)
    ha, hb = workloads.make(wa, "cpu"), workloads.make(wb, "cpu")
    da, db = to_device(ha), to_device(hb)
    wsa = dsa.alloc_workspace(gpu_shape(wa), gpu_batch(wa, da), dsa.OP_DECODE_STEP)
    wsb = dsa.alloc_workspace(gpu_shape(wb), gpu_batch(wb, db), dsa.OP_DECODE_STEP)
    ws = wsa if wsa.numel() >= wsb.numel() else wsb
    fresh_a = _step(wa, da)
    fresh_b = _step(wb, db)
    for _ in range(3):
        for wl, d, fresh in ((wa, da, fresh_a), (wb, db, fresh_b)):
            got = _step(wl, d, ws)
            for x, y in zip(got, fresh):
                assert np.array_equal(x, y)


@pytest.mark.parametrize("wl", [FUSED[0], FUSED[2],
                                workloads.small("twenty_queries", [9000] * 20, top_k=2048, seed=5)],
                         ids=lambda w: w.name)
def test_index_select_entry_matches_decode_step(wl):
    """dsa_index_select (steps 1 and 2 alone) writes the selection the whole
    step uses, on the fused path and (20 queries) on the two-launch path."""
    host = workloads.make(wl, "cpu")
    d = to_device(host)
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    _, _, idx_ref, n_ref = _step(wl, d)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_INDEX_SELECT)
    width = dsa.dsa_index_row_width(sh)
    idx = torch.full((wl.n_q, width), -7, dtype=torch.int32, device="cuda")
    n_sel = torch.full((wl.n_q,), -7, dtype=torch.int32, device="cuda")
    for _ in range(2):                       # the second call reuses the workspace state
        dsa.dsa_index_select(sh, b, d["q_idx"], d["w"], d["k_idx"], idx, n_sel, ws)
        assert dsa.dsa_check_device_error(ws) == 0
        assert np.array_equal(idx.cpu().numpy(), idx_ref)
        assert np.array_equal(n_sel.cpu().numpy(), n_ref)


def test_wait_budget_runs_out_and_the_workspace_recovers():
    """The fused launch's CTAs wait on one another at grid barriers, each wait
    bounded by the workspace's budget.  With a budget of 1 ns the waits give up
    (a CTA reaching a barrier before the last one arrives records a timeout and
    returns): the call still completes, dsa_check_device_error reports
    DSA_ERR_TIMEOUT and re-zeroes the selection state, and the next call on the
    same workspace, at the default budget, is exact.  No wait is unbounded, so
    nothing hangs."""
    wl = FUSED[0]
    host = workloads.make(wl, "cpu")
    d = to_device(host)
    _assert_eligible(wl, d)
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    ref = _step(wl, d)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP)
    width = dsa.dsa_index_row_width(sh)
    idx = torch.empty((wl.n_q, width), dtype=torch.int32, device="cuda")
    n_sel = torch.empty((wl.n_q,), dtype=torch.int32, device="cuda")
    codes = []
    for _ in range(5):              # the CTAs' arrivals spread over microseconds
        dsa.dsa_workspace_set_wait_budget(ws, 1)
        dsa.dsa_index_select(sh, b, d["q_idx"], d["w"], d["k_idx"], idx, n_sel, ws)
        codes.append(dsa.dsa_check_device_error(ws))
        if codes[-1] != 0:
            break
    assert codes[-1] == 3, f"no wait ran out: {codes}"          # a bounded wait gave up
    for _ in range(2):
        got = _step(wl, d, ws)
        for x, y in zip(got, ref):
            assert np.array_equal(x, y)
