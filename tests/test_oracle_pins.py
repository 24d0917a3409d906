"""Pins of the host oracle against what the pages and the mathematics fix.

Each test pins one oracle function to something other than itself: a value
printed on (or worked by hand from) a page, a closed form, a special case that
reduces to a library routine, or a brute-force property on tiny inputs.  The
rival-reading tests check that a plausible wrong reading of a page would be
caught.  CPU only.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- indexer score

def test_index_scores_hand_worked_example():
    """'GLM 5.2 in one C file', 'The Lightning Indexer': worked by hand."""
    rows = _table("index_score_hand.txt")
    q = np.array([[1, 2, 0], [3, -1, 2]], dtype=np.float32)
    w = np.array([0.5, -2.0], dtype=np.float32)
    keys = np.array([[float(x) for x in r[1:4]] for r in rows], dtype=np.float32)
    expect = np.array([float(r[4]) for r in rows])
    got = oracle.index_scores(q, w, keys)
    assert np.array_equal(got, expect)


def test_index_scores_planted_closed_form():
    """q_h = u for every head, w_h = 1/heads, k_t = a_t u  =>  s_t = relu(a_t) |u|^2."""
    rng = np.random.default_rng(1)
    heads, dim, n = 32, 128, 300
    u = rng.integers(-3, 4, size=dim).astype(np.float32)        # small ints: exact
    a = rng.integers(-20, 21, size=n).astype(np.float32) / 4.0
    q = np.tile(u, (heads, 1))
    w = np.full(heads, 1.0 / heads, dtype=np.float32)            # 1/32 exact in float
    keys = (a[:, None] * u[None, :]).astype(np.float32)
    got = oracle.index_scores(q, w, keys)
    expect = np.maximum(a.astype(np.float64), 0.0) * float(np.dot(u, u))
    np.testing.assert_allclose(got, expect, rtol=0, atol=1e-9)
    # and the selection is the k largest a_t (ties to the lower index)
    k = 40
    sel = oracle.topk(got, k)
    order = sorted(range(n), key=lambda t: (-max(a[t], 0.0), t))[:k]
    assert sel.tolist() == sorted(order)


def test_index_scores_positive_homogeneity():
    """Scaling w by c > 0 scales every score by c, so the selection is unchanged
    (why the page's positive factors 1/sqrt(128), 1/sqrt(32) may be dropped)."""
    rng = np.random.default_rng(2)
    q = rng.standard_normal((32, 128)).astype(np.float32)
    w = rng.standard_normal(32).astype(np.float32)
    keys = rng.standard_normal((500, 128)).astype(np.float32)
    s1 = oracle.index_scores(q, w, keys)
    c = np.float32(1.0 / (math.sqrt(128.0) * math.sqrt(32.0)))
    s2 = oracle.index_scores(q, (w * c).astype(np.float32), keys)
    np.testing.assert_allclose(s2, s1 * float(c), rtol=1e-6, atol=1e-12)
    assert oracle.topk(s1, 64).tolist() == oracle.topk(s2, 64).tolist()


def test_index_scores_key_permutation_equivariance():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((4, 16)).astype(np.float32)
    w = rng.standard_normal(4).astype(np.float32)
    keys = rng.standard_normal((50, 16)).astype(np.float32)
    perm = rng.permutation(50)
    np.testing.assert_array_equal(oracle.index_scores(q, w, keys)[perm],
                                  oracle.index_scores(q, w, keys[perm]))


# ---------------------------------------------------------------------- top-k

def _valid_selection(scores, sel, k):
    """Brute force: |S| = min(n, k) and every member beats every non-member under
    (score desc, index asc)."""
    n = len(scores)
    S = set(sel.tolist())
    if len(S) != min(n, k) or len(sel) != len(S):
        return False
    if list(sel) != sorted(sel):
        return False
    for i in S:
        for j in range(n):
            if j in S:
                continue
            if not (scores[i] > scores[j] or (scores[i] == scores[j] and i < j)):
                return False
    return True


@pytest.mark.parametrize("seed", range(20))
def test_topk_brute_force_with_ties(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 40))
    k = int(rng.integers(1, 12))
    scores = rng.integers(-3, 4, size=n).astype(np.float64)      # many exact ties
    sel = oracle.topk(scores, k)
    assert _valid_selection(scores, sel, k)


def test_topk_exhaustive_small():
    """Every score vector over {0,1,2}^5 and every k: brute-force validity."""
    for vals in itertools.product([0.0, 1.0, 2.0], repeat=5):
        s = np.array(vals)
        for k in range(1, 7):
            assert _valid_selection(s, oracle.topk(s, k), k)


def test_topk_all_equal_takes_lowest_indices():
    """Ties go to the lower index ('Add GLM-5.3-Flash support', router: ties by
    ascending index); the rival 'ties to the higher index' would give the top."""
    s = np.zeros(100)
    assert oracle.topk(s, 10).tolist() == list(range(10))


def test_topk_dense_when_n_le_k():
    """'GLM-5.x (glm-dsa, glm5next)', 'The sparse-attention path': top-k over
    n_kv <= k keeps every cell."""
    s = np.random.default_rng(4).standard_normal(2048)
    assert oracle.topk(s, 2048).tolist() == list(range(2048))
    assert oracle.topk(s[:17], 2048).tolist() == list(range(17))


def test_topk_exact_count_not_strict_threshold():
    """The page's scan keeps scores strictly above the k-th largest, which keeps
    at most k-1; the reading adopted keeps exactly k."""
    s = np.arange(10, dtype=np.float64)
    sel = oracle.topk(s, 4)
    assert sel.tolist() == [6, 7, 8, 9]
    strict = [t for t in range(10) if s[t] > np.sort(s)[::-1][3]]
    assert len(strict) == 3 and len(sel) == 4


# --------------------------------------------------------------------- k-pool

@pytest.mark.parametrize("row", _table("pool_arithmetic.txt"))
def test_kpool_count_table(row):
    L, k, kp, n_pool, tail, dense, n_sel = (int(x) for x in row[:7])
    assert L // kp == n_pool and L % kp == tail
    rng = np.random.default_rng(L)
    ps = rng.standard_normal(n_pool)
    sel = oracle.kpool_select(ps, L, k, kp)
    assert len(sel) == n_sel
    if dense:
        assert sel.tolist() == list(range(L))
    else:
        assert sel.tolist() == sorted(sel.tolist())
        # the tail is always attended and every pool is taken whole
        assert all(t in set(sel.tolist()) for t in range(n_pool * kp, L))
        body = [t for t in sel.tolist() if t < n_pool * kp]
        assert len(body) == k and all(body[i] // kp == body[i + 3] // kp
                                      for i in range(0, len(body), kp))


def test_kpool_planted_pools():
    """Pool scores planted so the kept pools are known: 16 tokens, top-k 8,
    pools of 4 ('GLM-5.3-Flash on WASTE', 'What is checked')."""
    ps = np.array([0.1, 3.0, -1.0, 2.0])
    sel = oracle.kpool_select(ps, 16, 8, 4)
    assert sel.tolist() == [4, 5, 6, 7, 12, 13, 14, 15]
    # 19 tokens: same pools plus the 3-token tail 16, 17, 18
    sel = oracle.kpool_select(ps, 19, 8, 4)
    assert sel.tolist() == [4, 5, 6, 7, 12, 13, 14, 15, 16, 17, 18]


def test_kpool_zero_scores_tie_to_lower_pool():
    """A pool whose every head scored negative lands at exactly 0 after the ReLU
    ('GLM-5.3-Flash on WASTE', k-pool flavour); among equal pools the lower
    index is kept."""
    ps = np.array([0.0, 0.0, 0.0, 5.0, 0.0])
    assert oracle.kpool_select(ps, 20, 8, 4).tolist() == [0, 1, 2, 3, 12, 13, 14, 15]


def test_kpool_one_is_token_mode():
    rng = np.random.default_rng(5)
    s = rng.standard_normal(3000)
    assert oracle.kpool_select(s, 3000, 2048, 1).tolist() == oracle.topk(s, 2048).tolist()


def test_kpool_equal_member_keys_gives_same_pools():
    """When a pool's four member keys all equal its pool key, token mode ranks the
    members exactly as pool mode ranks the pool."""
    rng = np.random.default_rng(6)
    q = rng.standard_normal((8, 16)).astype(np.float32)
    w = rng.standard_normal(8).astype(np.float32)
    pool_keys = rng.standard_normal((30, 16)).astype(np.float32)
    member_keys = np.repeat(pool_keys, 4, axis=0)
    ps = oracle.index_scores(q, w, pool_keys)
    ts = oracle.index_scores(q, w, member_keys)
    assert oracle.kpool_select(ps, 120, 32, 4).tolist() == oracle.topk(ts, 32).tolist()


# ----------------------------------------------------------------- attention

def test_attention_identical_rows_return_the_latent():
    rng = np.random.default_rng(7)
    row = rng.standard_normal(576).astype(np.float32)
    rows = np.tile(row, (10, 1))
    q = rng.standard_normal((64, 576)).astype(np.float32)
    out, lse = oracle.sparse_mla(q, rows, np.arange(10), 1 / 16, 512)
    np.testing.assert_allclose(out, np.tile(row[:512].astype(np.float64), (64, 1)), atol=1e-12)
    z = (q.astype(np.float64) @ row.astype(np.float64)) / 16
    np.testing.assert_allclose(lse, z + math.log(10), atol=1e-9)


def test_attention_zero_query_is_mean_latent():
    rng = np.random.default_rng(8)
    rows = rng.standard_normal((40, 576)).astype(np.float32)
    idx = np.array([3, 9, 17, 25, 39], dtype=np.int32)
    out, lse = oracle.sparse_mla(np.zeros((64, 576), np.float32), rows, idx, 1 / 16, 512)
    mean = rows[idx, :512].astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(out, np.tile(mean, (64, 1)), atol=1e-12)
    np.testing.assert_allclose(lse, math.log(5), atol=1e-12)


def test_attention_two_rows_sigmoid_pins_scale_1_over_16():
    """Two rows: p_1 = sigmoid(z_1 - z_2) with z = dot/16 ('GLM-5.x', 'The block':
    softmax scale 1/16, not 1/sqrt(576) nor 1/sqrt(512))."""
    width, dv = 576, 512
    q = np.zeros((1, width), np.float32)
    q[0, 0] = 8.0
    rows = np.zeros((2, width), np.float32)
    rows[0, 0], rows[0, 1] = 1.0, 1.0
    rows[1, 0], rows[1, 1] = -1.0, 3.0
    out, lse = oracle.sparse_mla(q, rows, np.array([0, 1]), 1 / 16, dv)
    # z_1 = 8/16 = 0.5, z_2 = -0.5
    p1 = 1.0 / (1.0 + math.exp(-1.0))
    assert out[0, 0] == pytest.approx(p1 * 1.0 + (1 - p1) * -1.0, abs=1e-14)
    assert out[0, 1] == pytest.approx(p1 * 1.0 + (1 - p1) * 3.0, abs=1e-14)
    assert lse[0] == pytest.approx(math.log(math.exp(0.5) + math.exp(-0.5)), abs=1e-14)
    # rival scales would give a visibly different weight
    for rival in (1 / math.sqrt(576), 1 / math.sqrt(512)):
        pr = 1.0 / (1.0 + math.exp(-16.0 * rival))
        assert abs((pr - (1 - pr)) - out[0, 0]) > 1e-3


def test_attention_rope_columns_score_but_never_enter_output():
    """576 = 512 latent + 64 rope: the rope part adds to the score, the value is
    the 512-wide latent only ('GLM 5.2 in one C file', MLA decode path)."""
    width, dv = 576, 512
    q = np.zeros((2, width), np.float32)
    q[:, 512] = 16.0                       # rope-only query
    rows = np.zeros((2, width), np.float32)
    rows[0, :512] = 1.0
    rows[1, :512] = 2.0
    rows[0, 512] = 1.0                     # z_1 = 1, z_2 = 0
    rows[1, 575] = 100.0                   # rope column the query does not read
    out, _ = oracle.sparse_mla(q, rows, np.array([0, 1]), 1 / 16, dv)
    assert out.shape == (2, 512)
    p1 = 1.0 / (1.0 + math.exp(-1.0))
    np.testing.assert_allclose(out, p1 * 1.0 + (1 - p1) * 2.0, atol=1e-14)


def test_attention_large_gap_selects_argmax_row():
    rng = np.random.default_rng(9)
    rows = rng.standard_normal((6, 64)).astype(np.float32)
    q = np.zeros((1, 64), np.float32)
    q[0] = rows[4] * 1000.0
    out, _ = oracle.sparse_mla(q, rows, np.arange(6), 1.0, 32)
    np.testing.assert_allclose(out[0], rows[4, :32], atol=1e-12)


def test_sparse_equals_dense_masked_brute_force():
    """The gather formulation equals dense attention with a -inf mask on every
    tiny case ('GLM-5.x', 'The sparse-attention path': a mask that starts fully
    masked and is unmasked at the selected positions)."""
    rng = np.random.default_rng(10)
    for L in (1, 2, 5, 17, 64):
        for k in (1, 3, 8):
            q = rng.standard_normal((4, 24)).astype(np.float32)
            rows = rng.standard_normal((L, 24)).astype(np.float32)
            scores = rng.standard_normal(L)
            sel = oracle.topk(scores, k)
            mask = np.zeros(L, np.uint8)
            mask[sel] = 1
            o1, l1 = oracle.sparse_mla(q, rows, sel, 0.3, 16)
            o2, l2 = oracle.dense_masked_mla(q, rows, mask, 0.3, 16)
            np.testing.assert_allclose(o1, o2, atol=1e-12)
            np.testing.assert_allclose(l1, l2, atol=1e-12)


def test_sparse_equals_dense_when_context_le_k():
    """'GLM 5.2 in one C file': below index_topk keys the indexer keeps all of
    them and attention is exactly dense."""
    rng = np.random.default_rng(11)
    L = 300
    q_idx = rng.standard_normal((32, 128)).astype(np.float32)
    w = rng.standard_normal(32).astype(np.float32)
    keys = rng.standard_normal((L, 128)).astype(np.float32)
    q = rng.standard_normal((64, 576)).astype(np.float32)
    rows = rng.standard_normal((L, 576)).astype(np.float32)
    r = oracle.decode_step(q_idx, w, keys, q, rows, L, 2048, 1, 1 / 16, 512)
    assert r["idx"].tolist() == list(range(L))
    o2, l2 = oracle.dense_masked_mla(q, rows, np.ones(L, np.uint8), 1 / 16, 512)
    np.testing.assert_allclose(r["out"], o2, atol=1e-12)
    np.testing.assert_allclose(r["lse"], l2, atol=1e-12)


def test_attention_row_permutation_invariance():
    rng = np.random.default_rng(12)
    rows = rng.standard_normal((30, 40)).astype(np.float32)
    q = rng.standard_normal((3, 40)).astype(np.float32)
    idx = np.array([1, 4, 9, 20, 29], dtype=np.int32)
    o1, l1 = oracle.sparse_mla(q, rows, idx, 0.2, 32)
    o2, l2 = oracle.sparse_mla(q, rows, idx[::-1].copy(), 0.2, 32)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_decode_step_kpool_nope_composition():
    """k-pool NoPE: scores over pool keys, 512 pools kept, tail appended, 512-wide
    rows that are both key and value ('Add GLM-5.3-Flash support': K and V are
    the same tensor)."""
    rng = np.random.default_rng(13)
    L, k, kp = 4 * 40 + 3, 32, 4
    q_idx = rng.standard_normal((32, 128)).astype(np.float32)
    w = rng.standard_normal(32).astype(np.float32)
    pkeys = rng.standard_normal((L // kp, 128)).astype(np.float32)
    q = rng.standard_normal((64, 512)).astype(np.float32)
    rows = rng.standard_normal((L, 512)).astype(np.float32)
    r = oracle.decode_step(q_idx, w, pkeys, q, rows, L, k, kp, 1 / 16, 512)
    pools = oracle.topk(oracle.index_scores(q_idx, w, pkeys), k // kp)
    expect = [4 * p + j for p in pools for j in range(4)] + [160, 161, 162]
    assert r["idx"].tolist() == expect
    o, l = oracle.sparse_mla(q, rows, np.array(expect, np.int32), 1 / 16, 512)
    np.testing.assert_array_equal(r["out"], o)


# ---------------------------------------------------------------- pool-key compression
# "GLM-5.x (glm-dsa, glm5next)", table "GLM-5.3-Flash", row "Pooled indexer":
# [key|gate] per cell, a softmax over the gates plus a per-slot position
# embedding compresses each pool.  "GLM-5.3-Flash on WASTE", "DeepSeek Sparse
# Attention, k-pool flavour": one 128-wide key per pool of 4 tokens.

def _cells(keys, gates):
    """[n_pools, kpool, dim] keys and gates -> [n_pools, kpool, 2*dim] cells."""
    return np.concatenate([keys, gates], axis=2).astype(np.float32)


def test_pool_compress_equal_logits_give_the_mean_key():
    """Equal gates and a zero embedding: every slot weighs 1/kpool."""
    rng = np.random.default_rng(40)
    keys = rng.integers(-8, 9, size=(5, 4, 128)).astype(np.float32)
    gates = np.tile(rng.standard_normal((5, 1, 128)).astype(np.float32), (1, 4, 1))
    out = oracle.pool_compress(_cells(keys, gates), np.zeros((4, 128), np.float32))
    np.testing.assert_allclose(out, keys.astype(np.float64).mean(axis=1), rtol=0, atol=1e-12)


def test_pool_compress_position_embedding_weights_the_slots():
    """Zero gates and pos_i = ln(i + 1): the weights are 1/10, 2/10, 3/10, 4/10
    in slot order -- the embedding sits inside the softmax, per slot."""
    keys = np.zeros((1, 4, 128), np.float32)
    keys[0, :, 0] = [10, 20, 30, 40]                    # channel 0: 1 + 4 + 9 + 16 = 30
    keys[0, :, 1] = [1, 0, 0, 0]                        # channel 1: the first weight, 0.1
    keys[0, :, 2] = [0, 0, 0, 1]                        # channel 2: the last weight, 0.4
    pos = np.tile(np.log(np.arange(1, 5, dtype=np.float64)).astype(np.float32)[:, None], (1, 128))
    out = oracle.pool_compress(_cells(keys, np.zeros_like(keys)), pos)
    np.testing.assert_allclose(out[0, :3], [30.0, 0.1, 0.4], rtol=1e-6)
    assert np.all(out[0, 3:] == 0.0)


def test_pool_compress_masked_slots_weigh_nothing():
    """A gate of -inf masks its slot: the key is the softmax over the other
    slots alone (equal gates: their mean), and a channel with every slot masked
    is 0 -- never NaN, which would sort above every score in the selection."""
    keys = np.zeros((1, 4, 128), np.float32)
    keys[0, :, :] = np.array([1.0, 2.0, 4.0, 8.0], np.float32)[:, None]
    gates = np.zeros((1, 4, 128), np.float32)
    gates[0, 0, :] = -np.inf                            # slot 0 masked everywhere
    gates[0, :, 7] = -np.inf                            # channel 7: every slot masked
    out = oracle.pool_compress(_cells(keys, gates), np.zeros((4, 128), np.float32))
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(np.delete(out[0], 7), (2 + 4 + 8) / 3.0, rtol=1e-15)
    assert out[0, 7] == 0.0


def test_pool_compress_dominant_gate_selects_its_key():
    rng = np.random.default_rng(41)
    keys = rng.standard_normal((3, 4, 128)).astype(np.float32)
    gates = rng.standard_normal((3, 4, 128)).astype(np.float32)
    gates[:, 2, :] += 60.0                              # slot 2 outweighs the others by e^55
    out = oracle.pool_compress(_cells(keys, gates), np.zeros((4, 128), np.float32))
    np.testing.assert_allclose(out, keys[:, 2, :].astype(np.float64), rtol=0, atol=1e-20)


def test_pool_compress_softmax_runs_over_the_slots_per_channel():
    """Keys all one: the output is one in every channel (the slot weights of a
    channel sum to one -- a softmax over channels would not give this); a shift
    of one channel's four gates leaves that channel unchanged."""
    rng = np.random.default_rng(42)
    gates = (3 * rng.standard_normal((4, 4, 128))).astype(np.float32)
    pos = rng.standard_normal((4, 128)).astype(np.float32)
    ones = oracle.pool_compress(_cells(np.ones((4, 4, 128), np.float32), gates), pos)
    np.testing.assert_allclose(ones, 1.0, rtol=0, atol=1e-14)
    keys = rng.standard_normal((4, 4, 128)).astype(np.float32)
    shift = np.zeros((4, 1, 128), np.float32)
    shift[:, :, 5] = 7.0                                # exact in float: small-integer shift
    a = oracle.pool_compress(_cells(keys, gates), pos)
    b = oracle.pool_compress(_cells(keys, np.round(gates) + shift), pos)
    c = oracle.pool_compress(_cells(keys, np.round(gates)), pos)
    np.testing.assert_allclose(b, c, rtol=1e-12, atol=1e-12)
    assert np.all(a.min() >= keys.min()) and np.all(a.max() <= keys.max())
    # each output lies between the smallest and largest key of its channel
    assert np.all(a >= keys.min(axis=1) - 1e-12) and np.all(a <= keys.max(axis=1) + 1e-12)


def test_pool_compress_slot_order_and_pool_independence():
    """Permuting the cells of a pool together with the embedding rows leaves the
    key unchanged; permuting the cells alone changes it (the embedding belongs to
    the slot); each pool depends only on its own cells."""
    rng = np.random.default_rng(43)
    keys = rng.standard_normal((6, 4, 128)).astype(np.float32)
    gates = rng.standard_normal((6, 4, 128)).astype(np.float32)
    pos = (2 * rng.standard_normal((4, 128))).astype(np.float32)
    base = oracle.pool_compress(_cells(keys, gates), pos)
    perm = np.array([2, 0, 3, 1])
    both = oracle.pool_compress(_cells(keys[:, perm], gates[:, perm]), pos[perm])
    np.testing.assert_allclose(both, base, rtol=1e-12, atol=1e-12)
    cells_only = oracle.pool_compress(_cells(keys[:, perm], gates[:, perm]), pos)
    assert np.abs(cells_only - base).max() > 1e-3
    alone = np.stack([oracle.pool_compress(_cells(keys[p:p + 1], gates[p:p + 1]), pos)[0]
                      for p in range(6)])
    assert np.array_equal(alone, base)


def test_pool_compress_rival_reading_fails():
    """The embedding added to the keys (after a softmax of the gates alone) is a
    plausible misreading: with zero gates it would give mean(key) + mean(pos)."""
    keys = np.zeros((1, 4, 128), np.float32)
    keys[0, :, 0] = [10, 20, 30, 40]
    pos = np.tile(np.log(np.arange(1, 5, dtype=np.float64)).astype(np.float32)[:, None], (1, 128))
    out = oracle.pool_compress(_cells(keys, np.zeros_like(keys)), pos)
    rival = keys[0, :, 0].astype(np.float64).mean() + pos[:, 0].astype(np.float64).mean()
    assert abs(out[0, 0] - rival) > 1.0


def test_pool_compress_rival_whole_block_softmax_fails():
    """"Add GLM-5.3-Flash support", "Tests": one softmax over the whole pool block
    instead of per key-dim is a rival reading that must disagree.  With all keys
    one, the per-dimension softmax returns one in every dimension; a softmax over
    the block's 4 x 128 logits would return each dimension's share of the block."""
    rng = np.random.default_rng(44)
    gates = rng.standard_normal((1, 4, 128)).astype(np.float32)
    pos = rng.standard_normal((4, 128)).astype(np.float32)
    ours = oracle.pool_compress(_cells(np.ones((1, 4, 128), np.float32), gates), pos)
    z = gates[0].astype(np.float64) + pos.astype(np.float64)
    block = np.exp(z - z.max()) / np.exp(z - z.max()).sum()        # the rival's weights
    rival = block.sum(axis=0)                                      # keys all one
    np.testing.assert_allclose(ours[0], 1.0, atol=1e-14)
    assert np.abs(rival - ours[0]).max() > 0.5


def test_new_pools_golden_table():
    for r in _table("new_pools.txt"):
        L, q_len, kpool, j0, j1 = (int(x) for x in r[:5])
        assert oracle.new_pools(L, q_len, kpool) == (j0, j1), r


def test_new_pools_brute_force():
    """A pool is made by the call iff its last token is one of the new tokens."""
    for kpool in (1, 2, 4, 5):
        for L in range(0, 23):
            for q_len in range(0, L + 1):
                made = [j for j in range(L // kpool)
                        if L - q_len <= kpool * j + kpool - 1 < L]
                j0, j1 = oracle.new_pools(L, q_len, kpool)
                assert list(range(j0, j1)) == made, (L, q_len, kpool)


# ---------------------------------------------------------------- indexer rope + Hadamard
# "GLM-5.x (glm-dsa, glm5next)", "The sparse-attention path": past top-k the
# indexer applies rope, then a Walsh-Hadamard rotation -- an orthonormal
# involution on both sides of the dot product -- before the keys are rounded;
# "The block", row "RoPE": NORM mode, base 8e6.

def test_hadamard_equals_the_library_matrix():
    """The special case a library computes: scipy's Sylvester Hadamard matrix,
    scaled by 1/sqrt(n), times the vector."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(50)
    for n in (1, 2, 4, 128):
        x = rng.standard_normal(n)
        ref = scipy_linalg.hadamard(n).astype(np.float64) @ x / math.sqrt(n)
        np.testing.assert_allclose(oracle.hadamard(x), ref, rtol=0, atol=1e-13)


def test_hadamard_closed_forms_and_involution():
    n = 128
    e0 = np.zeros(n); e0[0] = 1.0
    np.testing.assert_allclose(oracle.hadamard(e0), np.full(n, 1 / math.sqrt(n)), atol=1e-15)
    e1 = np.zeros(n); e1[1] = 1.0                       # column 1: +, -, +, -, ...
    np.testing.assert_allclose(oracle.hadamard(e1), np.tile([1, -1], n // 2) / math.sqrt(n),
                               atol=1e-15)
    np.testing.assert_allclose(oracle.hadamard(np.array([3.0, 1.0])),
                               [4 / math.sqrt(2), 2 / math.sqrt(2)], atol=1e-15)
    rng = np.random.default_rng(51)
    q, k = rng.standard_normal(n), rng.standard_normal(n)
    hq, hk = oracle.hadamard(q), oracle.hadamard(k)
    np.testing.assert_allclose(oracle.hadamard(hq), q, atol=1e-13)      # its own inverse
    assert abs(np.dot(hq, hk) - np.dot(q, k)) < 1e-12                  # dot products kept
    assert abs(np.linalg.norm(hq) - np.linalg.norm(q)) < 1e-12


def test_rope_closed_forms():
    d, base = 64, 8e6
    x = np.zeros(128, np.float32); x[0] = 1.0
    for pos in (0, 1, 5, 70000):
        out = oracle.rope(x, d, base, pos)                 # pair 0: theta = 1 rad per position
        np.testing.assert_allclose(out[:2], [math.cos(pos), math.sin(pos)], atol=1e-12)
        assert np.all(out[2:] == 0)
    i = d // 2 - 1                                         # the last pair: theta = base^(-(d-2)/d)
    x = np.zeros(128, np.float32); x[2 * i + 1] = 2.0
    a = 1000 * base ** (-(d - 2) / d)
    np.testing.assert_allclose(oracle.rope(x, d, base, 1000)[2 * i: 2 * i + 2],
                               [-2 * math.sin(a), 2 * math.cos(a)], atol=1e-12)
    rng = np.random.default_rng(52)
    y = rng.standard_normal(128).astype(np.float32)
    assert np.array_equal(oracle.rope(y, d, base, 0), y.astype(np.float64))      # position 0
    assert np.array_equal(oracle.rope(y, d, base, 12345)[d:], y[d:].astype(np.float64))


def test_rope_pairs_adjacent_dims_and_keeps_relative_position():
    """NORM mode rotates adjacent pairs (2i, 2i+1): e_1 moves into dim 0, not
    into dim 1 + d/2 (the rival NEOX pairing); the rotated dot product depends
    only on the position difference."""
    d, base = 64, 8e6
    e1 = np.zeros(128, np.float32); e1[1] = 1.0
    out = oracle.rope(e1, d, base, 3)
    np.testing.assert_allclose(out[:2], [-math.sin(3), math.cos(3)], atol=1e-12)
    assert np.all(out[2:] == 0)
    rng = np.random.default_rng(53)
    q, k = rng.standard_normal(128).astype(np.float32), rng.standard_normal(128).astype(np.float32)
    a = np.dot(oracle.rope(q, d, base, 900), oracle.rope(k, d, base, 850))
    b = np.dot(oracle.rope(q, d, base, 150), oracle.rope(k, d, base, 100))
    assert abs(a - b) < 1e-9


def test_index_prepare_is_rope_then_hadamard():
    """rope first, then the rotation: the order matters (the two do not commute)
    and the indexer score of prepared vectors equals that of roped ones -- the
    rotation cancels in exact arithmetic."""
    rng = np.random.default_rng(54)
    x = rng.standard_normal((6, 128)).astype(np.float32)
    pos = np.array([0, 1, 7, 4096, 65535, 1048575], np.int64)
    got = oracle.index_prepare(x, pos, 64, 8e6)
    for v in range(6):
        r = oracle.rope(x[v], 64, 8e6, int(pos[v]))
        np.testing.assert_allclose(got[v], oracle.hadamard(r), atol=1e-12)
        rival = oracle.rope(oracle.hadamard(x[v].astype(np.float64)).astype(np.float32), 64, 8e6,
                            int(pos[v]))
        if pos[v] != 0:
            assert np.abs(rival - got[v]).max() > 1e-3
    q = rng.standard_normal((32, 128)).astype(np.float32)
    w = rng.standard_normal(32).astype(np.float32)
    qp = oracle.index_prepare(q, np.full(32, 70000, np.int64), 64, 8e6)
    qr = np.stack([oracle.rope(q[h], 64, 8e6, 70000) for h in range(32)])
    kr = np.stack([oracle.rope(x[v], 64, 8e6, int(pos[v])) for v in range(6)])
    s_prep = np.maximum(got @ qp.T, 0) @ w.astype(np.float64)
    s_rope = np.maximum(kr @ qr.T, 0) @ w.astype(np.float64)
    np.testing.assert_allclose(s_prep, s_rope, rtol=1e-12, atol=1e-10)


# ---------------------------------------------------------------- absorption
# "GLM 5.2 in one C file", "Attention: Multi head Latent Attention With a Tiny
# KV Cache": the key up-projection is absorbed into the query and the value
# up-projection applied to the pooled latent -- "a reformulation, not an
# approximation".  "GLM-5.x (glm-dsa, glm5next)", "The block": 64 heads, head
# size 256 with n_rot 64 (so a 192-wide nope part), kv_lora 512.

H, NOPE, ROPE, KVL, VD = 64, 192, 64, 512, 256


def test_absorbed_scores_equal_explicit_decompression():
    """q_abs . [latent, rope key] equals q_nope . (W_UK latent) + q_rope . rope key
    for every head and row: the order of the two products is all that changes."""
    rng = np.random.default_rng(80)
    q = rng.standard_normal((H, NOPE + ROPE)).astype(np.float32)
    w_uk = (rng.standard_normal((H, NOPE, KVL)) / 16).astype(np.float32)
    rows = rng.standard_normal((7, KVL + ROPE)).astype(np.float32)
    q_abs = oracle.absorb_q(q, w_uk, ROPE)
    absorbed = q_abs @ rows.astype(np.float64).T                       # [H, 7]
    k_nope = np.einsum("hdi,ji->hjd", w_uk.astype(np.float64), rows[:, :KVL].astype(np.float64))
    explicit = (np.einsum("hd,hjd->hj", q[:, :NOPE].astype(np.float64), k_nope) +
                q[:, NOPE:].astype(np.float64) @ rows[:, KVL:].astype(np.float64).T)
    np.testing.assert_allclose(absorbed, explicit, rtol=1e-12, atol=1e-10)


def test_absorption_closed_forms():
    """W_UK = [I | 0] per head: the query's nope part lands in the first 192
    latent dims, the rest zero, the rope part copied behind the latent."""
    rng = np.random.default_rng(81)
    q = rng.standard_normal((H, NOPE + ROPE)).astype(np.float32)
    w = np.zeros((H, NOPE, KVL), np.float32)
    w[:, np.arange(NOPE), np.arange(NOPE)] = 1.0
    out = oracle.absorb_q(q, w, ROPE)
    assert np.array_equal(out[:, :NOPE], q[:, :NOPE].astype(np.float64))
    assert np.all(out[:, NOPE:KVL] == 0)
    assert np.array_equal(out[:, KVL:], q[:, NOPE:].astype(np.float64))


def test_up_projection_equals_explicit_values():
    """Attention over explicitly decompressed values (v_j = W_UV latent_j) equals
    the up-projection of the attention over the latents (linearity), with the
    attention itself from the oracle."""
    rng = np.random.default_rng(82)
    q_abs = (rng.standard_normal((H, KVL + ROPE)) * 0.2).astype(np.float32)
    rows = rng.standard_normal((9, KVL + ROPE)).astype(np.float32)
    w_uv = (rng.standard_normal((H, VD, KVL)) / 16).astype(np.float32)
    idx = np.arange(9, dtype=np.int32)
    o_lat, lse = oracle.sparse_mla(q_abs, rows, idx, 1 / 16, KVL)
    got = oracle.up_project(o_lat, w_uv)
    # the softmax weights from the oracle's lse: p_j = exp(z_j - lse)
    z = (q_abs.astype(np.float64) @ rows.astype(np.float64).T) / 16
    p = np.exp(z - lse[:, None])
    v = np.einsum("hvi,ji->hjv", w_uv.astype(np.float64), rows[:, :KVL].astype(np.float64))
    explicit = np.einsum("hj,hjv->hv", p, v)
    np.testing.assert_allclose(got, explicit, rtol=1e-10, atol=1e-10)
    sel = np.zeros((H, VD, KVL), np.float32)              # a selection matrix: out = o[perm]
    perm = rng.permutation(KVL)[:VD]
    sel[:, np.arange(VD), perm] = 1.0
    np.testing.assert_array_equal(oracle.up_project(o_lat, sel), o_lat[:, perm])


def test_oracle_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.sparse_mla(np.zeros((2, 8), np.float32), np.zeros((4, 8), np.float32),
                          np.array([0, 4]), 1.0, 8)        # index out of range
    with pytest.raises(ValueError):
        oracle.kpool_select(np.zeros(2), 8, 6, 4)          # top_k not a multiple of kpool


# ------------------------------------------------------------ descending order

def _order_by_repeated_max(scores, units):
    """Brute force: repeatedly take the unit of largest score, the lowest unit
    among equals (an O(n^2) scan, independent of any sort routine)."""
    left = list(units)
    out = []
    while left:
        best = left[0]
        for u in left[1:]:
            if scores[u] > scores[best] or (scores[u] == scores[best] and u < best):
                best = u
        out.append(best)
        left.remove(best)
    return out


@pytest.mark.parametrize("kpool,L,k", [(1, 300, 64), (1, 50, 64), (4, 403, 64), (4, 130, 64),
                                       (4, 2059, 2048), (1, 40, 8)])
def test_order_desc_matches_brute_force(kpool, L, k):
    rng = np.random.default_rng(L + kpool)
    n_units = L // kpool
    s = rng.integers(-3, 4, n_units).astype(np.float64)      # many ties
    sel = oracle.kpool_select(s, L, k, kpool) if kpool > 1 else oracle.topk(s, k)
    got = oracle.order_desc(s, sel, L, kpool)
    tail = L % kpool if kpool > 1 else 0
    units = [int(sel[i]) // kpool for i in range(0, len(sel) - tail, kpool)]
    want = []
    for u in _order_by_repeated_max(s, units):
        want += [u * kpool + r for r in range(kpool)]
    want += list(sel[len(sel) - tail:]) if tail else []
    assert got.tolist() == want
    assert sorted(got.tolist()) == sorted(sel.tolist())       # same set


def test_order_desc_invariants_and_rivals():
    """Scores never increase along the list; equal scores keep ascending units;
    the tail comes last.  Rival readings (ties to the higher unit; the tail
    first) give other lists."""
    rng = np.random.default_rng(77)
    L, kp = 4000 * 4 + 3, 4
    s = rng.integers(0, 6, L // kp).astype(np.float64)
    sel = oracle.kpool_select(s, L, 2048, kp)
    got = oracle.order_desc(s, sel, L, kp)
    body = got[:-3]
    units = body[::kp] // kp
    assert np.all(np.diff(s[units]) <= 0)
    for a, b in zip(units[:-1], units[1:]):
        if s[a] == s[b]:
            assert a < b
    for i in range(0, len(body), kp):                          # pools stay whole, ascending
        assert np.array_equal(body[i:i + kp], body[i] + np.arange(kp))
    assert np.array_equal(got[-3:], [L - 3, L - 2, L - 1])
    higher_first = sorted(units.tolist(), key=lambda u: (-s[u], -u))
    assert higher_first != units.tolist()
    assert not np.array_equal(np.concatenate([got[-3:], got[:-3]]), got)
