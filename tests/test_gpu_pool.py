"""GPU parity of the pool-key compression (dsa_pool_compress) against the host
oracle, through the C ABI: the pools each call writes, their values, the keys
it must leave alone, incremental decode against one bulk call, and the
compressed keys feeding the k-pool decode step."""
import numpy as np
import pytest
import torch

import deepseek_sparse_attention_gb300 as dsa
import oracle
import workloads
from parity_util import (check_attention, check_selection, gpu_batch, gpu_shape, host_f32,
                         oracle_query)

pytestmark = pytest.mark.gpu

KPOOL = 4
DIM = 128
SENTINEL = 7.0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dsa.load()
    oracle.build()


def _batch(kv_lens, q_lens, kpool=KPOOL, device="cuda"):
    """Offsets of sequences with kv_lens rows (cells), the last q_lens new, and
    room for floor(kv_len / kpool) pool keys each."""
    def prefix(xs):
        return torch.tensor(np.concatenate([[0], np.cumsum(xs)]), dtype=torch.int64, device=device)
    row_off, q_off = prefix(kv_lens), prefix(q_lens)
    key_off = prefix([L // kpool for L in kv_lens])
    b = dsa.make_batch(row_off, key_off, q_off, int(sum(q_lens)), max(q_lens), max(kv_lens),
                       int(sum(kv_lens)), int(sum(L // kpool for L in kv_lens)))
    return b, (row_off, key_off, q_off)


def _inputs(total_rows, dtype, seed, kpool=KPOOL):
    g = torch.Generator().manual_seed(seed)
    cells = torch.randn(total_rows, 2 * DIM, generator=g)
    cells[:, DIM:] *= 2.0                                   # gates spread the weights
    pos = 0.5 * torch.randn(kpool, DIM, generator=g)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return cells.to(tdt), pos.float()


def _compress(kv_lens, q_lens, cells, pos, pool_keys, dtype, kpool=KPOOL):
    sh = dsa.make_shape(kpool=kpool, rope_dim=0, dtype=dtype)
    b, keep = _batch(kv_lens, q_lens, kpool)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_POOL_COMPRESS)
    dsa.dsa_pool_compress(sh, b, cells, pos, pool_keys, ws)
    return dsa.dsa_check_device_error(ws)


def _check_pools(got, ref, keys_max, dtype):
    """float32 arithmetic, then rounded to bf16 (8 significant bits: at most
    half an ulp, 2^-8 of the value), plus the float32 error of a convex
    combination of keys bounded by keys_max."""
    err = np.abs(got.astype(np.float64) - ref)
    if dtype == "bf16":
        bound = 2.0 ** -8 * np.abs(ref) * 1.001 + 4e-6 * keys_max + 1e-30
    else:
        bound = 2e-6 * np.abs(ref) + 4e-6 * keys_max + 1e-30
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} of {bad.size} off; worst {err.max():.3e}"


CASES = [
    # (kv_len, q_len): decode steps that do and do not complete a pool, chunks
    # that complete some, a whole prompt, a prompt shorter than one pool
    [(4, 1), (5, 1), (8, 1), (10, 3), (11, 2), (12, 4), (4096, 4096), (3, 3), (9000, 517),
     (131, 131), (20000, 1)],
]


@pytest.mark.parametrize("kpool", [4, 2])          # 4: the unrolled kernel; 2: the general one
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", CASES, ids=["ragged"])
def test_pool_compress_matches_oracle(dtype, case, kpool):
    KPOOL = kpool
    kv_lens, q_lens = [c[0] for c in case], [c[1] for c in case]
    total_rows, total_keys = sum(kv_lens), sum(L // KPOOL for L in kv_lens)
    cells, pos = _inputs(total_rows, dtype, seed=5, kpool=KPOOL)
    tdt = cells.dtype
    pool_keys = torch.full((total_keys, DIM), SENTINEL, dtype=tdt, device="cuda")
    assert _compress(kv_lens, q_lens, cells.cuda(), pos.cuda(), pool_keys, dtype, KPOOL) == 0
    got = host_f32(pool_keys)
    cf, pf = host_f32(cells), host_f32(pos)
    r0 = k0 = 0
    for L, q in zip(kv_lens, q_lens):
        j0, j1 = oracle.new_pools(L, q, KPOOL)
        n_keys = L // KPOOL
        written = np.zeros(n_keys, bool)
        written[j0:j1] = True
        if j1 > j0:
            pools = cf[r0 + KPOOL * j0: r0 + KPOOL * j1].reshape(j1 - j0, KPOOL, 2 * DIM)
            ref = oracle.pool_compress(pools, pf)
            keys_max = np.abs(pools[:, :, :DIM]).max(axis=1)
            _check_pools(got[k0 + j0: k0 + j1], ref, keys_max, dtype)
        # every other pool key of the sequence is left as it was
        assert np.all(got[k0: k0 + n_keys][~written] == SENTINEL), (L, q)
        r0 += L
        k0 += n_keys


@pytest.mark.parametrize("kpool", [4, 2])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_masked_gates_match_oracle(dtype, kpool):
    """Gates of -inf (masked slots), in some channels every slot of a pool:
    the masked slots weigh 0 and an all-masked channel gives 0, as the oracle."""
    L = 64 * kpool
    cells, pos = _inputs(L, dtype, seed=9, kpool=kpool)
    c = cells.float()
    g = torch.Generator().manual_seed(10)
    mask = torch.rand(L, DIM, generator=g) < 0.4
    c[:, DIM:][mask] = float("-inf")
    c[: kpool * 8, DIM + 3] = float("-inf")              # channel 3 of the first 8 pools
    cells = c.to(cells.dtype)
    pool_keys = torch.full((L // kpool, DIM), SENTINEL, dtype=cells.dtype, device="cuda")
    assert _compress([L], [L], cells.cuda(), pos.cuda(), pool_keys, dtype, kpool) == 0
    got = host_f32(pool_keys)
    pools = host_f32(cells).reshape(L // kpool, kpool, 2 * DIM)
    ref = oracle.pool_compress(pools, host_f32(pos))
    assert np.all(np.isfinite(got)) and np.all(got[:8, 3] == 0.0)
    _check_pools(got, ref, np.abs(pools[:, :, :DIM]).max(axis=1), dtype)


def test_incremental_decode_equals_one_bulk_call():
    """A prompt of 4093 tokens, then seven decode steps (4094 .. 4100 tokens):
    the pool keys made one step at a time equal, bit for bit, those of one call
    over all 4100 tokens (each key is one pool's arithmetic either way)."""
    L0, steps = 4093, 7
    Lf = L0 + steps
    cells, pos = _inputs(Lf, "bf16", seed=6)
    cells, pos = cells.cuda(), pos.cuda()
    inc = torch.full((Lf // KPOOL, DIM), SENTINEL, dtype=torch.bfloat16, device="cuda")
    # the prompt: its rows are the first L0 cells; key capacity for its pools
    assert _compress([L0], [L0], cells[:L0], pos, inc[: L0 // KPOOL], "bf16") == 0
    for L in range(L0 + 1, Lf + 1):
        # the sequence now has L rows; only the new token's pool may be made
        assert _compress([L], [1], cells[:L], pos, inc[: L // KPOOL], "bf16") == 0
    bulk = torch.full_like(inc, SENTINEL)
    assert _compress([Lf], [Lf], cells, pos, bulk, "bf16") == 0
    assert torch.equal(inc, bulk)


def test_compressed_keys_feed_the_kpool_decode_step():
    """Pool keys compressed on the GPU are the k_idx of a k-pool NoPE decode
    step; the oracle scores the same (host-copied) keys."""
    kv_lens = [9000, 20001, 2055]
    wl = workloads.small("pool_feed", kv_lens, top_k=2048, kpool=KPOOL, rope=0, seed=12)
    host = workloads.make(wl, "cpu")
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    cells, pos = _inputs(sum(kv_lens), "bf16", seed=7)
    k_idx = torch.zeros((sum(L // KPOOL for L in kv_lens), DIM), dtype=torch.bfloat16,
                        device="cuda")
    assert _compress(kv_lens, kv_lens, cells.cuda(), pos.cuda(), k_idx, "bf16") == 0
    sh = gpu_shape(wl)
    d["k_idx"] = k_idx
    b = gpu_batch(wl, d)
    ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP)
    width = dsa.dsa_index_row_width(sh)
    out = torch.empty((wl.n_q, wl.heads, wl.kv_lora), device="cuda")
    lse = torch.empty((wl.n_q, wl.heads), device="cuda")
    idx = torch.full((wl.n_q, width), -7, dtype=torch.int32, device="cuda")
    n_sel = torch.zeros(wl.n_q, dtype=torch.int32, device="cuda")
    dsa.dsa_decode_step(sh, b, d["q_idx"], d["w"], k_idx, d["q_abs"], d["cache"], out, lse, idx,
                        n_sel, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    host["k_idx"] = k_idx.cpu()
    out, lse, idx, n_sel = out.cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy(), n_sel.cpu().numpy()
    for q in range(wl.n_q):
        r = oracle_query(wl, host, q)
        sel = idx[q, : n_sel[q]]
        check_selection(sel, r, wl.top_k, wl.kpool)
        o_ref, l_ref = oracle.sparse_mla(r["q_abs"], r["rows"], sel, wl.scale, wl.kv_lora)
        check_attention(out[q], lse[q], o_ref, l_ref, wl.dtype)


def test_bad_offsets_set_the_error_word():
    """A sequence whose pool-key range is too short for its rows is skipped and
    reported; the others are compressed."""
    kv_lens, q_lens = [16, 16], [16, 16]
    cells, pos = _inputs(32, "bf16", seed=8)
    sh = dsa.make_shape(kpool=KPOOL, rope_dim=0)
    row_off = torch.tensor([0, 16, 32], dtype=torch.int64, device="cuda")
    q_off = torch.tensor([0, 16, 32], dtype=torch.int64, device="cuda")
    key_off = torch.tensor([0, 2, 6], dtype=torch.int64, device="cuda")   # sequence 0: 2 < 4 keys
    b = dsa.make_batch(row_off, key_off, q_off, 32, 16, 16, 32, 6)
    pool_keys = torch.full((6, DIM), SENTINEL, dtype=torch.bfloat16, device="cuda")
    ws = dsa.alloc_workspace(sh, b, dsa.OP_POOL_COMPRESS)
    dsa.dsa_pool_compress(sh, b, cells.cuda(), pos.cuda(), pool_keys, ws)
    assert dsa.dsa_check_device_error(ws) == 2                      # a bad batch
    got = host_f32(pool_keys)
    assert np.all(got[:2] == SENTINEL)
    ref = oracle.pool_compress(host_f32(cells)[16:32].reshape(4, KPOOL, 2 * DIM), host_f32(pos))
    _check_pools(got[2:6], ref, np.abs(host_f32(cells)[16:32, :DIM]).reshape(4, KPOOL, DIM).max(1),
                 "bf16")
