"""The C-ABI library loads, exports every symbol its header declares, and
rejects bad arguments on the host before touching a device.  CPU only."""
import ctypes
import os
import re

import pytest
import torch

import deepseek_sparse_attention_gb300 as dsa
from deepseek_sparse_attention_gb300 import build as dsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dsa_build.build()
    return dsa.load()


def _declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(dsa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("dsa_index_scores", "dsa_topk_select", "dsa_sparse_mla_attn", "dsa_decode_step",
              "dsa_workspace_size", "dsa_check_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert missing == []


def test_version_and_row_width(lib):
    assert dsa.dsa_version() == 2
    assert dsa.dsa_index_row_width(dsa.make_shape(kpool=1)) == 2048
    assert dsa.dsa_index_row_width(dsa.make_shape(kpool=4)) == 2051
    assert dsa.dsa_index_row_width(dsa.make_shape(heads=32)) == -1   # unsupported geometry


def _batch(n_seq=1, n_q=1, max_q=1, max_kv=4096, flags=0):
    b = dsa.Batch(n_seq, n_q, max_q, flags, max_kv, max_kv, max_kv, ctypes.c_void_p(16),
                  ctypes.c_void_p(16), ctypes.c_void_p(16))
    return b


def _size(shape, batch, op):
    n = ctypes.c_size_t(0)
    rc = dsa.load().dsa_workspace_size(ctypes.byref(shape), ctypes.byref(batch), op,
                                       ctypes.byref(n))
    return rc, n.value


def test_workspace_sizes(lib):
    sh = dsa.make_shape()
    rc, n = _size(sh, _batch(max_kv=131072), dsa.OP_DECODE_STEP)
    assert rc == 0
    # header + scores (131072 floats) + one index row + n_sel, 256-byte aligned
    assert n >= 256 + 131072 * 4 + 2048 * 4 + 4 and n % 256 == 0
    rc, n = _size(sh, _batch(), dsa.OP_INDEX_SCORES)
    assert rc == 0 and n >= 256 and n % 256 == 0
    rc, n = _size(sh, _batch(), dsa.OP_TOPK_SELECT)
    assert rc == 0 and n == 256
    rc, n_sel = _size(sh, _batch(max_kv=131072), dsa.OP_INDEX_SELECT)
    rc2, n_step = _size(sh, _batch(max_kv=131072), dsa.OP_DECODE_STEP)
    # everything the decode step needs but the attention scratch; the fixed
    # selection state of the fused launch comes first
    assert rc == 0 and rc2 == 0 and n_sel % 256 == 0
    assert 256 + 131072 * 4 <= n_sel <= n_step
    assert n_sel >= 256 + 16 * 25604 * 4 + 16 * 256 * 8          # DSA_WS_ZERO_BYTES of dsa.h
    rc, n = _size(sh, _batch(), dsa.OP_POOL_COMPRESS)     # the header: the error word
    assert rc == 0 and n == 256
    rc, n = _size(sh, _batch(), dsa.OP_PROJECT)            # the header: the error word
    assert rc == 0 and n == 256
    # the host-fed step: the step's workspace, then the staged query inputs
    # (8 KB of indexer queries, 128 B of weights, 72 KB of absorbed queries)
    rc, n_host = _size(sh, _batch(max_kv=131072), dsa.OP_DECODE_STEP_HOST)
    assert rc == 0 and n_host % 256 == 0
    assert n_host >= n_step + 32 * 128 * 2 + 32 * 4 + 64 * 576 * 2
    rc, _ = _size(sh, _batch(), 8)
    assert rc == 1
    # the single-step entry points keep their scratch clear of the zeroed prefix
    rc, n_idx = _size(sh, _batch(), dsa.OP_INDEX_SCORES)
    assert n_idx >= 256 + 16 * 25604 * 4 + 16 * 256 * 8


@pytest.mark.parametrize("field,value,code", [
    ("heads", 32, 2), ("idx_dim", 64, 2), ("kv_lora", 256, 2), ("rope_dim", 32, 2),
    ("top_k", 0, 1), ("kpool", 0, 1), ("scale", float("nan"), 1), ("scale", -1.0, 1),
    ("dtype", 7, 1),
])
def test_shape_validation(lib, field, value, code):
    sh = dsa.make_shape(kpool=1)
    setattr(sh, field, value)
    rc, _ = _size(sh, _batch(), dsa.OP_DECODE_STEP)
    assert rc == code


def test_topk_not_multiple_of_kpool_rejected(lib):
    sh = dsa.make_shape(top_k=2046, kpool=4)
    assert _size(sh, _batch(), dsa.OP_DECODE_STEP)[0] == 1


def test_entry_points_reject_before_enqueue(lib):
    """Each call below is malformed; it must return its status without any CUDA
    call (there is no device here, so an enqueue would surface as DSA_ERR_CUDA)."""
    sh = dsa.make_shape()
    P = ctypes.c_void_p
    good = P(256)
    b = _batch()
    assert lib.dsa_index_scores(None, ctypes.byref(b), good, good, good, good, 4096, good, 256,
                                None) == 1
    assert lib.dsa_index_scores(ctypes.byref(sh), ctypes.byref(b), None, good, good, good, 4096,
                                good, 256, None) == 1
    assert lib.dsa_index_scores(ctypes.byref(sh), ctypes.byref(b), good, good, good, good, 100,
                                good, 256, None) == 1          # ld too small
    assert lib.dsa_index_scores(ctypes.byref(sh), ctypes.byref(b), good, good, good, good, 4096,
                                None, 256, None) == 3          # no workspace
    assert lib.dsa_index_scores(ctypes.byref(sh), ctypes.byref(b), good, good, good, good, 4096,
                                P(264), 256, None) == 3        # misaligned workspace
    assert lib.dsa_index_scores(ctypes.byref(sh), ctypes.byref(b), P(258), good, good, good,
                                4096, good, 256, None) == 1    # misaligned tensor
    bad = _batch(max_q=2, max_kv=1)
    assert lib.dsa_topk_select(ctypes.byref(sh), ctypes.byref(bad), good, 4096, good, good, good,
                               256, None) == 1
    big = _batch(max_kv=1 << 31)
    assert lib.dsa_sparse_mla_attn(ctypes.byref(sh), ctypes.byref(big), good, good, good, good,
                                   good, None, good, 1 << 20, None) == 2
    assert lib.dsa_decode_step(ctypes.byref(sh), ctypes.byref(b), good, good, good, good, good,
                               good, None, None, None, good, 16, None) == 3   # ws too small
    # a NULL workspace reads the no-allocation scratch array: a CUDA call,
    # which fails on a machine without a device
    if not torch.cuda.is_available():
        assert lib.dsa_check_device_error(None, 0, None, None) == 4
    assert lib.dsa_check_device_error(P(256), 16, None, None) == 3   # smaller than the header


def test_flags_validation(lib):
    """Unknown flag bits are malformed; the dense switch leaves the selection
    entry points nothing to do and takes no selection outputs in the step."""
    P = ctypes.c_void_p
    good = P(256)
    sh = dsa.make_shape()
    assert _size(sh, _batch(flags=0x8), dsa.OP_DECODE_STEP)[0] == 1
    assert _size(sh, _batch(flags=0x7), dsa.OP_DECODE_STEP)[0] == 0
    dense = _batch(flags=dsa.FLAG_DENSE)
    assert lib.dsa_topk_select(ctypes.byref(sh), ctypes.byref(dense), good, 4096, good, good,
                               good, 256, None) == 1
    assert lib.dsa_index_select(ctypes.byref(sh), ctypes.byref(dense), good, good, good, good,
                                good, good, 1 << 30, None) == 1
    # the step with the dense switch: selection outputs must be NULL ...
    assert lib.dsa_decode_step(ctypes.byref(sh), ctypes.byref(dense), None, None, None, good,
                               good, good, None, good, None, good, 1 << 30, None) == 1
    # ... and the indexer inputs may be (the workspace check comes next)
    assert lib.dsa_decode_step(ctypes.byref(sh), ctypes.byref(dense), None, None, None, good,
                               good, good, None, None, None, good, 16, None) == 3
    # descending order sorts at most 16384 units per query
    big_k = dsa.make_shape(top_k=32768)
    assert _size(big_k, _batch(flags=dsa.FLAG_DESC_ORDER), dsa.OP_DECODE_STEP)[0] == 0
    assert lib.dsa_topk_select(ctypes.byref(big_k), ctypes.byref(_batch(flags=dsa.FLAG_DESC_ORDER)),
                               good, 4096, good, good, good, 256, None) == 2


def test_noalloc_checks_everything_before_enqueue(lib):
    """dsa_decode_step_noalloc validates its arguments before it clears its
    scratch, and a batch without queries enqueues nothing (no device here: any
    CUDA call would surface as DSA_ERR_CUDA)."""
    P = ctypes.c_void_p
    good = P(256)
    sh = dsa.make_shape()
    f = lib.dsa_decode_step_noalloc
    b = _batch()
    assert f(ctypes.byref(sh), ctypes.byref(b), good, good, good, good, good, P(260), None, None,
             None, None) == 1                                    # misaligned output
    assert f(ctypes.byref(sh), ctypes.byref(b), good, good, good, good, good, good, None, P(258),
             None, None) == 1                                    # misaligned selection
    assert f(ctypes.byref(sh), ctypes.byref(_batch(flags=0x10)), good, good, good, good, good,
             good, None, None, None, None) == 1                  # unknown flag
    empty = _batch(n_q=0, max_q=0)
    assert f(ctypes.byref(sh), ctypes.byref(empty), None, None, None, None, None, None, None,
             None, None, None) == 0


def test_pool_compress_rejects_before_enqueue(lib):
    """dsa_pool_compress: token mode has no pools, and the usual argument,
    alignment and workspace checks run before anything is enqueued."""
    P = ctypes.c_void_p
    good = P(256)
    b = _batch()
    sh1, sh4 = dsa.make_shape(kpool=1), dsa.make_shape(kpool=4, rope_dim=0)
    f = lib.dsa_pool_compress
    assert f(ctypes.byref(sh1), ctypes.byref(b), good, good, good, good, 256, None) == 1
    assert f(ctypes.byref(sh4), ctypes.byref(b), None, good, good, good, 256, None) == 1
    assert f(ctypes.byref(sh4), ctypes.byref(b), good, P(260), good, good, 256, None) == 1
    assert f(ctypes.byref(sh4), ctypes.byref(b), good, good, good, good, 16, None) == 3
    assert f(ctypes.byref(sh4), ctypes.byref(b), good, good, good, P(264), 256, None) == 3
    assert f(ctypes.byref(sh4), ctypes.byref(_batch(max_q=2, max_kv=1)), good, good, good, good,
             256, None) == 1
    plan = dsa.dsa_plan(sh4, b, dsa.OP_POOL_COMPRESS)
    assert plan["kernel_launches"] == 1


def test_index_prepare_rejects_before_enqueue(lib):
    P = ctypes.c_void_p
    good = P(256)
    sh = dsa.make_shape()
    f = lib.dsa_index_prepare
    assert f(ctypes.byref(sh), 4, good, good, 63, 8e6, good, None) == 1      # odd rope width
    assert f(ctypes.byref(sh), 4, good, good, 130, 8e6, good, None) == 1     # wider than a head
    assert f(ctypes.byref(sh), 4, good, good, 64, 0.0, good, None) == 1      # base must be > 0
    assert f(ctypes.byref(sh), 4, good, None, 64, 8e6, good, None) == 1      # rope needs positions
    assert f(ctypes.byref(sh), 4, P(260), good, 64, 8e6, good, None) == 1    # misaligned x
    assert f(ctypes.byref(sh), -1, good, good, 64, 8e6, good, None) == 1
    assert f(ctypes.byref(sh), 0, None, None, 0, 8e6, None, None) == 0       # nothing to do


@pytest.mark.parametrize("name,launches,splits,rows_per_split", [
    # decode of one query: the fused indexer + selection, 32 one-tile attention
    # splits (one wave of CTAs), the split merge
    ("glm52_decode_128k", 3, 32, 64),
    # 64 decode queries: the indexer, the selection, the attention with two
    # splits per query merged inside its launch by a CTA pair
    ("ragged_decode_64", 3, 2, 1024),
    # a prefill chunk: the indexer's group plan and the indexer, the selection,
    # one attention split per query (no merge)
    ("chunked_prefill_4096", 4, 1, 2048),
    # four 1M-token k-pool decode queries: fused, 16 splits of two tiles over
    # the 2048 rows of the 512 selected pools and one more split for the tail
    # of up to 3 rows, merge
    ("kpool_nope_1m", 3, 17, 128),
])
def test_plan_of_the_benchmark_workloads(lib, name, launches, splits, rows_per_split):
    """The host-side plan (launch count, attention splits) of each benchmark
    workload, from the batch's host scalars alone."""
    import workloads
    wl = workloads.named(name)
    sh = dsa.make_shape(wl.idx_heads, wl.idx_dim, wl.heads, wl.kv_lora, wl.rope, wl.top_k,
                        wl.kpool, wl.scale, wl.dtype)
    P = ctypes.c_void_p(16)
    b = dsa.Batch(len(wl.kv_lens), wl.n_q, max(wl.q_lens), 0, max(wl.kv_lens), sum(wl.kv_lens),
                  sum(wl.key_counts()), P, P, P)
    plan = dsa.dsa_plan(sh, b, dsa.OP_DECODE_STEP)
    assert plan == {"kernel_launches": launches, "attn_splits": splits,
                    "attn_rows_per_split": rows_per_split}
    assert splits * rows_per_split >= min(max(wl.kv_lens), dsa.dsa_index_row_width(sh))
    # the two-launch plan adds the indexer's own launch where the fused one
    # applied; descending order one more; the dense switch only attends
    b.flags = dsa.FLAG_TWO_LAUNCH
    two = dsa.dsa_plan(sh, b, dsa.OP_DECODE_STEP)["kernel_launches"]
    b.flags = dsa.FLAG_DESC_ORDER
    desc = dsa.dsa_plan(sh, b, dsa.OP_DECODE_STEP)["kernel_launches"]
    assert desc == two + 1 and two >= launches
    b.flags = dsa.FLAG_DENSE
    dense = dsa.dsa_plan(sh, b, dsa.OP_DECODE_STEP)
    assert dense["attn_splits"] * dense["attn_rows_per_split"] >= max(wl.kv_lens)
    assert dense["kernel_launches"] == (2 if dense["attn_splits"] > 2 else 1)


def test_projections_reject_before_enqueue(lib):
    """dsa_absorb_q / dsa_up_project: widths (no-rope part a multiple of 64,
    value width of 128, at most 512), pointers, alignment and the workspace are
    checked before anything is enqueued."""
    P = ctypes.c_void_p
    good = P(256)
    sh = dsa.make_shape()
    fa, fu = lib.dsa_absorb_q, lib.dsa_up_project
    assert fa(ctypes.byref(sh), 4, 100, good, good, good, good, 256, None) == 1     # nope % 64
    assert fa(ctypes.byref(sh), 4, 576, good, good, good, good, 256, None) == 2     # > 512
    assert fa(ctypes.byref(sh), 4, 192, None, good, good, good, 256, None) == 1
    assert fa(ctypes.byref(sh), 4, 192, good, P(264), good, good, 256, None) == 1   # misaligned
    assert fa(ctypes.byref(sh), 4, 192, good, good, good, good, 16, None) == 3      # workspace
    assert fa(ctypes.byref(sh), -1, 192, good, good, good, good, 256, None) == 1
    assert fu(ctypes.byref(sh), 4, 200, good, good, good, good, 256, None) == 1     # v % 128
    assert fu(ctypes.byref(sh), 4, 256, good, good, None, good, 256, None) == 1
    assert fu(ctypes.byref(sh), 4, 256, good, good, good, None, 256, None) == 3
    # nothing to do: no query
    assert fa(ctypes.byref(sh), 0, 192, None, None, None, good, 256, None) == 0
    assert fu(ctypes.byref(sh), 0, 256, None, None, None, good, 256, None) == 0


def test_decode_step_host_rejects_before_enqueue(lib):
    """dsa_decode_step_host: a per-step buffer the device cannot address
    (here: any pointer, the runtime having no device to classify it against;
    on a GPU, pageable host memory) is refused before anything is enqueued,
    as are missing buffers and a short workspace; no query, nothing to do."""
    P = ctypes.c_void_p
    good = P(256)
    sh = dsa.make_shape()
    f = lib.dsa_decode_step_host
    b = _batch(max_kv=4096)
    n = _size(sh, b, dsa.OP_DECODE_STEP_HOST)[1]
    host = (ctypes.c_uint8 * 4096)()                     # pageable host memory
    hp = P(ctypes.addressof(host) + (-ctypes.addressof(host)) % 16)
    args = [hp, hp, good, hp, good, hp, None, None, None, good, n, None]
    assert f(ctypes.byref(sh), ctypes.byref(b), *args) == 1
    no_out = list(args)
    no_out[5] = None
    assert f(ctypes.byref(sh), ctypes.byref(b), *no_out) == 1
    b0 = _batch(n_q=0)
    assert f(ctypes.byref(sh), ctypes.byref(b0), None, None, None, None, None, None, None,
             None, None, good, 256 + 16 * 25604 * 4 + 16 * 256 * 8 + 4096, None) == 0
    # one more launch than the step: the input copy
    step = dsa.dsa_plan(sh, b, dsa.OP_DECODE_STEP)["kernel_launches"]
    assert dsa.dsa_plan(sh, b, dsa.OP_DECODE_STEP_HOST)["kernel_launches"] == step + 1
    with pytest.raises(ValueError):
        dsa.dsa_decode_step_host(sh, b, torch.zeros(4), None, None, None, None, None)


def test_python_binding_rejects_host_tensors(lib):
    sh = dsa.make_shape()
    with pytest.raises(ValueError):
        dsa._ptr(torch.zeros(4))
