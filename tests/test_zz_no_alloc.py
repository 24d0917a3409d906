"""dsa_decode_step_noalloc: the whole hot path for callers that cannot allocate
device memory (a framework capturing the stream into a CUDA graph, where
cudaMalloc is not allowed; a host engine that hands a plugin only its input and
output buffers).  It must give the results of dsa_decode_step, which uses a
caller-allocated workspace, on consecutive calls that share its fixed scratch
array.  Collected last so that a failure here stops a run only after every
other test has run."""
import numpy as np
import pytest
import torch

import deepseek_sparse_attention_gb300 as dsa
import workloads
from parity_util import gpu_batch, gpu_shape

pytestmark = pytest.mark.gpu


def _outputs(wl, dev):
    width = dsa.dsa_index_row_width(gpu_shape(wl))
    return (torch.full((wl.n_q, wl.heads, wl.kv_lora), float("nan"), device=dev),
            torch.full((wl.n_q, wl.heads), float("nan"), device=dev),
            torch.full((wl.n_q, width), -7, dtype=torch.int32, device=dev),
            torch.full((wl.n_q,), -7, dtype=torch.int32, device=dev))


@pytest.mark.parametrize("name", ["glm52_decode_128k", "tiny_fp32"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(name):
    dsa.load()
    wl = workloads.named(name)
    d = workloads.make(wl, "cuda")
    sh, b = gpu_shape(wl), gpu_batch(wl, d)
    args = (d["q_idx"], d["w"], d["k_idx"], d["q_abs"], d["cache"])

    ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP)
    ref_out, ref_lse, ref_idx, ref_n = _outputs(wl, "cuda")
    dsa.dsa_decode_step(sh, b, *args, ref_out, ref_lse, ref_idx, ref_n, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    ref = [t.cpu().numpy() for t in (ref_out, ref_lse, ref_idx, ref_n)]

    for _ in range(2):                       # the second call reuses the scratch array
        out, lse, idx, n_sel = _outputs(wl, "cuda")
        dsa.dsa_decode_step_noalloc(sh, b, *args, out, lse, idx, n_sel)
        assert dsa.dsa_check_device_error(None) == 0          # the scratch's error word
        got = [t.cpu().numpy() for t in (out, lse, idx, n_sel)]
        # the same kernels on the same inputs, deterministic: the same bits
        for x, y in zip(got, ref):
            assert np.array_equal(x, y)


def test_noalloc_reports_device_errors_through_its_scratch():
    """A batch whose offsets break its host bounds is caught on the device: the
    error word of the scratch array reports it (read with a NULL workspace),
    the read clears it, and the next call is clean and exact."""
    dsa.load()
    wl = workloads.small("noalloc_err", [9000, 4000], top_k=512)
    d = workloads.make(wl, "cuda")
    sh = gpu_shape(wl)
    args = (d["q_idx"], d["w"], d["k_idx"], d["q_abs"], d["cache"])
    good = gpu_batch(wl, d)
    # total_rows one short of the last sequence's end: the device skips it
    bad = dsa.make_batch(d["row_off"], d["key_off"], d["q_off"], wl.n_q, 1, max(wl.kv_lens),
                         sum(wl.kv_lens) - 1, sum(wl.key_counts()))
    out, lse, idx, n_sel = _outputs(wl, "cuda")
    dsa.dsa_decode_step_noalloc(sh, bad, *args, out, lse, idx, n_sel)
    assert dsa.dsa_check_device_error(None) == 2              # a batch inconsistent with its bounds
    assert dsa.dsa_check_device_error(None) == 0              # read once, cleared
    ws = dsa.alloc_workspace(sh, good, dsa.OP_DECODE_STEP)
    ref = _outputs(wl, "cuda")
    dsa.dsa_decode_step(sh, good, *args, *ref, ws)
    assert dsa.dsa_check_device_error(ws) == 0
    out, lse, idx, n_sel = _outputs(wl, "cuda")
    dsa.dsa_decode_step_noalloc(sh, good, *args, out, lse, idx, n_sel)
    assert dsa.dsa_check_device_error(None) == 0
    for x, y in zip((out, lse, idx, n_sel), ref):
        assert torch.equal(x, y)


def test_noalloc_rejects_steps_larger_than_its_scratch():
    dsa.load()
    wl = workloads.named("chunked_prefill_4096")       # 1 GiB of scores: over the limit
    dev = "cuda"
    offs = [torch.tensor([0, 65536], dtype=torch.int64, device=dev),
            torch.tensor([0, 65536], dtype=torch.int64, device=dev),
            torch.tensor([0, 4096], dtype=torch.int64, device=dev)]
    sh = gpu_shape(wl)
    b = dsa.make_batch(*offs, 4096, 4096, 65536, 65536, 65536)
    assert dsa.dsa_workspace_size(sh, b, dsa.OP_DECODE_STEP) > (8 << 20)
    t = torch.empty(16, device=dev)
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_decode_step_noalloc(sh, b, t, t, t, t, t, t)
    assert e.value.status == 2
