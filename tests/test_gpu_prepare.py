"""GPU parity of the indexer query / key preparation (dsa_index_prepare: rope,
then the orthonormal Walsh-Hadamard rotation, rounded) against the host
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import deepseek_sparse_attention_gb300 as dsa
import oracle
from parity_util import host_f32

pytestmark = pytest.mark.gpu

BASE = 8e6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dsa.load()
    oracle.build()


def _check(got, ref, x, dtype):
    """float32 transform (the rope angle in double): a few units of 2^-24 of the
    vector's size; bf16 adds half an ulp of the value (2^-8 of it)."""
    scale = np.abs(x).max(axis=1, keepdims=True).astype(np.float64)
    err = np.abs(got.astype(np.float64) - ref)
    bound = 1e-5 * scale + (2.0 ** -8 * np.abs(ref) * 1.001 if dtype == "bf16" else 0.0)
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} of {bad.size} off; worst {err.max():.3e}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rope_dims", [64, 0, 128, 2])
def test_index_prepare_matches_oracle(dtype, rope_dims):
    rng = np.random.default_rng(60 + rope_dims)
    n = 1029                                           # not a multiple of the 8 rows a CTA takes
    x = (rng.standard_normal((n, 128)) * rng.uniform(0.1, 4.0, (n, 1))).astype(np.float32)
    pos = np.concatenate([[0, 1, 2, 4095, 65535, 131071, 1048575],
                          rng.integers(0, 1 << 20, n - 7)]).astype(np.int64)
    sh = dsa.make_shape(dtype=dtype)
    out = torch.empty((n, 128), dtype=torch.bfloat16 if dtype == "bf16" else torch.float32,
                      device="cuda")
    dsa.dsa_index_prepare(sh, torch.from_numpy(x).cuda(), torch.from_numpy(pos).cuda(), rope_dims,
                          BASE, out)
    torch.cuda.synchronize()
    _check(host_f32(out), oracle.index_prepare(x, pos, rope_dims, BASE), x, dtype)


def test_index_prepare_twice_without_rope_is_identity():
    """The rotation is its own inverse: preparing a prepared float32 vector with
    no rope returns it, to float32 rounding (7 butterfly stages each way: at
    most about 14 x 2^-24 x sqrt(128) of the largest component)."""
    rng = np.random.default_rng(70)
    x = torch.from_numpy(rng.standard_normal((77, 128)).astype(np.float32)).cuda()
    sh = dsa.make_shape(dtype="f32")
    y, z = torch.empty_like(x), torch.empty_like(x)
    dsa.dsa_index_prepare(sh, x, None, 0, BASE, y)
    dsa.dsa_index_prepare(sh, y, None, 0, BASE, z)
    torch.cuda.synchronize()
    assert torch.allclose(z, x, rtol=0, atol=2e-5 * float(x.abs().max()))
