"""Seeded synthetic inputs for the DSA hot path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path (through the tests and the benchmark)
and the host oracle read the tensors it makes: the oracle always receives host
copies of exactly the tensors the GPU receives.

Layout (the C-ABI layout, packed over sequences):

* ``q_idx``  [n_q, idx_heads, idx_dim]  indexer queries (dtype)
* ``w``      [n_q, idx_heads]           per-head indexer weights (float32)
* ``k_idx``  [n_keys_total, idx_dim]    indexer keys: one per token when
  ``kpool == 1``, one per complete pool of ``kpool`` tokens otherwise (dtype)
* ``q_abs``  [n_q, heads, width]        absorbed MLA queries, width =
  kv_lora + rope (dtype)
* ``cache``  [n_rows_total, width]      latent cache rows (dtype)
* ``row_off`` [n_seq+1] int64, ``key_off`` [n_seq+1] int64,
  ``q_off`` [n_seq+1] int64: prefix offsets of rows, keys and queries.

Queries of a sequence are its last ``q_len`` positions (causal, aligned to the
end of the cache): query ``i`` of a sequence with ``kv_len`` rows and ``q_len``
queries sees ``L = kv_len - q_len + 1 + i`` rows, its own row included.

Every tensor has its own stream: ``torch.Generator`` seeded from the workload
seed and a fixed per-tensor tag.  Floating values are drawn as float32 N(0,1),
scaled, then rounded to bfloat16 (round to nearest even) for bf16 workloads.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

_TAGS = {"q_idx": 1, "w": 2, "k_idx": 3, "q_abs": 4, "cache": 5, "lengths": 6, "q_full": 7,
         "w_uk": 8, "w_uv": 9, "o": 10}


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str                  # "f32" or "bf16"
    kv_lens: List[int]          # rows per sequence
    q_lens: List[int]           # queries per sequence (1 = decode)
    top_k: int = 2048
    kpool: int = 1
    idx_heads: int = 32
    idx_dim: int = 128
    heads: int = 64
    kv_lora: int = 512
    rope: int = 64
    scale: float = 1.0 / 16.0
    w_std: float = 1.0
    cache_scale: float = 1.0
    seed: int = 0
    description: str = ""

    @property
    def width(self) -> int:
        return self.kv_lora + self.rope

    @property
    def n_seq(self) -> int:
        return len(self.kv_lens)

    @property
    def n_q(self) -> int:
        return sum(self.q_lens)

    def key_counts(self) -> List[int]:
        return [L // self.kpool for L in self.kv_lens]

    def q_nvis(self) -> List[int]:
        """Visible rows L of every query, in query order."""
        out = []
        for kv, nq in zip(self.kv_lens, self.q_lens):
            out.extend(kv - nq + 1 + i for i in range(nq))
        return out

    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


def _lengths_cfg3(seed: int) -> List[int]:
    g = torch.Generator(device="cpu").manual_seed(seed * 1000 + _TAGS["lengths"])
    return torch.randint(8192, 131072 + 1, (64,), generator=g).tolist()


def named(name: str, seed: int = 0) -> Workload:
    """The five workloads of the method's benchmark suite, by name."""
    if name == "tiny_fp32":
        return Workload(name, "f32", [4096], [1], top_k=256, seed=seed,
                        description="1 query, 4096 cached tokens, top-k 256, fp32, all N(0,1)")
    if name == "glm52_decode_128k":
        return Workload(name, "bf16", [131072], [1], top_k=2048, w_std=1.0 / math.sqrt(32.0),
                        cache_scale=0.5, seed=seed,
                        description="batch 1 decode, 131072 cached tokens, top-k 2048, bf16; "
                                    "cache rows N(0,1)*0.5, w ~ N(0,1/32)")
    if name == "ragged_decode_64":
        lens = _lengths_cfg3(seed)
        return Workload(name, "bf16", lens, [1] * 64, top_k=2048, seed=seed,
                        description="64 decode sequences, lengths uniform in [8192, 131072], "
                                    "top-k 2048, bf16, N(0,1)")
    if name == "chunked_prefill_4096":
        return Workload(name, "bf16", [65536], [4096], top_k=2048, seed=seed,
                        description="4096 new queries after 61440 cached tokens (65536 rows), "
                                    "causal, top-k 2048, bf16, N(0,1)")
    if name == "chunked_prefill_1024":
        return Workload(name, "bf16", [65536], [1024], top_k=2048, seed=seed,
                        description="1024 new queries after 64512 cached tokens (65536 rows), "
                                    "causal, top-k 2048, bf16, N(0,1); the prefill chunk reduced "
                                    "for profiling captures")
    if name == "kpool_nope_1m":
        return Workload(name, "bf16", [1048576] * 4, [1] * 4, top_k=2048, kpool=4, rope=0,
                        seed=seed,
                        description="batch 4 decode, 1048576 tokens, NoPE 512-wide rows, "
                                    "one pool key per 4 tokens, top 512 pools + tail, bf16, N(0,1)")
    raise KeyError(name)


NAMES = ["tiny_fp32", "glm52_decode_128k", "ragged_decode_64", "chunked_prefill_4096",
         "kpool_nope_1m"]


def _randn(shape, tag: int, seed: int, std: float, dtype, device, chunk_rows: int = 1 << 20):
    """N(0, std^2) drawn in float32 from a per-tensor stream, rounded to dtype."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed * 1000 + tag)
    out = torch.empty(shape, dtype=dtype, device=dev)
    flat = out.view(shape[0], -1) if len(shape) > 1 else out.view(-1, 1)
    rows = flat.shape[0]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=dev, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[r0:r1].copy_(x)
    return out


def make(wl: Workload, device="cpu", copies: int = 1) -> Dict[str, object]:
    """Draw every input tensor of a workload on ``device``.

    ``copies > 1`` draws extra independent copies of the large streamed tensors
    (``k_idx`` and ``cache``) with distinct seeds, for benchmarks that rotate
    inputs so that the timed working set exceeds the L2 cache.
    """
    dt = wl.torch_dtype()
    n_q = wl.n_q
    keys_total = sum(wl.key_counts())
    rows_total = sum(wl.kv_lens)
    d: Dict[str, object] = {"workload": wl}
    d["q_idx"] = _randn((n_q, wl.idx_heads, wl.idx_dim), _TAGS["q_idx"], wl.seed, 1.0, dt, device)
    d["w"] = _randn((n_q, wl.idx_heads), _TAGS["w"], wl.seed, wl.w_std, torch.float32, device)
    d["q_abs"] = _randn((n_q, wl.heads, wl.width), _TAGS["q_abs"], wl.seed, 1.0, dt, device)
    ks, cs = [], []
    for c in range(copies):
        ks.append(_randn((keys_total, wl.idx_dim), _TAGS["k_idx"], wl.seed + 7919 * c, 1.0, dt,
                         device))
        cs.append(_randn((rows_total, wl.width), _TAGS["cache"], wl.seed + 7919 * c,
                         wl.cache_scale, dt, device))
    d["k_idx"], d["cache"] = ks[0], cs[0]
    d["k_idx_copies"], d["cache_copies"] = ks, cs

    def prefix(xs):
        out = [0]
        for x in xs:
            out.append(out[-1] + x)
        return torch.tensor(out, dtype=torch.int64, device=device)

    d["row_off"] = prefix(wl.kv_lens)
    d["key_off"] = prefix(wl.key_counts())
    d["q_off"] = prefix(wl.q_lens)
    # host-side bookkeeping (never passed to the library)
    d["q_nvis"] = torch.tensor(wl.q_nvis(), dtype=torch.int64)
    d["q_seq"] = torch.tensor([s for s, nq in enumerate(wl.q_lens) for _ in range(nq)],
                              dtype=torch.int32)
    return d


def small(name: str, kv_lens: List[int], q_lens: Optional[List[int]] = None, top_k: int = 2048,
          kpool: int = 1, rope: int = 64, dtype: str = "bf16", seed: int = 0,
          w_std: float = 1.0, cache_scale: float = 1.0) -> Workload:
    """A reduced workload with the same structure, for parity tests."""
    return Workload(name, dtype, list(kv_lens), list(q_lens or [1] * len(kv_lens)), top_k=top_k,
                    kpool=kpool, rope=rope, seed=seed, w_std=w_std, cache_scale=cache_scale,
                    description=f"reduced {name}")


def projections(wl: Workload, device="cpu", nope: int = 192, v_dim: int = 256, copies: int = 1,
                seed_offset: int = 0) -> Dict[str, object]:
    """Seeded inputs of the two projections around the attention, for the
    workload's queries and heads:

    * ``q_full`` [n_q, heads, nope + rope]  per head the no-rope query, then the
      rope part (N(0,1), dtype)
    * ``w_uk``   [heads, nope, kv_lora]     key up-projection, N(0, 1/nope) (dtype)
    * ``w_uv``   [heads, v_dim, kv_lora]    value up-projection, N(0, 1/kv_lora)
      (dtype)
    * ``o``      [n_q, heads, kv_lora]      an attention output, N(0, 1/16) float32

    ``copies > 1`` draws further independent weight sets (``w_uk_copies``,
    ``w_uv_copies``) for timing loops that must not find the weights in L2.
    """
    dt = wl.torch_dtype()
    seed = wl.seed + seed_offset
    d: Dict[str, object] = {}
    d["q_full"] = _randn((wl.n_q, wl.heads, nope + wl.rope), _TAGS["q_full"], seed, 1.0, dt, device)
    d["o"] = _randn((wl.n_q, wl.heads, wl.kv_lora), _TAGS["o"], seed, 0.25, torch.float32, device)
    d["w_uk_copies"] = [_randn((wl.heads, nope, wl.kv_lora), _TAGS["w_uk"], seed + 7919 * c,
                               1.0 / math.sqrt(nope), dt, device) for c in range(copies)]
    d["w_uv_copies"] = [_randn((wl.heads, v_dim, wl.kv_lora), _TAGS["w_uv"], seed + 7919 * c,
                               1.0 / math.sqrt(wl.kv_lora), dt, device) for c in range(copies)]
    d["w_uk"], d["w_uv"] = d["w_uk_copies"][0], d["w_uv_copies"][0]
    return d
