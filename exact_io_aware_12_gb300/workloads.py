"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and arranges them; it holds none of the
attention arithmetic.  The CUDA path's tests, the benchmark and the oracle
checks all take their inputs from here, so both sides see the same bf16 values.

The five named workloads follow the shapes the pages discuss: a GPT-2-style
N=1024, d=64 self-attention ("o problema" section of the tonho.wtf
"flash attention" entry quotes GPT-2 medium at sequence 1024) and the long
contexts of the QK^T size table in "Atencao eficiente - FlashAttention, sparse
e hibrida" (16k and 128k tokens).

Recipe (one CPU ``torch.Generator`` per workload, seeded with its index):
  draw Q, K, V, dO in that order as float32 N(0, 1) of shape [B, H, N, d];
  scale Q and K by ``qk_scale`` (peaky rows); for the sink workload set key
  row 0 of every head to 4 x the mean of that head's query rows; round to
  bf16 (round to nearest even).  Sampled query rows for the oracle come from a
  second generator seeded with 1000 + index and always include rows 0, 127,
  128, N-1 and, for the 128k workload, every 8192-row boundary and the row
  before it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    qk_scale: float = 1.0
    sink: bool = False
    backward: bool = True
    fwd_rows_per_head: Optional[int] = None   # None: the oracle checks every row
    bwd_slice: Optional[int] = None           # prefix length for the full-tensor bwd check

    @property
    def tau(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def shape(self):
        return (self.B, self.H, self.N, self.d)


WORKLOADS: List[Workload] = [
    Workload("tiny_b1h2_n128_d64_full", 1, 2, 128, 64, False, 0),
    Workload("gpt2s_b8h12_n1024_d64_causal", 8, 12, 1024, 64, True, 1),
    Workload("gpt2m_peaky_b16h16_n1024_d64_causal", 16, 16, 1024, 64, True, 2, qk_scale=3.0),
    Workload("long_sink_b1h16_n16384_d128_causal", 1, 16, 16384, 128, True, 3, sink=True,
             fwd_rows_per_head=512, bwd_slice=2048),
    Workload("long_b1h8_n131072_d128_causal_fwd", 1, 8, 131072, 128, True, 4,
             backward=False, fwd_rows_per_head=256),
]
BY_NAME: Dict[str, Workload] = {w.name: w for w in WORKLOADS}


def flops_fwd(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """Counted forward FLOPs: 4*B*H*N^2*d, halved for a causal mask."""
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def flops_bwd(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """Counted backward FLOPs: 2.5 x the forward count."""
    return 2.5 * flops_fwd(B, H, N, d, causal)


def draw(B: int, H: int, N: int, d: int, seed: int, qk_scale: float = 1.0,
         sink: bool = False, with_do: bool = True) -> Dict[str, torch.Tensor]:
    """Seeded bf16 CPU tensors q, k, v (and do), each [B, H, N, d]."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32) if with_do else None
    if qk_scale != 1.0:
        q.mul_(qk_scale)
        k.mul_(qk_scale)
    if sink and N > 0:
        k[:, :, 0, :] = 4.0 * q.mean(dim=2)
    out = {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}
    if do is not None:
        out["do"] = do.to(torch.bfloat16)
    return out


def make_inputs(w: Workload) -> Dict[str, torch.Tensor]:
    return draw(w.B, w.H, w.N, w.d, w.seed, w.qk_scale, w.sink, with_do=w.backward)


def sample_rows(w: Workload, per_head: Optional[int] = None) -> np.ndarray:
    """Sorted flat row ids (bh * N + i) for an oracle row check."""
    per_head = per_head or w.fwd_rows_per_head or w.N
    N = w.N
    fixed = {0, N - 1, min(127, N - 1), min(128, N - 1)}
    if N >= 131072:
        for b in range(8192, N, 8192):
            fixed.update((b - 1, b))
    g = np.random.default_rng(1000 + w.seed)
    fixed_arr = np.asarray(sorted(fixed), dtype=np.int64)
    pool = np.setdiff1d(np.arange(N, dtype=np.int64), fixed_arr)
    need = max(0, min(per_head, N) - fixed_arr.size)
    rows = []
    for bh in range(w.B * w.H):
        extra = g.choice(pool, size=need, replace=False) if need else pool[:0]
        head = np.union1d(fixed_arr, extra)
        rows.append(bh * N + head)
    return np.concatenate(rows).astype(np.int64)


def local_global_block_mask(n_blocks: int, local: int, anchors: int, heads: int = 1,
                            extra: float = 0.0, seed: int = 0) -> np.ndarray:
    """Seeded block mask, uint8 [heads, n_blocks, n_blocks], of the sparse
    pattern sketched in "Atencao eficiente - FlashAttention, sparse e hibrida",
    section "Sparse e hibrida" (a local window plus global anchor tokens): row
    block i sees key blocks [i - local + 1, i] and the first ``anchors`` key
    blocks; ``extra`` sets that fraction of the remaining blocks at random,
    drawn per head from ``numpy.random.default_rng(seed)``."""
    m = np.zeros((heads, n_blocks, n_blocks), dtype=np.uint8)
    i = np.arange(n_blocks)[:, None]
    j = np.arange(n_blocks)[None, :]
    m[:] = ((j <= i) & (j > i - local)) | (j < anchors)
    if extra > 0:
        g = np.random.default_rng(seed)
        m |= (g.random(m.shape) < extra).astype(np.uint8)
    return m


def random_block_mask(n_blocks: int, heads: int, density: float, seed: int,
                      empty_rows: int = 0) -> np.ndarray:
    """Seeded random block mask, uint8 [heads, n_blocks, n_blocks]: each entry
    set with probability ``density``; then ``empty_rows`` row blocks per head
    (chosen from the same generator) are cleared entirely."""
    g = np.random.default_rng(seed)
    m = (g.random((heads, n_blocks, n_blocks)) < density).astype(np.uint8)
    for h in range(heads):
        for r in g.choice(n_blocks, size=min(empty_rows, n_blocks), replace=False):
            m[h, r] = 0
    return m


@dataclass(frozen=True)
class DecodeWorkload:
    """A decode step: Nq new query rows per (batch, head) against an Nk-key KV
    cache.  Inputs: one CPU generator seeded with ``seed``, Q then K then V as
    float32 N(0, 1), rounded to bf16."""
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    seed: int

    @property
    def tau(self) -> float:
        return 1.0 / math.sqrt(self.d)


DECODE_WORKLOADS: List[DecodeWorkload] = [
    # one new token per sequence, 8 sequences x 16 heads reading a 32k-token cache (2.1 GB of K, V)
    DecodeWorkload("decode_b8h16_nq1_nk32768_d128", 8, 16, 1, 32768, 128, True, 10),
    # 4 tokens per step (draft tokens checked together) against a 128k-token cache
    DecodeWorkload("decode_b1h8_nq4_nk131072_d128_causal", 1, 8, 4, 131072, 128, True, 11),
]
DECODE_BY_NAME: Dict[str, DecodeWorkload] = {w.name: w for w in DECODE_WORKLOADS}


def draw_decode(B: int, H: int, Nq: int, Nk: int, d: int, seed: int) -> Dict[str, torch.Tensor]:
    """Seeded bf16 CPU tensors q [B, H, Nq, d], k and v [B, H, Nk, d]."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32)
    return {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}


def draw_fp8(B: int, H: int, N: int, d: int, seed: int) -> Dict[str, object]:
    """Seeded FP8 inputs: Q, K, V drawn as float32 N(0, 1) (one CPU generator,
    in that order), each given the per-tensor scale amax / 448 and rounded to
    e4m3 (torch float8_e4m3fn, round to nearest even).  Returns the e4m3 bytes
    (uint8 [B, H, N, d]) as q8, k8, v8 and the scales q_scale, k_scale, v_scale."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    out: Dict[str, object] = {}
    for name in ("q", "k", "v"):
        x = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
        scale = float(x.abs().max()) / 448.0
        out[name + "8"] = (x / scale).to(torch.float8_e4m3fn).view(torch.uint8)
        out[name + "_scale"] = scale
    return out
