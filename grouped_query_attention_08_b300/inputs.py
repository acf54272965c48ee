"""Seeded synthetic workloads for grouped-query attention.

This module only draws random numbers and fixes shapes; it holds none of the
attention arithmetic.  Both the CUDA path's tests/benchmark and the oracle's
tests take their inputs from here, so the two always see the same values.

Recipe: ``torch.Generator('cpu').manual_seed(seed)``; draws in the order Q,
K, V, then key lengths; values are ``randn`` in float32, cast to bfloat16 by
round-to-nearest-even for bf16 workloads; lengths are ``randint(lo, hi+1)``.
The workloads stand in for the pages' BERT-base seq-1024 encoder, a
BERT-large long-document encoder, a Llama-style 64/8-head decode step and a
long causal prefill; no dataset is used.

Packed (variable-length) workloads draw the per-sequence lengths first
(``randint(lo, hi+1)``, queries and keys sharing a length for
self-attention), then Q [total_q,Hq,D], K and V [total_k,Hkv,D] in that
order, cast as above; sequences are packed back to back in index order.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    causal: bool
    lens: Optional[Tuple[int, int]]  # key lengths ~ U[lo, hi] per batch entry, None = full
    dtype: str                       # "bf16" or "fp32"
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    Smax: int
    lens: Tuple[int, int]            # cached lengths ~ U[lo, hi]
    dtype: str
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


@dataclasses.dataclass(frozen=True)
class VarlenWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    causal: bool
    lens: Tuple[int, int]            # sequence lengths ~ U[lo, hi] (queries = keys)
    dtype: str
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


@dataclasses.dataclass(frozen=True)
class SparseWorkload:
    name: str
    base: str                        # the dense workload whose inputs are used
    block_size: int
    pattern: str                     # "band": |qb - kb| <= window, plus key block 0
    window: int


WORKLOADS = {
    # tiny fp32 check case: B=1 Hq=4 Hkv=2 S=64 D=64, no padding
    "tiny": PrefillWorkload("tiny", 1, 4, 2, 64, 64, 64, False, None, "fp32", 0),
    # BERT-base-shaped encoder attention, key padding U[512,1024]
    "bert_base": PrefillWorkload("bert_base", 32, 12, 3, 1024, 1024, 64, False, (512, 1024),
                                 "bf16", 1),
    # BERT-large-shaped long-document encoder attention, full length
    "bert_large_long": PrefillWorkload("bert_large_long", 8, 24, 4, 4096, 4096, 64, False, None,
                                       "bf16", 2),
    # Llama-style 64/8-head decode over a cache with lengths U[1024,8192]
    "llama_decode": DecodeWorkload("llama_decode", 64, 64, 8, 128, 8192, (1024, 8192), "bf16", 3),
    # the same decode shapes with a quarter of the batch (smaller device footprint for profiling)
    "llama_decode_small": DecodeWorkload("llama_decode_small", 16, 64, 8, 128, 8192, (1024, 8192), "bf16", 3),
    # long causal prefill, D=128
    "causal_long": PrefillWorkload("causal_long", 4, 32, 8, 8192, 8192, 128, True, None, "bf16", 4),
    # llama_decode with the cache quantised to FP8 e4m3 (one scale per tensor)
    "llama_decode_fp8": DecodeWorkload("llama_decode_fp8", 64, 64, 8, 128, 8192, (1024, 8192), "fp8kv", 3),
    "llama_decode_fp8_small": DecodeWorkload("llama_decode_fp8_small", 16, 64, 8, 128, 8192, (1024, 8192),
                                             "fp8kv", 3),
    # bert_large_long under a block-sparse band: 128-token blocks, a window of
    # +-2 blocks plus the first key block (global tokens), ~18 % of the blocks
    "bert_large_long_sparse": SparseWorkload("bert_large_long_sparse", "bert_large_long", 128, "band", 2),
    # bert_base's batch packed without padding: each sequence's query and key
    # length ~ U[512,1024]
    "bert_base_varlen": VarlenWorkload("bert_base_varlen", 32, 12, 3, 64, False, (512, 1024), "bf16", 1),
}


def _cast(x: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "fp32":
        return x
    raise ValueError("dtype must be 'bf16' or 'fp32'")


def make_prefill(B, Hq, Hkv, Sq, Sk, D, *, seed=0, lens=None, dtype="bf16", q_mult=1.0):
    """Return dict(q [B,Sq,Hq,D], k, v [B,Sk,Hkv,D], seqlens_k int32 [B] or None) on the CPU.

    ``q_mult`` multiplies Q before the cast (a "peaky" variant whose softmax
    is concentrated on few keys).
    """
    g = torch.Generator("cpu").manual_seed(int(seed))
    q = torch.randn((B, Sq, Hq, D), generator=g, dtype=torch.float32)
    k = torch.randn((B, Sk, Hkv, D), generator=g, dtype=torch.float32)
    v = torch.randn((B, Sk, Hkv, D), generator=g, dtype=torch.float32)
    seqlens = None
    if lens is not None:
        lo, hi = lens
        seqlens = torch.randint(int(lo), int(hi) + 1, (B,), generator=g, dtype=torch.int64)
        seqlens = seqlens.to(torch.int32)
    if q_mult != 1.0:
        q = q * float(q_mult)
    return dict(q=_cast(q, dtype), k=_cast(k, dtype), v=_cast(v, dtype), seqlens_k=seqlens)


def make_backward(B, Hq, Hkv, Sq, Sk, D, *, seed=0, lens=None):
    """make_prefill's bf16 inputs plus an upstream gradient dout [B,Sq,Hq,D] (standard normal,
    drawn after them from the same generator)."""
    d = make_prefill(B, Hq, Hkv, Sq, Sk, D, seed=seed, lens=lens, dtype="bf16")
    g = torch.Generator("cpu").manual_seed(int(seed) + 7919)
    d["dout"] = _cast(torch.randn((B, Sq, Hq, D), generator=g, dtype=torch.float32), "bf16")
    return d


def make_decode(B, Hq, Hkv, D, Smax, *, seed=0, lens=(1, None), dtype="bf16"):
    """Return dict(q [B,Hq,D], kcache, vcache [B,Smax,Hkv,D], cache_seqlens int32 [B])."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    q = torch.randn((B, Hq, D), generator=g, dtype=torch.float32)
    kc = torch.randn((B, Smax, Hkv, D), generator=g, dtype=torch.float32)
    vc = torch.randn((B, Smax, Hkv, D), generator=g, dtype=torch.float32)
    lo, hi = lens
    hi = Smax if hi is None else hi
    seqlens = torch.randint(int(lo), int(hi) + 1, (B,), generator=g, dtype=torch.int64)
    return dict(q=_cast(q, dtype), kcache=_cast(kc, dtype), vcache=_cast(vc, dtype),
                cache_seqlens=seqlens.to(torch.int32))


def make_varlen(B, Hq, Hkv, D, *, seed=0, lens=(1, 16), lens_k=None, dtype="bf16"):
    """Packed sequences: dict(q [total_q,Hq,D], k, v [total_k,Hkv,D], cu_seqlens_q,
    cu_seqlens_k int32 [B+1], max_seqlen_q, max_seqlen_k) on the CPU.

    ``lens`` = (lo, hi) tuple draws one length per sequence, used for queries
    and keys alike; ``lens_k`` = (lo, hi) draws separate key lengths after
    them.  A list instead of a tuple gives the lengths explicitly.
    """
    g = torch.Generator("cpu").manual_seed(int(seed))

    def draw(spec):
        if isinstance(spec, list):          # explicit lengths
            if len(spec) != B:
                raise ValueError("need one length per sequence")
            return [int(x) for x in spec]
        lo, hi = spec                        # (lo, hi): drawn
        return torch.randint(int(lo), int(hi) + 1, (B,), generator=g, dtype=torch.int64).tolist()

    lq = draw(lens)
    lk = lq if lens_k is None else draw(lens_k)
    total_q, total_k = max(sum(lq), 1), max(sum(lk), 1)
    q = torch.randn((total_q, Hq, D), generator=g, dtype=torch.float32)
    k = torch.randn((total_k, Hkv, D), generator=g, dtype=torch.float32)
    v = torch.randn((total_k, Hkv, D), generator=g, dtype=torch.float32)
    cq = torch.tensor([0] + lq, dtype=torch.int64).cumsum(0).to(torch.int32)
    ck = torch.tensor([0] + lk, dtype=torch.int64).cumsum(0).to(torch.int32)
    return dict(q=_cast(q, dtype), k=_cast(k, dtype), v=_cast(v, dtype), cu_seqlens_q=cq, cu_seqlens_k=ck,
                max_seqlen_q=max(max(lq), 1), max_seqlen_k=max(max(lk), 1))


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor FP8 e4m3 quantisation as a caller would do it: scale =
    max|x| / 448 (rounded to float32), values round(x / scale) to e4m3 by
    round-to-nearest-even, clamped to the finite range.  Returns (x8, scale)."""
    amax = float(x.abs().max())
    scale = float(torch.tensor(amax / 448.0 if amax > 0 else 1.0, dtype=torch.float32))
    x8 = (x / scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return x8, scale


def make_decode_fp8(B, Hq, Hkv, D, Smax, *, seed=0, lens=(1, None), q_mult=1.0):
    """make_decode's draws with the caches quantised to e4m3: dict(q bf16 [B,Hq,D],
    kcache, vcache float8_e4m3fn [B,Smax,Hkv,D], k_scale, v_scale, cache_seqlens)."""
    d = make_decode(B, Hq, Hkv, D, Smax, seed=seed, lens=lens, dtype="fp32")
    k8, ks = quantize_e4m3(d["kcache"])
    v8, vs = quantize_e4m3(d["vcache"])
    q = d["q"] * float(q_mult) if q_mult != 1.0 else d["q"]
    return dict(q=q.to(torch.bfloat16), kcache=k8, vcache=v8, k_scale=ks, v_scale=vs,
                cache_seqlens=d["cache_seqlens"])


def make_block_mask(n_qb, n_kb, pattern="band", window=2, density=0.5, seed=0):
    """uint8 [n_qb, n_kb] block mask: "band" keeps |qb - kb| <= window (query and key
    blocks aligned at their starts) plus key block 0; "random" keeps each block with
    probability ``density``; "ones" keeps all, "zeros" none."""
    if pattern == "band":
        qb = torch.arange(n_qb)[:, None]
        kb = torch.arange(n_kb)[None, :]
        m = ((qb - kb).abs() <= window) | (kb == 0)
    elif pattern == "random":
        g = torch.Generator("cpu").manual_seed(int(seed))
        m = torch.rand((n_qb, n_kb), generator=g) < float(density)
    elif pattern == "ones":
        m = torch.ones((n_qb, n_kb), dtype=torch.bool)
    elif pattern == "zeros":
        m = torch.zeros((n_qb, n_kb), dtype=torch.bool)
    else:
        raise ValueError("unknown pattern %r" % pattern)
    return m.to(torch.uint8)


def make_sparse_workload(w):
    """Inputs of a SparseWorkload: its base workload's tensors plus block_mask."""
    base = WORKLOADS[w.base]
    d = make_prefill(base.B, base.Hq, base.Hkv, base.Sq, base.Sk, base.D, seed=base.seed, lens=base.lens,
                     dtype=base.dtype)
    bs = w.block_size
    d["block_mask"] = make_block_mask((base.Sq + bs - 1) // bs, (base.Sk + bs - 1) // bs, w.pattern, w.window)
    return d


def make_workload(w, seed=None):
    """Inputs of a named workload (a key of WORKLOADS or a workload object)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    if isinstance(w, SparseWorkload):
        return make_sparse_workload(w)
    s = w.seed if seed is None else seed
    if isinstance(w, DecodeWorkload) and w.dtype == "fp8kv":
        return make_decode_fp8(w.B, w.Hq, w.Hkv, w.D, w.Smax, seed=s, lens=w.lens)
    if isinstance(w, DecodeWorkload):
        return make_decode(w.B, w.Hq, w.Hkv, w.D, w.Smax, seed=s, lens=w.lens, dtype=w.dtype)
    if isinstance(w, VarlenWorkload):
        return make_varlen(w.B, w.Hq, w.Hkv, w.D, seed=s, lens=w.lens, dtype=w.dtype)
    return make_prefill(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, seed=s, lens=w.lens, dtype=w.dtype)


def sample_rows(n_total: int, n: int, seed: int, must=()) -> torch.Tensor:
    """Deterministic sorted sample of ``n`` distinct row ids in [0, n_total), including ``must``."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    picked = set(int(m) for m in must if 0 <= int(m) < n_total)
    if n >= n_total:
        return torch.arange(n_total, dtype=torch.int64)
    perm = torch.randperm(n_total, generator=g)[: n + len(picked)].tolist()
    for r in perm:
        if len(picked) >= n:
            break
        picked.add(int(r))
    return torch.tensor(sorted(picked), dtype=torch.int64)
