"""Algorithmic work and traffic of the attention calls (the roofline numerators).

Counts only what the method must do, never what a kernel happens to do:

* flops: 4 * D per admissible (query row, key) pair -- 2*D for the score
  q.k and 2*D for adding p * v -- summed over every (b, h, i) row.  Keys
  masked by padding or by the causal rule are not counted, nor is rounding up
  to a tile.
* bytes: every input element the result depends on read once, every output
  element written once.

KV-cache bytes follow the cache-size formula of the GQA paper summary
("GQA: Training Generalized Multi-Query Transformer Models from Multi-Head
Checkpoints", azimuth.plus/paper/gqa, the KV_cache_size equation):
2 * L * G * d_k * n elements (layers, K/V groups, head size, tokens), times
the element size in bytes.
"""
from __future__ import annotations

from typing import Optional, Sequence


def kv_cache_bytes(layers: int, groups: int, d_k: int, tokens: int, elem_bytes: int = 2) -> int:
    """Size of a K/V cache: 2 (K and V) * layers * groups * d_k * tokens * elem_bytes."""
    return 2 * layers * groups * d_k * tokens * elem_bytes


def _row_key_count(i: int, Sq: int, Sk: int, Lb: int, causal: bool) -> int:
    lim = Lb
    if causal:
        lim = min(lim, i + Sk - Sq + 1)
    return max(0, lim)


def prefill_pairs(B: int, Hq: int, Sq: int, Sk: int, causal: bool,
                  seqlens_k: Optional[Sequence[int]] = None) -> int:
    """Number of admissible (b, h, i, j) query/key pairs."""
    total = 0
    for b in range(B):
        Lb = Sk if seqlens_k is None else int(seqlens_k[b])
        if not causal:
            total += Sq * max(0, min(Lb, Sk))
            continue
        # rows i with i + Sk - Sq + 1 >= Lb see all Lb keys; the others see i + Sk - Sq + 1
        s = 0
        for i in range(Sq):
            s += _row_key_count(i, Sq, Sk, Lb, True)
        total += s
    return total * Hq


def prefill_flops(B, Hq, Sq, Sk, D, causal, seqlens_k=None) -> int:
    return 4 * D * prefill_pairs(B, Hq, Sq, Sk, causal, seqlens_k)


def backward_flops(B, Hq, Sq, Sk, D, causal, seqlens_k=None) -> int:
    """Algorithmic flops of one backward call: per admissible (query row, key)
    pair five D-long multiply-adds -- the recomputed score q.k, dP = dO.v, and
    the three gradient products P dO (dV), dS k (dQ), dS q (dK) -- i.e.
    10 * D flops, 2.5 times the forward's 4 * D."""
    return 10 * D * prefill_pairs(B, Hq, Sq, Sk, causal, seqlens_k)


def blockmask_pairs(B: int, Hq: int, Sq: int, Sk: int, causal: bool, block_mask, block_size: int,
                    seqlens_k: Optional[Sequence[int]] = None) -> int:
    """Admissible (b, h, i, j) pairs under a block mask [ceil(Sq/bs), ceil(Sk/bs)]
    (nonzero = kept), the key lengths and the causal condition."""
    bs = int(block_size)
    rows = [[int(x) != 0 for x in r] for r in (block_mask.tolist() if hasattr(block_mask, "tolist")
                                                 else block_mask)]
    total = 0
    for b in range(B):
        Lb = Sk if seqlens_k is None else int(seqlens_k[b])
        for i in range(Sq):
            lim = min(Lb, i + Sk - Sq + 1) if causal else Lb
            if lim <= 0:
                continue
            kept = rows[i // bs]
            for kb in range((lim + bs - 1) // bs):
                if kept[kb]:
                    total += min(lim, (kb + 1) * bs) - kb * bs
    return total * Hq


def varlen_pairs(Hq: int, lens_q: Sequence[int], lens_k: Sequence[int], causal: bool) -> int:
    """Admissible (sequence, h, i, j) pairs of packed sequences; causal is
    bottom-right aligned per sequence (j <= i + Lk - Lq)."""
    total = 0
    for lq, lk in zip(lens_q, lens_k):
        total += prefill_pairs(1, 1, int(lq), int(lk), causal) if lq > 0 and lk > 0 else 0
    return total * Hq


def varlen_flops(Hq, D, lens_q, lens_k, causal) -> int:
    return 4 * D * varlen_pairs(Hq, lens_q, lens_k, causal)


def varlen_bytes(Hq, Hkv, D, total_q, total_k, elem_bytes=2, with_lse=True) -> int:
    """Q, K, V and out once each (+ fp32 lse)."""
    b = elem_bytes * D * (2 * total_q * Hq + 2 * total_k * Hkv)
    return b + (4 * Hq * total_q if with_lse else 0)


def prefill_bytes(B, Hq, Hkv, Sq, Sk, D, seqlens_k=None, elem_bytes=2, with_lse=True) -> int:
    """Q read + valid K/V rows read + out written (+ fp32 lse written)."""
    valid_keys = B * Sk if seqlens_k is None else sum(int(x) for x in seqlens_k)
    q = B * Sq * Hq * D * elem_bytes
    kv = kv_cache_bytes(1, Hkv, D, valid_keys, elem_bytes)
    out = q
    lse = B * Hq * Sq * 4 if with_lse else 0
    return q + kv + out + lse


def decode_kv_bytes(Hkv: int, D: int, cache_seqlens: Sequence[int], elem_bytes: int = 2) -> int:
    """Cache bytes one decode step must read: the formula at L = 1 over all cached tokens."""
    return kv_cache_bytes(1, Hkv, D, sum(int(x) for x in cache_seqlens), elem_bytes)


def decode_bytes(B, Hq, Hkv, D, cache_seqlens, elem_bytes=2) -> int:
    """KV-cache read + q read + out written."""
    return decode_kv_bytes(Hkv, D, cache_seqlens, elem_bytes) + 2 * B * Hq * D * elem_bytes


def decode_flops(Hq, D, cache_seqlens) -> int:
    return 4 * D * Hq * sum(int(x) for x in cache_seqlens)
