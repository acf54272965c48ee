"""Pure-Python brute-force GQA attention -- TEST INFRASTRUCTURE ONLY.

An independent restatement of the oracle's definition with nested Python
lists, ``math.fsum`` and ``math.exp`` (no numpy, no C).  It is used only on
tiny shapes to pin ``oracle.c``.  Its steps follow the plain softmax
attention written on the aifullclass.xyz BERT attention article (scores =
q.k * scale, masked keys dropped, softmax over keys, weighted sum of V) with
the head-to-group map of "3个GQA核心优化技巧" (blog.gitcode.com, section
"Flash-Attention的稀疏分组优化": kv head = query head // group size).

Where the C oracle takes the maximum and normalises in two passes, this one
exponentiates every admissible score against its own maximum computed by
``max()`` over a list, then divides each weight by an ``fsum`` of them; the
output component is an ``fsum`` of products.
"""
from __future__ import annotations

import math


def attention(q, k, v, scale, causal=False, seqlens_k=None):
    """q[b][i][h][d], k[b][j][g][d], v[b][j][g][d] nested lists of floats.

    Returns (out[b][i][h][d], lse[b][h][i]) as nested lists of floats.
    """
    B = len(q)
    Sq = len(q[0])
    Hq = len(q[0][0])
    D = len(q[0][0][0])
    Sk = len(k[0])
    Hkv = len(k[0][0])
    if Hq % Hkv:
        raise ValueError("Hq must be divisible by Hkv")
    group = Hq // Hkv
    out = [[[[0.0] * D for _ in range(Hq)] for _ in range(Sq)] for _ in range(B)]
    lse = [[[0.0] * Sq for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        length = Sk if seqlens_k is None else int(seqlens_k[b])
        for i in range(Sq):
            for h in range(Hq):
                g = h // group
                keys = [j for j in range(length) if (not causal) or j <= i + Sk - Sq]
                if not keys:
                    lse[b][h][i] = -math.inf
                    continue
                scores = [scale * math.fsum(q[b][i][h][d] * k[b][j][g][d] for d in range(D))
                          for j in keys]
                top = max(scores)
                weights = [math.exp(s - top) for s in scores]
                total = math.fsum(weights)
                probs = [w / total for w in weights]
                for d in range(D):
                    out[b][i][h][d] = math.fsum(p * v[b][j][g][d] for p, j in zip(probs, keys))
                lse[b][h][i] = top + math.log(total)
    return out, lse


def attention_packed(q, k, v, cu_q, cu_k, scale, causal=False):
    """Sequences packed without padding, addressed through their row offsets.

    q[r][h][d] for packed query rows r, k[r][g][d] / v[r][g][d] for packed key
    rows; sequence b owns query rows cu_q[b] .. cu_q[b+1]-1 and key rows
    cu_k[b] .. cu_k[b+1]-1.  Query i of sequence b (packed row cu_q[b] + i)
    attends to its own sequence's keys j (packed row cu_k[b] + j) with, when
    causal, j <= i + Lk - Lq for that sequence's lengths.  Returns
    (out[r][h][d], lse[h][r]); rows of no sequence keep out = 0, lse = -inf.
    """
    total_q = len(q)
    Hq = len(q[0])
    D = len(q[0][0])
    Hkv = len(k[0])
    if Hq % Hkv:
        raise ValueError("Hq must be divisible by Hkv")
    group = Hq // Hkv
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(total_q)]
    lse = [[-math.inf] * total_q for _ in range(Hq)]
    for b in range(len(cu_q) - 1):
        q_lo, q_hi = int(cu_q[b]), int(cu_q[b + 1])
        k_lo, k_hi = int(cu_k[b]), int(cu_k[b + 1])
        n_q, n_k = q_hi - q_lo, k_hi - k_lo
        for r in range(q_lo, q_hi):
            i = r - q_lo
            for h in range(Hq):
                g = h // group
                rows = [k_lo + j for j in range(n_k) if (not causal) or j <= i + n_k - n_q]
                if not rows:
                    continue
                scores = [scale * math.fsum(q[r][h][d] * k[kr][g][d] for d in range(D)) for kr in rows]
                top = max(scores)
                weights = [math.exp(s - top) for s in scores]
                total = math.fsum(weights)
                for d in range(D):
                    out[r][h][d] = math.fsum(w / total * v[kr][g][d] for w, kr in zip(weights, rows))
                lse[h][r] = top + math.log(total)
    return out, lse


def attention_blockmask(q, k, v, scale, block_mask, block_size, causal=False, seqlens_k=None):
    """``attention`` restricted by a block mask: key j is a candidate for query
    i only when block_mask[i // block_size][j // block_size] is nonzero (in
    addition to the key length and the causal condition)."""
    B, Sq, Sk = len(q), len(q[0]), len(k[0])
    Hq, D, Hkv = len(q[0][0]), len(q[0][0][0]), len(k[0][0])
    group = Hq // Hkv
    out = [[[[0.0] * D for _ in range(Hq)] for _ in range(Sq)] for _ in range(B)]
    lse = [[[-math.inf] * Sq for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        length = Sk if seqlens_k is None else int(seqlens_k[b])
        for i in range(Sq):
            keys = [j for j in range(length) if ((not causal) or j <= i + Sk - Sq)
                    and block_mask[i // block_size][j // block_size]]
            if not keys:
                continue
            for h in range(Hq):
                g = h // group
                scores = [scale * math.fsum(q[b][i][h][d] * k[b][j][g][d] for d in range(D)) for j in keys]
                top = max(scores)
                weights = [math.exp(s - top) for s in scores]
                total = math.fsum(weights)
                for d in range(D):
                    out[b][i][h][d] = math.fsum(w / total * v[b][j][g][d] for w, j in zip(weights, keys))
                lse[b][h][i] = top + math.log(total)
    return out, lse
