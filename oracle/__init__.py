"""fp64 CPU oracle for grouped-query attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``grouped_query_attention_08_b300``) never imports it and shares no code
with it; both sides only share the seeded input generators.

``oracle.c`` holds the definition (plain two-pass softmax in fp64, one row at
a time); this module compiles it with gcc on first use and wraps it with
ctypes.  ``brute.py`` is an independent pure-Python restatement used to pin
the C code on tiny inputs.

Sources: see the header of ``oracle.c`` (pages "3个GQA核心优化技巧" on
blog.gitcode.com, the GQA paper summary on azimuth.plus, the aifullclass.xyz
BERT attention article, and "FlashAttention Serisi" on webturing.pages.dev).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.oracle_gqa_attention.restype = i32
            lib.oracle_gqa_attention.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                 i32, i32, dbl, i32, vp, vp, i64]
            _lib = lib
    return _lib


def _f32(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor: widen exactly to float32 on the CPU
        a = a.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def attention(q, k, v, *, scale=None, causal=False, seqlens_k=None, rows=None, sk=None):
    """Oracle GQA attention.

    q [B,Sq,Hq,D]; k,v [B,Skcap,Hkv,D] (float arrays or CPU tensors holding the
    exact input values); ``sk`` = logical key count (default Skcap);
    ``seqlens_k`` int [B] or None; ``rows`` optional int64 array of
    (b*Hq+h)*Sq+i row ids.  Returns (out, lse) in float64: out [B,Sq,Hq,D] and
    lse [B,Hq,Sq], or out [nrows,D] and lse [nrows] when ``rows`` is given.
    ``scale`` defaults to 1/sqrt(D) ([GQA-BERT] "阶段二").
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Sq, Hq, D = q.shape
    Bk, Skcap, Hkv, Dk = k.shape
    if Bk != B or Dk != D or v.shape != k.shape:
        raise ValueError("shape mismatch")
    Sk = Skcap if sk is None else int(sk)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lens = None
    if seqlens_k is not None:
        if hasattr(seqlens_k, "detach"):
            seqlens_k = seqlens_k.detach().cpu().numpy()
        lens = np.ascontiguousarray(seqlens_k, dtype=np.int32)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.zeros((rows.shape[0], D), np.float64)
        lse = np.zeros((rows.shape[0],), np.float64)
    else:
        out = np.zeros((B, Sq, Hq, D), np.float64)
        lse = np.zeros((B, Hq, Sq), np.float64)
    lib = _load()
    rc = lib.oracle_gqa_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                  B, Hq, Hkv, Sq, Sk, Skcap, D, float(scale), int(bool(causal)),
                                  _ptr(lens) if lens is not None else None,
                                  _ptr(rows) if rows is not None else None,
                                  0 if rows is None else rows.shape[0])
    if rc != 0:
        raise ValueError("oracle rejected the arguments (code %d)" % rc)
    return out, lse


def decode(q, kcache, vcache, cache_seqlens, *, scale=None, rows=None):
    """Oracle single-token decode: q [B,Hq,D]; caches [B,Smax,Hkv,D].

    The new token attends to cache rows [0, cache_seqlens[b]) with no causal
    term.  Returns (out [B,Hq,D], lse [B,Hq]) in float64.
    """
    q = _f32(q)
    B, Hq, D = q.shape
    out, lse = attention(q.reshape(B, 1, Hq, D), kcache, vcache, scale=scale, causal=False,
                         seqlens_k=cache_seqlens, rows=rows)
    if rows is not None:
        return out, lse
    return out.reshape(B, Hq, D), lse.reshape(B, Hq)


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, *, scale=None, causal=False):
    """Oracle GQA attention over sequences packed without padding.

    q [total_q,Hq,D], k/v [total_k,Hkv,D]; cu_seqlens_q/k int [B+1] row offsets.
    Sequence b is the plain definition of ``attention`` with B = 1, Sq = its
    query count, Sk = its key count (so causal is bottom-right aligned per
    sequence), applied to its own rows.  Returns out [total_q,Hq,D] and lse
    [Hq,total_q] in float64; rows that belong to no sequence stay out = 0,
    lse = -inf.
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    total_q, Hq, D = q.shape
    total_k, Hkv, Dk = k.shape
    if Dk != D or v.shape != k.shape:
        raise ValueError("shape mismatch")
    cq = [int(x) for x in (cu_seqlens_q.tolist() if hasattr(cu_seqlens_q, "tolist") else cu_seqlens_q)]
    ck = [int(x) for x in (cu_seqlens_k.tolist() if hasattr(cu_seqlens_k, "tolist") else cu_seqlens_k)]
    if len(cq) != len(ck) or len(cq) < 2:
        raise ValueError("cu_seqlens must both be [B+1]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.zeros((total_q, Hq, D), np.float64)
    lse = np.full((Hq, total_q), -np.inf, np.float64)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if not (0 <= q0 <= q1 <= total_q and 0 <= k0 <= k1 <= total_k):
            raise ValueError("cu_seqlens out of range at sequence %d" % b)
        if q1 == q0 or k1 == k0:
            continue   # no query rows, or no keys: out = 0, lse = -inf
        o_b, l_b = attention(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], scale=scale, causal=causal)
        out[q0:q1] = o_b[0]
        lse[:, q0:q1] = l_b[0]
    return out, lse


def decode_fp8(q, kcache8, vcache8, k_scale, v_scale, cache_seqlens, *, scale=None, rows=None):
    """Oracle decode over an e4m3 cache with one scale per tensor: the attended
    key is k_scale * k8 and the value v_scale * v8.

    Since scale * q.(k_scale k8) = (scale * k_scale) * q.k8 and the output is
    linear in V, this is ``decode`` on the e4m3 values themselves (exact in
    float32) with the softmax scale scale * k_scale (in fp64), its output
    multiplied by v_scale (in fp64); lse is unchanged.
    """
    def f8(a):
        if hasattr(a, "detach"):
            return a.detach().cpu().float().numpy()
        return np.asarray(a, dtype=np.float32)
    q = _f32(q)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    out, lse = decode(q, f8(kcache8), f8(vcache8), cache_seqlens, scale=float(scale) * float(k_scale), rows=rows)
    return out * float(v_scale), lse


def attention_blockmask(q, k, v, block_mask, block_size, *, scale=None, causal=False, seqlens_k=None):
    """Oracle GQA attention with a block-sparsity mask ([GQA-BERT] "阶段二":
    block_size, sparse=True; the pattern is the caller's).

    q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D]; block_mask [ceil(Sq/bs), ceil(Sk/bs)] (nonzero =
    attend), shared by every batch entry and head.  Key j is admissible for query i
    when j < L_b, (not causal or j <= i + Sk - Sq) and block_mask[i//bs][j//bs] != 0.
    Plain definition per (b, h) in fp64: scores by one matrix product, excluded keys
    dropped, softmax against the row maximum.  Returns out [B,Sq,Hq,D], lse [B,Hq,Sq].
    """
    q, k, v = _f32(q).astype(np.float64), _f32(k).astype(np.float64), _f32(v).astype(np.float64)
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    bm = np.asarray(block_mask.cpu().numpy() if hasattr(block_mask, "cpu") else block_mask) != 0
    bs = int(block_size)
    if bm.shape != ((Sq + bs - 1) // bs, (Sk + bs - 1) // bs):
        raise ValueError("block_mask must be [ceil(Sq/bs), ceil(Sk/bs)]")
    lens = None if seqlens_k is None else np.asarray(
        seqlens_k.cpu().numpy() if hasattr(seqlens_k, "cpu") else seqlens_k).astype(np.int64)
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    base = bm[i // bs, j // bs]
    if causal:
        base = base & (j <= i + Sk - Sq)
    out = np.zeros((B, Sq, Hq, D), np.float64)
    lse = np.full((B, Hq, Sq), -np.inf, np.float64)
    for b in range(B):
        allowed = base & (j < (Sk if lens is None else lens[b]))
        any_key = allowed.any(axis=1)
        for h in range(Hq):
            s = scale * (q[b, :, h, :] @ k[b, :, h // G, :].T)
            s = np.where(allowed, s, -np.inf)
            m = np.where(any_key, s.max(axis=1), 0.0)
            w = np.where(allowed, np.exp(s - m[:, None]), 0.0)
            l = w.sum(axis=1)
            ok = l > 0
            out[b, ok, h, :] = (w[ok] / l[ok, None]) @ v[b, :, h // G, :]
            lse[b, h, ok] = m[ok] + np.log(l[ok])
    return out, lse


def attention_backward(q, k, v, dout, *, scale=None, causal=False, seqlens_k=None):
    """Oracle gradients of GQA attention (the forward's definition above) for an
    upstream gradient dout [B,Sq,Hq,D].  Plain fp64 per (b, h) with P the exact
    softmax over the admissible keys:
        dV_j  += sum_i P_ij dO_i                 (summed over the G heads of the group)
        dP_ij  = dO_i . v_j,   Dsum_i = sum_j P_ij dP_ij   (= dO_i . O_i)
        dS_ij  = P_ij (dP_ij - Dsum_i)
        dQ_i   = scale sum_j dS_ij k_j,   dK_j += scale sum_i dS_ij q_i
    Returns dq [B,Sq,Hq,D], dk [B,Sk,Hkv,D], dv [B,Sk,Hkv,D] in float64.
    """
    q, k, v = (_f32(x).astype(np.float64) for x in (q, k, v))
    do = _f32(dout).astype(np.float64)
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lens = None if seqlens_k is None else np.asarray(
        seqlens_k.cpu().numpy() if hasattr(seqlens_k, "cpu") else seqlens_k).astype(np.int64)
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    dq = np.zeros_like(q)
    dk = np.zeros((B, Sk, Hkv, D), np.float64)
    dv = np.zeros((B, Sk, Hkv, D), np.float64)
    for b in range(B):
        allowed = j < (Sk if lens is None else lens[b])
        if causal:
            allowed = allowed & (j <= i + Sk - Sq)
        any_key = allowed.any(axis=1)
        for h in range(Hq):
            g = h // G
            s = scale * (q[b, :, h, :] @ k[b, :, g, :].T)
            s = np.where(allowed, s, -np.inf)
            m = np.where(any_key, s.max(axis=1), 0.0)
            w = np.where(allowed, np.exp(s - m[:, None]), 0.0)
            l = w.sum(axis=1)
            p = np.where(any_key[:, None], w / np.where(l > 0, l, 1.0)[:, None], 0.0)
            dp = do[b, :, h, :] @ v[b, :, g, :].T
            dsum = (p * dp).sum(axis=1)
            ds = p * (dp - dsum[:, None])
            dq[b, :, h, :] = scale * (ds @ k[b, :, g, :])
            dk[b, :, g, :] += scale * (ds.T @ q[b, :, h, :])
            dv[b, :, g, :] += p.T @ do[b, :, h, :]
    return dq, dk, dv


def attention_backward_dq_rows(q, k, v, dout, rows, *, scale=None, causal=False, seqlens_k=None):
    """dQ of `attention_backward` for selected query rows only, each computed on
    its own from the definition (the row's exact softmax P_i over its
    admissible keys, dP_i = dO_i V^T, Dsum_i = P_i . dP_i, dQ_i = scale
    (P_i * (dP_i - Dsum_i)) K): for checks at sizes where the full gradient is
    too large for the CPU.  rows: (b, h, i) triples.  Returns [len(rows), D]
    float64.
    """
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lens = None if seqlens_k is None else np.asarray(
        seqlens_k.cpu().numpy() if hasattr(seqlens_k, "cpu") else seqlens_k).astype(np.int64)
    out = np.zeros((len(rows), D), np.float64)
    for n, (b, h, i) in enumerate(rows):
        g = h // G
        kb = _f32(k[b, :, g, :]).astype(np.float64)
        vb = _f32(v[b, :, g, :]).astype(np.float64)
        qi = _f32(q[b, i, h, :]).astype(np.float64)
        doi = _f32(dout[b, i, h, :]).astype(np.float64)
        j = np.arange(Sk)
        allowed = j < (Sk if lens is None else lens[b])
        if causal:
            allowed &= j <= i + Sk - Sq
        if not allowed.any():
            continue
        s = scale * (kb @ qi)
        m = s[allowed].max()
        w = np.where(allowed, np.exp(np.where(allowed, s, m) - m), 0.0)
        p = w / w.sum()
        dp = vb @ doi
        dsum = float((p * dp).sum())
        out[n] = scale * ((p * (dp - dsum)) @ kb)
    return out
