"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every test here checks the oracle against something other than itself:
brute force on tiny inputs, a library routine (torch's CPU scaled
dot-product attention in fp64), a closed form, a hand-worked example or an
invariant.  Plausible mistakes -- a dropped scale, a wrong sign, a transposed
operand, an interleaved instead of contiguous head map, an off-by-one in the
padding or causal mask, a missing normalisation -- each fail at least one.
"""
import math
import os
import random

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import brute
from grouped_query_attention_08_b300 import inputs, roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, rng, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float32)


def _tolist(a):
    return a.astype(np.float64).tolist()


# ---------------------------------------------------------------- brute force

def _brute_cases(n, seed):
    rng = random.Random(seed)
    cases = []
    for _ in range(n):
        G = rng.choice([1, 2, 3, 4, 8])
        Hkv = rng.choice([1, 1, 2]) if G >= 4 else rng.choice([1, 2, 3])
        Hq = G * Hkv
        if Hq > 8:
            Hkv, Hq = 1, G
        B = rng.choice([1, 2])
        Sk = rng.randint(1, 20 if rng.random() < 0.9 else 37)
        Sq = rng.randint(1, 20 if rng.random() < 0.9 else 37)
        D = rng.choice([1, 3, 8, 16])
        causal = rng.random() < 0.5
        lens = None
        if rng.random() < 0.6:
            lens = [rng.randint(0, Sk) for _ in range(B)]
        scale = rng.choice([1.0 / math.sqrt(D), 0.3, -0.7, 0.0, 1.9])
        cases.append((B, Hq, Hkv, Sq, Sk, D, causal, lens, scale, rng.randint(0, 1 << 30)))
    return cases


@pytest.mark.parametrize("case", _brute_cases(200, 1234))
def test_oracle_matches_pure_python_brute_force(case):
    B, Hq, Hkv, Sq, Sk, D, causal, lens, scale, seed = case
    rng = np.random.default_rng(seed)
    q, k, v = _rand((B, Sq, Hq, D), rng), _rand((B, Sk, Hkv, D), rng), _rand((B, Sk, Hkv, D), rng)
    out, lse = oracle.attention(q, k, v, scale=scale, causal=causal, seqlens_k=lens)
    bout, blse = brute.attention(_tolist(q), _tolist(k), _tolist(v), scale, causal, lens)
    np.testing.assert_allclose(out, np.array(bout), rtol=0, atol=1e-12)
    blse = np.array(blse)
    assert np.array_equal(np.isneginf(lse), np.isneginf(blse))
    fin = np.isfinite(blse)
    np.testing.assert_allclose(lse[fin], blse[fin], rtol=0, atol=1e-12)


# ------------------------------------------------------------ library routine

def _sdpa(q, k, v, scale, mask=None, enable_gqa=False):
    # torch layout [B, H, S, D]
    tq = torch.from_numpy(q.astype(np.float64)).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k.astype(np.float64)).permute(0, 2, 1, 3)
    tv = torch.from_numpy(v.astype(np.float64)).permute(0, 2, 1, 3)
    o = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale,
                                       enable_gqa=enable_gqa)
    return o.permute(0, 2, 1, 3).numpy()


def _bool_mask(B, Sq, Sk, lens, causal):
    m = torch.ones(B, 1, Sq, Sk, dtype=torch.bool)
    for b in range(B):
        Lb = Sk if lens is None else lens[b]
        m[b, :, :, Lb:] = False
        if causal:
            i = torch.arange(Sq).view(Sq, 1)
            j = torch.arange(Sk).view(1, Sk)
            m[b, 0] &= j <= i + Sk - Sq
    return m


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (6, 6)])
def test_mha_special_case_matches_library_sdpa(Hq, Hkv):
    """GQA-H is MHA (GQA paper summary, Idea 2): no grouping at all."""
    rng = np.random.default_rng(7)
    B, S, D = 2, 33, 16
    q, k, v = _rand((B, S, Hq, D), rng), _rand((B, S, Hkv, D), rng), _rand((B, S, Hkv, D), rng)
    lens = [33, 17]
    out, _ = oracle.attention(q, k, v, scale=0.25, seqlens_k=lens)
    ref = _sdpa(q, k, v, 0.25, mask=_bool_mask(B, S, S, lens, False))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-10)


def test_mqa_special_case_matches_library_sdpa():
    """GQA-1 is MQA: every query head uses the single K/V head."""
    rng = np.random.default_rng(8)
    B, S, Hq, D = 2, 29, 5, 8
    q, k, v = _rand((B, S, Hq, D), rng), _rand((B, S, 1, D), rng), _rand((B, S, 1, D), rng)
    out, _ = oracle.attention(q, k, v, scale=0.4, causal=True)
    kb = np.repeat(k, Hq, axis=2)
    vb = np.repeat(v, Hq, axis=2)
    ref = _sdpa(q, kb, vb, 0.4, mask=_bool_mask(B, S, S, None, True))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-10)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (12, 3), (6, 2), (8, 1)])
def test_gqa_matches_library_sdpa_with_grouping(Hq, Hkv, causal):
    """torch's own GQA mode maps query head h to K/V head h // (Hq/Hkv)."""
    rng = np.random.default_rng(Hq * 10 + Hkv + causal)
    B, Sq, Sk, D = 2, 21, 30, 16
    q, k, v = _rand((B, Sq, Hq, D), rng), _rand((B, Sk, Hkv, D), rng), _rand((B, Sk, Hkv, D), rng)
    lens = None if causal else [30, 11]
    out, _ = oracle.attention(q, k, v, scale=0.3, causal=causal, seqlens_k=lens)
    ref = _sdpa(q, k, v, 0.3, mask=_bool_mask(B, Sq, Sk, lens, causal), enable_gqa=True)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-10)


# ------------------------------------------------------------------ invariants

def test_gqa_equals_mha_with_repeated_kv_heads_exactly():
    """GQA(Q,K,V) = MHA(Q, K and V with each head repeated Hq/Hkv times, contiguously)."""
    rng = np.random.default_rng(3)
    B, S, Hq, Hkv, D = 2, 40, 12, 3, 16
    q, k, v = _rand((B, S, Hq, D), rng), _rand((B, S, Hkv, D), rng), _rand((B, S, Hkv, D), rng)
    lens = [40, 23]
    a, la = oracle.attention(q, k, v, scale=0.2, seqlens_k=lens)
    kr, vr = np.repeat(k, Hq // Hkv, axis=2), np.repeat(v, Hq // Hkv, axis=2)
    b_, lb = oracle.attention(q, kr, vr, scale=0.2, seqlens_k=lens)
    assert np.array_equal(a, b_) and np.array_equal(la, lb)
    # an interleaved map (h % Hkv) gives a different answer
    ki, vi = np.tile(k, (1, 1, Hq // Hkv, 1)), np.tile(v, (1, 1, Hq // Hkv, 1))
    c, _ = oracle.attention(q, ki, vi, scale=0.2, seqlens_k=lens)
    assert np.abs(a - c).max() > 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one(causal):
    rng = np.random.default_rng(4)
    B, S, Hq, Hkv, D = 2, 37, 6, 2, 8
    q, k = _rand((B, S, Hq, D), rng, 3.0), _rand((B, S, Hkv, D), rng)
    v = np.ones((B, S, Hkv, D), np.float32)
    out, _ = oracle.attention(q, k, v, scale=0.5, causal=causal, seqlens_k=[37, 5])
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-13)


def test_one_hot_values_give_probability_rows():
    rng = np.random.default_rng(5)
    B, S, Hq, Hkv, D = 1, 16, 4, 2, 16
    q, k = _rand((B, S, Hq, D), rng, 2.0), _rand((B, S, Hkv, D), rng)
    v = np.zeros((B, S, Hkv, D), np.float32)
    for j in range(S):
        v[:, j, :, j] = 1.0
    out, _ = oracle.attention(q, k, v, scale=0.7, seqlens_k=[11])
    assert (out >= 0).all()
    np.testing.assert_allclose(out.sum(-1), 1.0, rtol=0, atol=1e-13)
    assert np.all(out[..., 11:] == 0.0)        # padded keys carry exactly zero weight


def test_identical_keys_give_mean_of_valid_values_and_closed_form_lse():
    rng = np.random.default_rng(6)
    B, S, Hq, Hkv, D = 3, 24, 8, 2, 8
    q = _rand((B, S, Hq, D), rng)
    k = np.broadcast_to(_rand((B, 1, Hkv, D), rng), (B, S, Hkv, D)).copy()
    v = _rand((B, S, Hkv, D), rng)
    lens = [24, 9, 1]
    out, lse = oracle.attention(q, k, v, scale=0.35, seqlens_k=lens)
    G = Hq // Hkv
    for b in range(B):
        L = lens[b]
        for h in range(Hq):
            mean = v[b, :L, h // G, :].astype(np.float64).mean(0)
            np.testing.assert_allclose(out[b, :, h, :], np.broadcast_to(mean, (S, D)), atol=1e-12)
            s = 0.35 * (q[b, :, h, :].astype(np.float64) @ k[b, 0, h // G, :].astype(np.float64))
            np.testing.assert_allclose(lse[b, h, :], s + math.log(L), atol=1e-12)


def test_zero_scale_gives_mean_of_valid_values():
    rng = np.random.default_rng(9)
    B, S, Hq, Hkv, D = 2, 19, 4, 1, 4
    q, k, v = _rand((B, S, Hq, D), rng), _rand((B, S, Hkv, D), rng), _rand((B, S, Hkv, D), rng)
    out, lse = oracle.attention(q, k, v, scale=0.0, seqlens_k=[19, 7])
    for b, L in enumerate([19, 7]):
        np.testing.assert_allclose(out[b], np.broadcast_to(v[b, :L, 0].astype(np.float64).mean(0),
                                                           (S, Hq, D)), atol=1e-13)
        np.testing.assert_allclose(lse[b], math.log(L), atol=1e-13)


def test_padded_keys_do_not_change_a_single_bit():
    rng = np.random.default_rng(10)
    B, S, Hq, Hkv, D = 2, 30, 4, 2, 8
    q, k, v = _rand((B, S, Hq, D), rng), _rand((B, S, Hkv, D), rng), _rand((B, S, Hkv, D), rng)
    lens = [12, 29]
    a, la = oracle.attention(q, k, v, scale=0.3, seqlens_k=lens)
    k2, v2 = k.copy(), v.copy()
    for b, L in enumerate(lens):
        k2[b, L:] = 1e4
        v2[b, L:] = -1e4
    b_, lb = oracle.attention(q, k2, v2, scale=0.3, seqlens_k=lens)
    assert np.array_equal(a, b_) and np.array_equal(la, lb)


def test_causal_first_row_and_single_key():
    rng = np.random.default_rng(11)
    B, S, Hq, Hkv, D = 2, 9, 4, 2, 8
    q, k, v = _rand((B, S, Hq, D), rng), _rand((B, S, Hkv, D), rng), _rand((B, S, Hkv, D), rng)
    out, lse = oracle.attention(q, k, v, scale=0.5, causal=True)
    G = Hq // Hkv
    for h in range(Hq):
        np.testing.assert_array_equal(out[:, 0, h, :], v[:, 0, h // G, :].astype(np.float64))
        s0 = 0.5 * np.einsum("bd,bd->b", q[:, 0, h].astype(np.float64), k[:, 0, h // G].astype(np.float64))
        np.testing.assert_allclose(lse[:, h, 0], s0, atol=1e-13)
    # Sk = 1: every row sees exactly key 0
    out1, lse1 = oracle.attention(q, k[:, :1], v[:, :1], scale=0.5)
    for h in range(Hq):
        np.testing.assert_array_equal(out1[:, :, h, :],
                                      np.broadcast_to(v[:, :1, h // G, :].astype(np.float64), (B, S, D)))


def test_causal_bottom_right_alignment_when_sq_less_than_sk():
    """The last query row of a causal call sees every key; row i sees keys j <= i + Sk - Sq."""
    rng = np.random.default_rng(12)
    B, Sq, Sk, Hq, Hkv, D = 1, 5, 13, 2, 1, 8
    q, k, v = _rand((B, Sq, Hq, D), rng), _rand((B, Sk, Hkv, D), rng), _rand((B, Sk, Hkv, D), rng)
    c, _ = oracle.attention(q, k, v, scale=0.4, causal=True)
    n, _ = oracle.attention(q, k, v, scale=0.4, causal=False)
    np.testing.assert_array_equal(c[:, -1], n[:, -1])
    # row 0 equals a non-causal call restricted to the first Sk - Sq + 1 keys
    r, _ = oracle.attention(q[:, :1], k[:, : Sk - Sq + 1], v[:, : Sk - Sq + 1], scale=0.4)
    np.testing.assert_allclose(c[:, :1], r, atol=1e-15)


def test_key_permutation_invariance():
    rng = np.random.default_rng(13)
    B, S, Hq, Hkv, D = 2, 31, 6, 3, 16
    q, k, v = _rand((B, S, Hq, D), rng), _rand((B, S, Hkv, D), rng), _rand((B, S, Hkv, D), rng)
    perm = rng.permutation(S)
    a, la = oracle.attention(q, k, v, scale=0.25)
    b_, lb = oracle.attention(q, k[:, perm], v[:, perm], scale=0.25)
    np.testing.assert_allclose(a, b_, atol=1e-12)
    np.testing.assert_allclose(la, lb, atol=1e-12)


def test_empty_key_set_gives_zero_output_and_minus_inf_lse():
    rng = np.random.default_rng(14)
    B, S, Hq, Hkv, D = 2, 6, 2, 1, 4
    q, k, v = _rand((B, S, Hq, D), rng), _rand((B, S, Hkv, D), rng), _rand((B, S, Hkv, D), rng)
    out, lse = oracle.attention(q, k, v, scale=1.0, seqlens_k=[0, 6])
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))
    # causal with Sq > Sk: the first Sq - Sk rows have no admissible key
    out2, lse2 = oracle.attention(q, k[:, :3], v[:, :3], scale=1.0, causal=True)
    assert np.all(out2[:, :3] == 0) and np.all(np.isneginf(lse2[:, :, :3]))


def test_two_key_closed_form_and_hand_worked_golden():
    lines = [ln for ln in open(os.path.join(GOLDEN, "two_key_example.txt"))
             if ln.strip() and not ln.startswith("#")]
    vals = [float(x) for x in lines[0].split()]
    q = np.array([[[[1, 0]]]], np.float32)
    k = np.array([[[[2, 0]], [[0, 3]]]], np.float32)
    v = np.array([[[[1, 0]], [[0, 1]]]], np.float32)
    out, lse = oracle.attention(q, k, v, scale=0.5)
    np.testing.assert_allclose(out.ravel(), vals[:2], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse.ravel(), vals[2:], rtol=0, atol=1e-15)
    # general two-key closed form: weights are the logistic function of s0 - s1
    rng = np.random.default_rng(15)
    q, k, v = _rand((1, 1, 1, 8), rng), _rand((1, 2, 1, 8), rng), _rand((1, 2, 1, 8), rng)
    out, lse = oracle.attention(q, k, v, scale=0.9)
    s = 0.9 * (k[0, :, 0].astype(np.float64) @ q[0, 0, 0].astype(np.float64))
    w0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
    ref = w0 * v[0, 0, 0].astype(np.float64) + (1 - w0) * v[0, 1, 0].astype(np.float64)
    np.testing.assert_allclose(out.ravel(), ref, atol=1e-14)
    np.testing.assert_allclose(lse.ravel(), max(s) + math.log1p(math.exp(-abs(s[0] - s[1]))),
                               atol=1e-14)


def test_row_sampling_returns_the_same_rows():
    rng = np.random.default_rng(16)
    B, S, Hq, Hkv, D = 2, 17, 6, 2, 8
    q, k, v = _rand((B, S, Hq, D), rng), _rand((B, S, Hkv, D), rng), _rand((B, S, Hkv, D), rng)
    full, lfull = oracle.attention(q, k, v, scale=0.3, causal=True, seqlens_k=[17, 8])
    rows = np.array([0, 5, 17 * 6 - 1, 17 * 6, 2 * 17 * 6 - 1], np.int64)
    part, lpart = oracle.attention(q, k, v, scale=0.3, causal=True, seqlens_k=[17, 8], rows=rows)
    for r, idx in enumerate(rows):
        i, h, b = idx % S, (idx // S) % Hq, idx // (S * Hq)
        np.testing.assert_array_equal(part[r], full[b, i, h])
        assert lpart[r] == lfull[b, h, i]


def test_decode_is_one_query_row_over_the_cache():
    rng = np.random.default_rng(17)
    B, Hq, Hkv, D, Smax = 3, 8, 2, 8, 12
    q = _rand((B, Hq, D), rng)
    kc, vc = _rand((B, Smax, Hkv, D), rng), _rand((B, Smax, Hkv, D), rng)
    lens = [12, 1, 7]
    out, lse = oracle.decode(q, kc, vc, lens, scale=0.33)
    bout, blse = brute.attention(_tolist(q.reshape(B, 1, Hq, D)), _tolist(kc), _tolist(vc), 0.33,
                                 False, lens)
    np.testing.assert_allclose(out, np.array(bout).reshape(B, Hq, D), atol=1e-12)
    np.testing.assert_allclose(lse, np.array(blse).reshape(B, Hq), atol=1e-12)


def test_oracle_rejects_indivisible_heads():
    q = np.zeros((1, 2, 3, 4), np.float32)
    k = np.zeros((1, 2, 2, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.attention(q, k, k, scale=1.0)


def test_bf16_workload_inputs_are_exact_in_float32():
    w = inputs.make_prefill(1, 4, 2, 8, 8, 64, seed=0, lens=(3, 8), dtype="bf16")
    assert w["q"].dtype == torch.bfloat16
    assert torch.equal(w["q"].float().to(torch.bfloat16), w["q"])
    assert 3 <= int(w["seqlens_k"][0]) <= 8


# ------------------------------------------------------------ byte model pins

def test_kv_cache_byte_model_matches_page_figures():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "kv_cache_bytes.txt"))
            if ln.strip() and not ln.startswith("#")]
    for label, h, g, ratio, red in rows:
        h, g, ratio, red = int(h), int(g), float(ratio), float(red)
        mha = roofline.kv_cache_bytes(1, h, 128, 4096)
        gqa = roofline.kv_cache_bytes(1, g, 128, 4096)
        assert mha / gqa == ratio, label
        assert 100.0 * (1 - gqa / mha) == red, label
    # 2 * L * G * d_k * n elements
    assert roofline.kv_cache_bytes(2, 3, 64, 10, elem_bytes=1) == 2 * 2 * 3 * 64 * 10


def test_flop_model_counts_only_admissible_pairs():
    # causal square: S(S+1)/2 pairs per head
    assert roofline.prefill_pairs(1, 1, 7, 7, True) == 28
    assert roofline.prefill_pairs(2, 3, 5, 5, False, [5, 2]) == 3 * 5 * 7
    assert roofline.prefill_flops(4, 32, 8192, 8192, 128, True) == 4 * 4 * 32 * 128 * 8192 * 8193 // 2


# ------------------------------------------------------ packed (varlen) oracle

def _varlen_cases(n, seed):
    rng = random.Random(seed)
    cases = []
    for _ in range(n):
        Hkv = rng.choice([1, 2])
        G = rng.choice([1, 2, 3, 4])
        B = rng.randint(1, 4)
        lq = [rng.choice([0, 1, 2, 5, 9]) for _ in range(B)]
        lk = [rng.choice([0, 1, 3, 6, 11]) for _ in range(B)]
        spare = rng.choice([0, 0, 2])      # packed rows after the last sequence
        if sum(lq) + spare == 0:
            spare = 1                       # at least one packed query row
        cases.append((B, G * Hkv, Hkv, lq, lk, spare, rng.choice([1, 4, 8]), rng.random() < 0.5,
                      rng.choice([0.35, -0.6, 1.3]), rng.randint(0, 1 << 30)))
    return cases


def _cu(lens):
    return [0] + list(np.cumsum(lens).astype(int))


@pytest.mark.parametrize("case", _varlen_cases(60, 777))
def test_varlen_oracle_matches_packed_brute_force(case):
    B, Hq, Hkv, lq, lk, spare, D, causal, scale, seed = case
    rng = np.random.default_rng(seed)
    tq, tk = sum(lq) + spare, max(sum(lk), 1)
    q, k, v = _rand((tq, Hq, D), rng), _rand((tk, Hkv, D), rng), _rand((tk, Hkv, D), rng)
    cq, ck = _cu(lq), _cu(lk)
    out, lse = oracle.attention_varlen(q, k, v, cq, ck, scale=scale, causal=causal)
    bo, bl = brute.attention_packed(_tolist(q), _tolist(k), _tolist(v), cq, ck, scale, causal)
    np.testing.assert_allclose(out, np.array(bo), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl), rtol=1e-12, atol=1e-12)


def test_varlen_equals_padded_dense_oracle_exactly():
    # every sequence has Sq query rows; keys are right-padded to Sk in the
    # dense batch and given per sequence through seqlens_k
    rng = np.random.default_rng(5)
    B, Hq, Hkv, Sq, Sk, D = 3, 8, 2, 7, 13, 16
    lk = [13, 4, 9]
    qd = _rand((B, Sq, Hq, D), rng)
    kd, vd = _rand((B, Sk, Hkv, D), rng), _rand((B, Sk, Hkv, D), rng)
    od, ld = oracle.attention(qd, kd, vd, scale=0.2, seqlens_k=np.array(lk, np.int32))
    qp = qd.reshape(B * Sq, Hq, D)
    kp = np.concatenate([kd[b, :lk[b]] for b in range(B)])
    vp = np.concatenate([vd[b, :lk[b]] for b in range(B)])
    op, lp = oracle.attention_varlen(qp, kp, vp, _cu([Sq] * B), _cu(lk), scale=0.2)
    assert np.array_equal(op.reshape(B, Sq, Hq, D), od)
    assert np.array_equal(lp.reshape(Hq, B, Sq).transpose(1, 0, 2), ld)


def test_varlen_sequence_order_permutes_rows_exactly():
    rng = np.random.default_rng(9)
    lq, lk, Hq, Hkv, D = [3, 5, 2], [4, 2, 6], 4, 2, 8
    seqs = [(_rand((lq[b], Hq, D), rng), _rand((lk[b], Hkv, D), rng), _rand((lk[b], Hkv, D), rng))
            for b in range(3)]

    def run(order):
        q = np.concatenate([seqs[b][0] for b in order])
        k = np.concatenate([seqs[b][1] for b in order])
        v = np.concatenate([seqs[b][2] for b in order])
        o, l = oracle.attention_varlen(q, k, v, _cu([lq[b] for b in order]), _cu([lk[b] for b in order]),
                                       scale=0.4, causal=True)
        starts = dict(zip(order, _cu([lq[b] for b in order])))
        return {b: (o[starts[b]:starts[b] + lq[b]], l[:, starts[b]:starts[b] + lq[b]]) for b in order}

    a, b_ = run([0, 1, 2]), run([2, 0, 1])
    for s in range(3):
        assert np.array_equal(a[s][0], b_[s][0]) and np.array_equal(a[s][1], b_[s][1])


# ------------------------------------------------------------ FP8 KV decode

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fp8_decode_oracle_matches_brute_force_on_dequantised_values(seed):
    # brute force on k_scale * k8 and v_scale * v8 formed exactly in fp64:
    # pins the folding of k_scale into the softmax scale and v_scale into out
    d = inputs.make_decode_fp8(2, 4, 2, 8, 9, seed=seed, lens=(0, 9))
    out, lse = oracle.decode_fp8(d["q"], d["kcache"], d["vcache"], d["k_scale"], d["v_scale"],
                                 d["cache_seqlens"], scale=0.3)
    qf = d["q"].float().numpy().astype(np.float64)
    kf = d["kcache"].float().numpy().astype(np.float64) * d["k_scale"]
    vf = d["vcache"].float().numpy().astype(np.float64) * d["v_scale"]
    lens = d["cache_seqlens"].tolist()
    bo, bl = brute.attention(qf[:, None].tolist(), kf.tolist(), vf.tolist(), 0.3, False, lens)
    np.testing.assert_allclose(out, np.array(bo)[:, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(bl)[:, :, 0], rtol=1e-12, atol=1e-12)


def test_fp8_decode_with_unit_scales_is_decode_on_the_e4m3_values():
    d = inputs.make_decode_fp8(3, 8, 2, 16, 20, seed=4, lens=(1, 20))
    a, la = oracle.decode_fp8(d["q"], d["kcache"], d["vcache"], 1.0, 1.0, d["cache_seqlens"], scale=0.25)
    b, lb = oracle.decode(d["q"], d["kcache"].float(), d["vcache"].float(), d["cache_seqlens"], scale=0.25)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_e4m3_quantisation_is_finite_and_within_half_an_ulp():
    x = torch.randn(4096, generator=torch.Generator().manual_seed(0)) * 3
    x8, s = inputs.quantize_e4m3(x)
    y = x8.float()
    assert torch.isfinite(y).all() and float(y.abs().max()) == 448.0
    # e4m3 keeps 3 mantissa bits: relative rounding error <= 2^-4 for normal values
    rel = ((y * s - x).abs() / x.abs().clamp_min(1e-30))[x.abs() / s >= 2 ** -6]
    assert float(rel.max()) <= 2 ** -4 + 1e-7


# ------------------------------------------------------------ block-sparse

def _bm_cases(n, seed):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        bs = rng.choice([1, 2, 4])
        Sq, Sk = rng.randint(1, 13), rng.randint(1, 13)
        Hkv = rng.choice([1, 2])
        out.append((rng.choice([1, 2]), Hkv * rng.choice([1, 2, 3]), Hkv, Sq, Sk, rng.choice([1, 4]), bs,
                    rng.random() < 0.5, rng.random() < 0.5, rng.choice([0.4, -0.8]), rng.randint(0, 1 << 30)))
    return out


@pytest.mark.parametrize("case", _bm_cases(60, 4242))
def test_blockmask_oracle_matches_brute_force(case):
    B, Hq, Hkv, Sq, Sk, D, bs, causal, padded, scale, seed = case
    rng = np.random.default_rng(seed)
    q, k, v = _rand((B, Sq, Hq, D), rng), _rand((B, Sk, Hkv, D), rng), _rand((B, Sk, Hkv, D), rng)
    bm = (rng.random(((Sq + bs - 1) // bs, (Sk + bs - 1) // bs)) < 0.6).astype(np.uint8)
    lens = [int(x) for x in rng.integers(0, Sk + 1, B)] if padded else None
    out, lse = oracle.attention_blockmask(q, k, v, bm, bs, scale=scale, causal=causal, seqlens_k=lens)
    bo, bl = brute.attention_blockmask(_tolist(q), _tolist(k), _tolist(v), scale, bm.tolist(), bs, causal, lens)
    np.testing.assert_allclose(out, np.array(bo), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_blockmask_all_ones_is_the_dense_oracle(causal):
    rng = np.random.default_rng(1)
    q, k, v = _rand((2, 50, 8, 16), rng), _rand((2, 70, 2, 16), rng), _rand((2, 70, 2, 16), rng)
    lens = np.array([70, 33], np.int32)
    bm = np.ones(((50 + 63) // 64, (70 + 63) // 64), np.uint8)
    a, la = oracle.attention_blockmask(q, k, v, bm, 64, scale=0.2, causal=causal, seqlens_k=lens)
    b, lb = oracle.attention(q, k, v, scale=0.2, causal=causal, seqlens_k=lens)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(la, lb, rtol=1e-12, atol=1e-12)


def test_block_diagonal_mask_is_separate_attention_per_segment():
    # with only the diagonal blocks kept, each segment of bs queries attends to
    # its own bs keys: the dense oracle on that segment alone
    rng = np.random.default_rng(2)
    bs, nb = 4, 3
    q, k, v = _rand((1, bs * nb, 4, 8), rng), _rand((1, bs * nb, 2, 8), rng), _rand((1, bs * nb, 2, 8), rng)
    out, lse = oracle.attention_blockmask(q, k, v, np.eye(nb, dtype=np.uint8), bs, scale=0.5)
    for s in range(nb):
        sl = slice(s * bs, (s + 1) * bs)
        o, l = oracle.attention(q[:, sl], k[:, sl], v[:, sl], scale=0.5)
        np.testing.assert_allclose(out[:, sl], o, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[:, :, sl], l, rtol=1e-12, atol=1e-12)


def test_empty_block_mask_gives_zero_output_and_minus_inf_lse():
    rng = np.random.default_rng(3)
    q, k, v = _rand((1, 5, 2, 4), rng), _rand((1, 6, 1, 4), rng), _rand((1, 6, 1, 4), rng)
    out, lse = oracle.attention_blockmask(q, k, v, np.zeros((1, 1), np.uint8), 8)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ------------------------------------------------------------------ backward

def _torch_reference_grads(q, k, v, do, scale, causal, lens):
    # torch autograd in fp64 on the CPU (a library routine): GQA as MHA on K/V
    # heads repeated per group, keys past the length or the diagonal masked
    qt = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    kt = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    vt = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    kr = kt.repeat_interleave(G, dim=2).permute(0, 2, 3, 1)     # [B,Hq,D,Sk]
    vr = vt.repeat_interleave(G, dim=2).permute(0, 2, 1, 3)     # [B,Hq,Sk,D]
    s = scale * (qt.permute(0, 2, 1, 3) @ kr)                    # [B,Hq,Sq,Sk]
    ii = torch.arange(Sq)[:, None]
    jj = torch.arange(Sk)[None, :]
    mask = torch.stack([(jj < (Sk if lens is None else lens[b])) & ((jj <= ii + Sk - Sq) if causal else True)
                        for b in range(B)])[:, None]
    s = s.masked_fill(~mask, float("-inf"))
    out = torch.softmax(s, dim=-1) @ vr                          # [B,Hq,Sq,D]
    out.permute(0, 2, 1, 3).backward(torch.tensor(do, dtype=torch.float64))
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


@pytest.mark.parametrize("causal,lens", [(False, None), (True, None), (False, [5, 9])])
def test_backward_oracle_matches_torch_autograd(causal, lens):
    rng = np.random.default_rng(11)
    B, Sq, Sk, Hq, Hkv, D = 2, 7, 9, 6, 2, 8
    q, k, v = _rand((B, Sq, Hq, D), rng), _rand((B, Sk, Hkv, D), rng), _rand((B, Sk, Hkv, D), rng)
    do = _rand((B, Sq, Hq, D), rng)
    got = oracle.attention_backward(q, k, v, do, scale=0.4, causal=causal, seqlens_k=lens)
    ref = _torch_reference_grads(q, k, v, do, 0.4, causal, lens)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-12)


def test_backward_oracle_matches_central_differences():
    # d<dO, out>/dx by central differences of the forward oracle (fp64)
    rng = np.random.default_rng(12)
    q, k, v = _rand((1, 3, 4, 2), rng), _rand((1, 4, 2, 2), rng), _rand((1, 4, 2, 2), rng)
    do = _rand((1, 3, 4, 2), rng)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, scale=0.7, causal=True)

    def loss(qq, kk, vv):
        o, _ = oracle.attention(qq.astype(np.float32), kk.astype(np.float32), vv.astype(np.float32), scale=0.7,
                                causal=True)
        return float((o * do).sum())
    def loss_with(which, x):
        args = [q, k, v]
        args[which] = x
        return loss(*args)
    eps = 1e-3
    for which, (x, g) in enumerate(((q, dq), (k, dk), (v, dv))):
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            fd = (loss_with(which, xp) - loss_with(which, xm)) / (2 * eps)
            assert abs(fd - g[idx]) <= 2e-4 * max(1.0, abs(g[idx])), (idx, fd, g[idx])


@pytest.mark.parametrize("causal,lens,G", [(False, None, 4), (True, None, 2), (True, [6, 0], 3), (False, [9, 3], 1)])
def test_backward_dq_rows_are_the_full_oracle_rows(causal, lens, G):
    # the row-by-row dQ (for checks at full size) against the full oracle gradient
    rng = np.random.default_rng(21 + G)
    B, Sq, Sk, Hkv, D = 2, 7, 9, 2, 8
    Hq = Hkv * G
    q, k, v = _rand((B, Sq, Hq, D), rng), _rand((B, Sk, Hkv, D), rng), _rand((B, Sk, Hkv, D), rng)
    do = _rand((B, Sq, Hq, D), rng)
    dq, _, _ = oracle.attention_backward(q, k, v, do, scale=0.3, causal=causal, seqlens_k=lens)
    rows = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(Sq)]
    got = oracle.attention_backward_dq_rows(q, k, v, do, rows, scale=0.3, causal=causal, seqlens_k=lens)
    ref = np.stack([dq[b, i, h] for b, h, i in rows])
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)
