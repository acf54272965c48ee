"""Host checks of the seeded input recipes and of the work counts the bench
divides by (no GPU).  The recipes are the only code the oracle and the CUDA
path share, so they are pinned to their stated draw order here."""
import itertools

import numpy as np
import pytest
import torch

from grouped_query_attention_08_b300 import inputs, roofline


def test_prefill_draw_order_is_q_k_v_then_lengths():
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 5, 7, 8
    d = inputs.make_prefill(B, Hq, Hkv, Sq, Sk, D, seed=9, lens=(1, 7), dtype="fp32")
    g = torch.Generator("cpu").manual_seed(9)
    q = torch.randn((B, Sq, Hq, D), generator=g)
    k = torch.randn((B, Sk, Hkv, D), generator=g)
    v = torch.randn((B, Sk, Hkv, D), generator=g)
    lens = torch.randint(1, 8, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    for a, b in ((d["q"], q), (d["k"], k), (d["v"], v), (d["seqlens_k"], lens)):
        assert torch.equal(a, b)
    bf = inputs.make_prefill(B, Hq, Hkv, Sq, Sk, D, seed=9, lens=(1, 7), dtype="bf16")
    assert bf["q"].dtype == torch.bfloat16 and torch.equal(bf["q"], q.to(torch.bfloat16))


@pytest.mark.parametrize("name", ["tiny", "bert_base", "llama_decode_small", "bert_base_varlen"])
def test_named_workloads_are_deterministic(name):
    a, b = inputs.make_workload(name), inputs.make_workload(name)
    assert a.keys() == b.keys()
    for key in a:
        if isinstance(a[key], torch.Tensor):
            assert torch.equal(a[key], b[key]), key
        else:
            assert a[key] == b[key], key


def test_backward_inputs_extend_the_prefill_draws():
    p = inputs.make_prefill(2, 4, 2, 6, 9, 16, seed=5, lens=(2, 9), dtype="bf16")
    d = inputs.make_backward(2, 4, 2, 6, 9, 16, seed=5, lens=(2, 9))
    for key in ("q", "k", "v", "seqlens_k"):
        assert torch.equal(p[key], d[key])
    g = torch.Generator("cpu").manual_seed(5 + 7919)
    assert torch.equal(d["dout"], torch.randn((2, 6, 4, 16), generator=g).to(torch.bfloat16))


def test_e4m3_quantisation_as_a_caller_would_do_it():
    x = torch.randn(4, 33, 2, 16, generator=torch.Generator("cpu").manual_seed(3)) * 7.0
    x8, s = inputs.quantize_e4m3(x)
    assert x8.dtype == torch.float8_e4m3fn
    assert s == pytest.approx(float(x.abs().max()) / 448.0, rel=1e-6)
    back = x8.float() * s
    assert torch.isfinite(back).all() and float(back.abs().max()) <= 448.0 * s * (1 + 1e-6)
    # e4m3 keeps 3 mantissa bits: round to nearest is within 2^-4 relative for normals
    normal = x.abs() >= s * 2.0 ** -6
    assert torch.all((back - x).abs()[normal] <= x.abs()[normal] * 2.0 ** -4 + 1e-12)


def test_block_mask_patterns():
    band = inputs.make_block_mask(6, 8, "band", window=1)
    for qb, kb in itertools.product(range(6), range(8)):
        assert bool(band[qb, kb]) == (abs(qb - kb) <= 1 or kb == 0)
    assert inputs.make_block_mask(3, 4, "ones").all() and not inputs.make_block_mask(3, 4, "zeros").any()
    r1 = inputs.make_block_mask(40, 40, "random", density=0.3, seed=2)
    r2 = inputs.make_block_mask(40, 40, "random", density=0.3, seed=2)
    assert torch.equal(r1, r2) and 0.2 < float(r1.float().mean()) < 0.4
    assert r1.dtype == torch.uint8


def test_varlen_offsets_match_the_lengths():
    d = inputs.make_varlen(4, 8, 2, 64, seed=1, lens=[3, 0, 7, 1], dtype="bf16")
    cu = d["cu_seqlens_q"].tolist()
    assert cu[0] == 0 and [cu[i + 1] - cu[i] for i in range(4)] == [3, 0, 7, 1]
    assert d["q"].shape[0] >= cu[-1] and d["k"].shape[0] >= d["cu_seqlens_k"][-1]
    assert d["max_seqlen_q"] == 7


def _pairs_brute(B, Hq, Sq, Sk, causal, lens, mask=None, bs=None):
    n = 0
    for b in range(B):
        L = Sk if lens is None else lens[b]
        for i in range(Sq):
            for j in range(Sk):
                ok = j < L and (not causal or j <= i + Sk - Sq)
                if mask is not None:
                    ok = ok and bool(mask[i // bs][j // bs])
                n += Hq if ok else 0
    return n


@pytest.mark.parametrize("Sq,Sk,causal,lens", [(5, 7, False, None), (7, 5, True, None), (6, 6, True, [6, 2]),
                                               (9, 4, False, [0, 4])])
def test_prefill_pairs_by_brute_force(Sq, Sk, causal, lens):
    B = 1 if lens is None else len(lens)
    assert roofline.prefill_pairs(B, 3, Sq, Sk, causal, lens) == _pairs_brute(B, 3, Sq, Sk, causal, lens)


@pytest.mark.parametrize("causal,lens,bs", [(False, None, 2), (True, None, 3), (True, [9, 4], 4), (False, [0, 7], 2)])
def test_blockmask_pairs_by_brute_force(causal, lens, bs):
    Sq, Sk = 8, 9
    rng = np.random.default_rng(bs + (7 if causal else 0))
    mask = (rng.random(((Sq + bs - 1) // bs, (Sk + bs - 1) // bs)) < 0.5).astype(np.uint8)
    B = 1 if lens is None else len(lens)
    got = roofline.blockmask_pairs(B, 2, Sq, Sk, causal, mask, bs, lens)
    assert got == _pairs_brute(B, 2, Sq, Sk, causal, lens, mask.tolist(), bs)


def test_varlen_pairs_by_brute_force():
    lq, lk = [3, 0, 5, 4], [4, 2, 5, 0]
    for causal in (False, True):
        want = sum(_pairs_brute(1, 2, a, b, causal, None) for a, b in zip(lq, lk) if a and b)
        assert roofline.varlen_pairs(2, lq, lk, causal) == want
