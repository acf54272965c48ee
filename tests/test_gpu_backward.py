"""GPU parity of gqa_bwd (dQ, dK, dV of grouped-query attention) against the
fp64 oracle, through the C ABI.

The kernel is given the forward's output and log-sum-exp.  The main cases
take both from the oracle's forward (rounded to bf16 / fp32 as the API
stores them), so that only the backward kernels are under test; one case
chains the library's own forward.

Tolerance (bf16 inputs and outputs, fp32 accumulation, P and dS rounded to
bf16 before the products, Dsum formed from the bf16 forward output): each
gradient rounds to bf16 on output (relative 2^-9), and the per-product
roundings add errors of the same relative size that partly cancel over the
sums.  The test asks for relative L2 error <= 1e-2 and max-abs error <=
2e-2 * max |ref| + 1e-4 for every gradient tensor.  The absolute floor
covers gradients that vanish exactly: with one admissible key P = 1 and
dS = dO.v - dO.O = 0 in exact arithmetic, but the kernel's Dsum uses the
bf16-rounded O, leaving |dS| ~ 2^-9 |dO| |O|, i.e. dq ~ 1e-7 here.
"""
import numpy as np
import pytest
import torch

import grouped_query_attention_08_b300 as gqa
import oracle
from grouped_query_attention_08_b300 import build, inputs

pytestmark = pytest.mark.gpu

REL_L2, MAX_REL, ABS_FLOOR = 1e-2, 2e-2, 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    gqa.load_library()


def _cmp(got, ref, what):
    got = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), "%s has non-finite values" % what
    err = np.abs(got - ref)
    scale = max(float(np.abs(ref).max()), 1e-30)
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    msg = "%s: rel-l2 %.3g, max-abs %.3g of max|ref| %.3g" % (what, rel, float(err.max()), scale)
    assert float(err.max()) <= MAX_REL * scale + ABS_FLOOR, msg
    if np.linalg.norm(ref) > 1e3 * ABS_FLOOR:
        assert rel <= REL_L2, msg


def _oracle_fwd(inp, scale, causal):
    out, lse = oracle.attention(inp["q"], inp["k"], inp["v"], scale=scale, causal=causal,
                                seqlens_k=inp.get("seqlens_k"))
    return (torch.from_numpy(np.ascontiguousarray(out)).to(torch.bfloat16),
            torch.from_numpy(np.ascontiguousarray(lse)).to(torch.float32))


def _run(inp, out, lse, scale, causal):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    dq, dk, dv = gqa.gqa_bwd(d["q"], d["k"], d["v"], out.cuda(), d["dout"], lse.cuda(), causal=causal,
                             seqlens_k=d["seqlens_k"], scale=scale)
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0
    return dq, dk, dv


# (B, Hq, Hkv, Sq, Sk, D, causal, lens)
CASES = [
    (2, 8, 2, 200, 300, 64, False, (1, 300)),    # G=4, ragged tiles, padded keys
    (1, 12, 3, 256, 256, 64, True, None),        # BERT-style grouping, causal
    (2, 8, 8, 130, 190, 128, False, None),       # MHA, D=128, ragged
    (1, 16, 2, 100, 400, 128, True, None),       # G=8, causal with Sq < Sk
    (1, 4, 1, 300, 120, 64, True, None),         # MQA, causal with Sq > Sk: rows with no key
    (2, 4, 2, 70, 70, 64, False, (0, 70)),       # an empty key set possible
    (1, 2, 1, 1, 1, 128, False, None),           # one query, one key
]


def _ids(c):
    return "B%dHq%dHkv%dSq%dSk%dD%d%s%s" % (c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n",
                                           "_lens" if c[7] else "")


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_bwd_matches_oracle(case):
    B, Hq, Hkv, Sq, Sk, D, causal, lens = case
    inp = inputs.make_backward(B, Hq, Hkv, Sq, Sk, D, seed=Sq * 3 + Sk + D, lens=lens)
    scale = 1.0 / np.sqrt(D)
    out, lse = _oracle_fwd(inp, scale, causal)
    rq, rk, rv = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["dout"], scale=scale, causal=causal,
                                           seqlens_k=inp["seqlens_k"])
    dq, dk, dv = _run(inp, out, lse, scale, causal)
    _cmp(dq, rq, "dq")
    _cmp(dk, rk, "dk")
    _cmp(dv, rv, "dv")


def test_bwd_after_library_forward():
    inp = inputs.make_backward(2, 12, 3, 333, 333, 64, seed=11, lens=(200, 333))
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out, lse = gqa.gqa_fwd(d["q"], d["k"], d["v"], causal=True, seqlens_k=d["seqlens_k"], scale=0.125)
    dq, dk, dv = gqa.gqa_bwd(d["q"], d["k"], d["v"], out, d["dout"], lse, causal=True, seqlens_k=d["seqlens_k"],
                             scale=0.125)
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0
    rq, rk, rv = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["dout"], scale=0.125, causal=True,
                                           seqlens_k=inp["seqlens_k"])
    _cmp(dq, rq, "dq")
    _cmp(dk, rk, "dk")
    _cmp(dv, rv, "dv")


def test_bwd_is_deterministic_and_zero_past_the_key_length():
    inp = inputs.make_backward(2, 8, 2, 150, 260, 128, seed=5, lens=(40, 200))
    out, lse = _oracle_fwd(inp, 0.09, False)
    a = _run(inp, out, lse, 0.09, False)
    b = _run(inp, out, lse, 0.09, False)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    lens = inp["seqlens_k"].tolist()
    for bi, L in enumerate(lens):
        assert torch.all(a[1][bi, L:] == 0) and torch.all(a[2][bi, L:] == 0)


def test_bwd_scheduler_slots_and_side_stream_across_many_calls():
    """dQ claims its tiles from a per-launch counter slot (shared with the
    prefill's, 64 slots reset by each launch's last CTA) and runs on a side
    stream beside dK/dV: 70 backward calls interleaved with prefill calls
    reuse every slot and must keep giving bitwise the first gradients, on
    the caller's stream order (each call's outputs read back on it)."""
    inp = inputs.make_backward(2, 12, 3, 300, 300, 64, seed=8, lens=(90, 300))
    out, lse = _oracle_fwd(inp, 0.125, False)
    first = _run(inp, out, lse, 0.125, False)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    o_d, l_d = out.cuda(), lse.cuda()
    for i in range(70):
        got = gqa.gqa_bwd(d["q"], d["k"], d["v"], o_d, d["dout"], l_d, seqlens_k=d["seqlens_k"], scale=0.125)
        gqa.gqa_fwd(d["q"], d["k"], d["v"], seqlens_k=d["seqlens_k"], scale=0.125)
        if i % 10 == 9:
            for x, y in zip(got, first):
                assert torch.equal(x, y), i
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0


def _full_size(name, seed):
    """The named workload at full size through the library's forward and
    backward, as bench.py times it; dO ~ N(0,1) from `seed`."""
    w = inputs.WORKLOADS[name]
    inp = inputs.make_workload(w)
    g = torch.Generator("cpu").manual_seed(seed)
    dout = torch.randn(tuple(inp["q"].shape), generator=g, dtype=torch.float32).to(torch.bfloat16)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out, lse = gqa.gqa_fwd(d["q"], d["k"], d["v"], causal=w.causal, seqlens_k=d["seqlens_k"], scale=w.scale)
    dq, dk, dv = gqa.gqa_bwd(d["q"], d["k"], d["v"], out, dout.cuda(), lse, causal=w.causal,
                             seqlens_k=d["seqlens_k"], scale=w.scale)
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0
    return w, inp, dout, dq.cpu(), dk.cpu(), dv.cpu()


def test_bwd_bert_base_full_size_two_batch_entries():
    # B = 32 launched whole; batch entries 0 and 21 (all their heads) against the oracle
    w, inp, dout, dq, dk, dv = _full_size("bert_base", 2024)
    for b in (0, 21):
        lens = None if inp["seqlens_k"] is None else inp["seqlens_k"][b:b + 1]
        rq, rk, rv = oracle.attention_backward(inp["q"][b:b + 1], inp["k"][b:b + 1], inp["v"][b:b + 1],
                                               dout[b:b + 1], scale=w.scale, causal=w.causal, seqlens_k=lens)
        _cmp(dq[b:b + 1], rq, "dq[b=%d]" % b)
        _cmp(dk[b:b + 1], rk, "dk[b=%d]" % b)
        _cmp(dv[b:b + 1], rv, "dv[b=%d]" % b)


def test_bwd_bert_large_long_full_size_one_group():
    # B = 8, S = 4096 launched whole; batch entry 5, K/V head 2 and its G = 6 query heads
    w, inp, dout, dq, dk, dv = _full_size("bert_large_long", 2025)
    b, kvh, G = 5, 2, w.Hq // w.Hkv
    hs = slice(kvh * G, (kvh + 1) * G)
    sl = lambda t, heads: t[b:b + 1, :, heads]
    rq, rk, rv = oracle.attention_backward(sl(inp["q"], hs), sl(inp["k"], slice(kvh, kvh + 1)),
                                           sl(inp["v"], slice(kvh, kvh + 1)), sl(dout, hs), scale=w.scale,
                                           causal=w.causal)
    _cmp(sl(dq, hs), rq, "dq")
    _cmp(sl(dk, slice(kvh, kvh + 1)), rk, "dk")
    _cmp(sl(dv, slice(kvh, kvh + 1)), rv, "dv")


def test_bwd_causal_long_full_size_sampled_dq_rows():
    # B = 4, Hq = 32, S = 8192, D = 128, causal, launched whole; 48 sampled
    # (b, h, i) rows of dQ, among them the first and last query rows, each
    # computed on its own by the oracle
    w, inp, dout, dq, dk, dv = _full_size("causal_long", 2026)
    rng = np.random.default_rng(7)
    rows = [(0, 0, 0), (w.B - 1, w.Hq - 1, w.Sq - 1), (1, 5, 1), (2, 17, w.Sq // 2)]
    rows += [(int(rng.integers(w.B)), int(rng.integers(w.Hq)), int(rng.integers(w.Sq))) for _ in range(44)]
    ref = oracle.attention_backward_dq_rows(inp["q"], inp["k"], inp["v"], dout, rows, scale=w.scale,
                                            causal=w.causal)
    got = torch.stack([dq[b, i, h] for b, h, i in rows])
    _cmp(got, ref, "dq rows")
    assert torch.isfinite(dk.float()).all() and torch.isfinite(dv.float()).all()
