"""GPU parity of gqa_fwd_varlen (packed sequences) against the fp64 oracle,
through the C ABI.

Packed rows are compared element by element with the oracle's per-sequence
definition; rows after the last sequence must keep whatever the caller left
there.  A batch of equal-length sequences must give exactly the dense
kernel's result.
"""
import numpy as np
import pytest
import torch

import grouped_query_attention_08_b300 as gqa
import oracle
from grouped_query_attention_08_b300 import build, inputs
from parity import compare, compare_lse, to_dev

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    gqa.load_library()


# (B, Hq, Hkv, D, causal, query lengths, key lengths or None (= query lengths), spare rows)
CASES = [
    (3, 8, 2, 64, False, [200, 1, 333], None, 0),            # G=4, ragged, a one-row sequence
    (4, 12, 3, 64, False, [300, 0, 64, 65], None, 0),         # empty sequence; 64 = one unit exactly
    (2, 24, 4, 64, False, [257, 100], [120, 257], 0),         # G=6 (21 tokens per tile), Lq != Lk
    (3, 8, 8, 128, True, [130, 7, 260], None, 0),             # MHA, causal, D=128
    (2, 8, 1, 128, True, [100, 40], [260, 20], 0),            # MQA, causal with Lq < Lk and Lq > Lk
    (2, 32, 8, 128, True, [513, 200], None, 3),               # long-causal grouping, spare rows
    (3, 6, 2, 64, False, [77, 33, 5], [0, 77, 3], 2),         # an empty key set, spare rows
    (2, 48, 1, 64, False, [33, 3], [190, 7], 0),              # G=48: 2 tokens x 48 heads per tile
]


def _make(case, dtype):
    B, Hq, Hkv, D, causal, lq, lk, spare = case
    inp = inputs.make_varlen(B, Hq, Hkv, D, seed=sum(lq) + Hq, lens=list(lq),
                             lens_k=None if lk is None else list(lk), dtype=dtype)
    if spare:
        # rows after the last sequence: part of the packed tensors, of no sequence
        pad = torch.zeros((spare,) + tuple(inp["q"].shape[1:]), dtype=inp["q"].dtype)
        inp["q"] = torch.cat([inp["q"], pad])
    return inp


def _run(d, causal, scale, out=None, lse=None):
    o, l = gqa.gqa_fwd_varlen(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"],
                              max_seqlen_q=d["max_seqlen_q"], max_seqlen_k=d["max_seqlen_k"],
                              causal=causal, scale=scale, out=out, lse=lse)
    torch.cuda.synchronize()
    return o, l


def _ids(c):
    return "B%dHq%dHkv%dD%d%s_sp%d" % (c[0], c[1], c[2], c[3], "c" if c[4] else "n", c[7])


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_packed_sequences_match_oracle(case, dtype):
    causal, D = case[4], case[3]
    inp = _make(case, dtype)
    scale = 1.0 / np.sqrt(D)
    ref_out, ref_lse = oracle.attention_varlen(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"],
                                               inp["cu_seqlens_k"], scale=scale, causal=causal)
    d = to_dev(inp)
    out = torch.full_like(d["q"], SENTINEL)
    lse = torch.full((d["q"].shape[1], d["q"].shape[0]), SENTINEL, dtype=torch.float32, device="cuda")
    out, lse = _run(d, causal, scale, out, lse)
    assert gqa.gqa_device_status() == 0
    used = int(inp["cu_seqlens_q"][-1])
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    compare(o[:used], ref_out[:used], tdt)
    compare_lse(l[:, :used], ref_lse[:, :used], tdt)
    # rows after the last sequence are not written
    assert np.all(o[used:] == SENTINEL) and np.all(l[:, used:] == SENTINEL)


@pytest.mark.parametrize("causal,D", [(False, 64), (True, 64), (True, 128)])
def test_equal_lengths_give_the_dense_result_bitwise(causal, D):
    B, S, Hq, Hkv = 3, 300, 12, 3
    dense = to_dev(inputs.make_prefill(B, Hq, Hkv, S, S, D, seed=11, dtype="bf16"))
    od, ld = gqa.gqa_fwd(dense["q"], dense["k"], dense["v"], causal=causal)
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device="cuda")
    ov, lv = gqa.gqa_fwd_varlen(dense["q"].reshape(B * S, Hq, D), dense["k"].reshape(B * S, Hkv, D),
                                dense["v"].reshape(B * S, Hkv, D), cu, cu, max_seqlen_q=S, max_seqlen_k=S,
                                causal=causal)
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0
    assert torch.equal(ov.reshape(B, S, Hq, D), od)
    assert torch.equal(lv.reshape(Hq, B, S).permute(1, 0, 2), ld)


def test_bert_base_varlen_workload_matches_oracle():
    w = inputs.WORKLOADS["bert_base_varlen"]
    inp = inputs.make_workload(w)
    ref_out, ref_lse = oracle.attention_varlen(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"],
                                               inp["cu_seqlens_k"], scale=w.scale)
    out, lse = _run(to_dev(inp), False, w.scale)
    assert gqa.gqa_device_status() == 0
    compare(out.float().cpu().numpy(), ref_out, torch.bfloat16, what="bert_base_varlen out")
    compare_lse(lse.cpu().numpy(), ref_lse, torch.bfloat16)


def test_inconsistent_offsets_report_bounds_and_skip_that_sequence():
    # sequence 1 claims more query rows than max_seqlen_q: it is not written,
    # the others are computed, and the device status reports the bounds error
    inp = inputs.make_varlen(3, 8, 2, 64, seed=3, lens=[50, 120, 40], dtype="bf16")
    ref_out, _ = oracle.attention_varlen(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"],
                                         inp["cu_seqlens_k"], scale=0.125)
    d = to_dev(inp)
    out = torch.full_like(d["q"], SENTINEL)
    out, _ = gqa.gqa_fwd_varlen(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"],
                                max_seqlen_q=100, max_seqlen_k=200, scale=0.125, out=out)
    assert gqa.gqa_device_status() == gqa.GQA_ERR_DEVICE_BOUNDS
    assert gqa.gqa_device_status() == 0          # the status word was cleared
    o = out.float().cpu().numpy()
    assert np.all(o[50:170] == SENTINEL)
    compare(o[:50], ref_out[:50], torch.bfloat16)
    compare(o[170:], ref_out[170:], torch.bfloat16)


def test_varlen_runs_are_bitwise_deterministic():
    d = to_dev(_make(CASES[0], "bf16"))
    a, la = _run(d, False, 0.125)
    b, lb = _run(d, False, 0.125)
    assert torch.equal(a, b) and torch.equal(la, lb)
