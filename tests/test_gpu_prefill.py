"""GPU parity of gqa_fwd (prefill) against the fp64 oracle, through the C ABI.

Small shapes span several 128-key tiles and a ragged tail and are compared
element by element; the full workloads are compared on deterministic row
samples the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import grouped_query_attention_08_b300 as gqa
from grouped_query_attention_08_b300 import build, inputs
from parity import compare, compare_lse, gather_rows, oracle_fwd, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    gqa.load_library()


# (B, Hq, Hkv, Sq, Sk, D, causal, lens)
SMALL = [
    (2, 8, 2, 200, 333, 64, False, (1, 333)),      # G=4, ragged, padding
    (1, 12, 3, 300, 300, 64, False, None),         # BERT-base grouping, several tiles
    (2, 24, 4, 257, 257, 64, False, (100, 257)),   # G=6: 21 tokens x 6 heads per tile
    (2, 8, 8, 130, 130, 128, True, None),          # G=1 (MHA), causal
    (1, 8, 1, 100, 260, 128, True, None),          # G=8 (MQA), causal with Sq < Sk
    (2, 32, 8, 513, 513, 128, True, None),         # long-causal grouping, ragged
    (3, 6, 2, 77, 77, 64, False, (0, 77)),         # G=3, an empty key set possible
    (3, 4, 2, 1, 1, 64, False, None),              # one query, one key
    (1, 16, 2, 64, 64, 64, True, None),            # G=8 causal
    (1, 4, 2, 40, 20, 64, True, None),             # Sq > Sk causal: first rows see no key
    (2, 4, 2, 129, 255, 128, False, (1, 255)),     # G=2, D=128
    (1, 48, 1, 33, 190, 64, False, None),          # G=48: 2 tokens x 48 heads per tile
]


def _run(inp, scale, causal):
    out, lse = gqa.gqa_fwd(inp["q"], inp["k"], inp["v"], causal=causal, seqlens_k=inp["seqlens_k"],
                           scale=scale)
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0
    return out, lse


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B%dHq%dHkv%dSq%dSk%dD%d%s" % (
    s[0], s[1], s[2], s[3], s[4], s[5], "c" if s[6] else "n"))
def test_small_shapes_match_oracle(shape, dtype):
    B, Hq, Hkv, Sq, Sk, D, causal, lens = shape
    inp = inputs.make_prefill(B, Hq, Hkv, Sq, Sk, D, seed=sum(shape[:6]), lens=lens, dtype=dtype)
    scale = 1.0 / np.sqrt(D)
    ref_out, ref_lse = oracle_fwd(inp, scale, causal)
    out, lse = _run(to_dev(inp), scale, causal)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    compare(out.float().cpu().numpy(), ref_out, tdt)
    compare_lse(lse.cpu().numpy(), ref_lse, tdt)
    # rows with no admissible key are exactly zero
    neg = np.isneginf(ref_lse)                         # [B, Hq, Sq]
    if neg.any():
        o = out.float().cpu().numpy().transpose(0, 2, 1, 3)[neg]
        assert np.all(o == 0)


def test_tiny_workload_fp32_and_bf16():
    w = inputs.WORKLOADS["tiny"]
    inp = inputs.make_workload(w)
    ref_out, ref_lse = oracle_fwd(inp, w.scale, w.causal)
    out, lse = _run(to_dev(inp), w.scale, w.causal)
    compare(out.cpu().numpy(), ref_out, torch.float32)
    compare_lse(lse.cpu().numpy(), ref_lse, torch.float32)
    # the bf16 path on the same values rounded to bf16
    inp_b = {k: (v.to(torch.bfloat16) if k in "qkv" else v) for k, v in inp.items()}
    ref_b, ref_lb = oracle_fwd(inp_b, w.scale, w.causal)
    out_b, lse_b = _run(to_dev(inp_b), w.scale, w.causal)
    compare(out_b.float().cpu().numpy(), ref_b, torch.bfloat16)
    compare_lse(lse_b.cpu().numpy(), ref_lb, torch.bfloat16)


def _sample(w, n, seed, extra=()):
    total = w.B * w.Hq * w.Sq
    must = [0, total - 1, w.Sq - 1, w.Sq, total - w.Sq] + list(extra)
    return inputs.sample_rows(total, n, seed, must=must).numpy()


def test_bert_base_workload_every_row():
    """The headline workload at full size, every one of its B * Hq * Sq =
    393,216 output rows against the oracle (a few seconds of oracle time)."""
    w = inputs.WORKLOADS["bert_base"]
    inp = inputs.make_workload(w)
    out, lse = _run(to_dev(inp), w.scale, w.causal)
    ref_o, ref_l = oracle_fwd(inp, w.scale, w.causal)
    compare(out.float().cpu().numpy(), ref_o, torch.bfloat16, what="bert_base")
    compare_lse(lse.cpu().numpy(), ref_l, torch.bfloat16)


@pytest.mark.parametrize("name", ["bert_large_long", "causal_long"])
def test_full_workloads_on_sampled_rows(name):
    w = inputs.WORKLOADS[name]
    inp = inputs.make_workload(w)
    extra = []
    if w.causal:   # rows of (b=0, h=0) along the causal diagonal
        extra = list(range(0, w.Sq, 97))
    rows = _sample(w, 1500, w.seed + 100, extra)
    out, lse = _run(to_dev(inp), w.scale, w.causal)
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all()
    ref_o, ref_l = oracle_fwd(inp, w.scale, w.causal, rows=rows)
    got_o, got_l = gather_rows(o, lse.cpu().numpy(), rows, w.Sq, w.Hq)
    compare(got_o, ref_o, torch.bfloat16, what=name)
    compare_lse(got_l, ref_l, torch.bfloat16)


def test_peaky_scores():
    """Q x 4 concentrates each softmax on a few keys, so the tolerance bites."""
    inp = inputs.make_prefill(2, 12, 3, 300, 300, 64, seed=5, lens=(200, 300), dtype="bf16", q_mult=4.0)
    ref_out, ref_lse = oracle_fwd(inp, 0.125, False)
    out, lse = _run(to_dev(inp), 0.125, False)
    compare(out.float().cpu().numpy(), ref_out, torch.bfloat16)
    compare_lse(lse.cpu().numpy(), ref_lse, torch.bfloat16)


@pytest.mark.parametrize("causal", [False, True])
def test_padded_keys_do_not_change_a_bit(causal):
    inp = inputs.make_prefill(2, 8, 2, 300, 300, 64, seed=9, lens=(50, 250), dtype="bf16")
    d = to_dev(inp)
    out1, lse1 = _run(d, 0.125, causal)
    k2, v2 = d["k"].clone(), d["v"].clone()
    for b, L in enumerate(inp["seqlens_k"].tolist()):
        k2[b, L:] = 1e4
        v2[b, L:] = -1e4
    out2, lse2 = gqa.gqa_fwd(d["q"], k2, v2, causal=causal, seqlens_k=d["seqlens_k"], scale=0.125)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_runs_are_bitwise_deterministic():
    inp = to_dev(inputs.make_prefill(2, 32, 8, 700, 700, 128, seed=3, dtype="bf16"))
    a = _run(inp, 0.088, True)
    b = _run(inp, 0.088, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_gqa_equals_mha_on_repeated_kv():
    inp = to_dev(inputs.make_prefill(2, 12, 3, 200, 200, 64, seed=4, lens=(100, 200), dtype="bf16"))
    out, _ = _run(inp, 0.125, False)
    rep = dict(inp)
    rep["k"] = inp["k"].repeat_interleave(4, dim=2).contiguous()
    rep["v"] = inp["v"].repeat_interleave(4, dim=2).contiguous()
    out_m, _ = _run(rep, 0.125, False)
    compare(out.float().cpu().numpy(), out_m.float().cpu().numpy(), torch.bfloat16,
            max_tol=1e-2, mean_tol=1e-3)


def test_out_of_range_length_reports_bounds_error_and_writes_zeros():
    inp = to_dev(inputs.make_prefill(2, 4, 2, 64, 64, 64, seed=1, dtype="bf16"))
    lens = torch.tensor([64, 65], dtype=torch.int32, device="cuda")
    out, lse = gqa.gqa_fwd(inp["q"], inp["k"], inp["v"], seqlens_k=lens, scale=0.125)
    assert gqa.gqa_device_status() == gqa.GQA_ERR_DEVICE_BOUNDS
    assert gqa.gqa_device_status() == 0           # cleared by the read
    assert torch.all(out[1] == 0)
    assert torch.isneginf(lse[1]).all()


def test_scheduler_slots_are_reset_between_launches():
    """Work units are claimed from a per-launch counter slot that the launch's
    last CTA resets; 130 launches reuse every slot twice and must keep giving
    the same result, on grids of different sizes."""
    small = to_dev(inputs.make_prefill(2, 8, 2, 300, 300, 64, seed=21, lens=(100, 300), dtype="bf16"))
    big = to_dev(inputs.make_prefill(4, 12, 3, 600, 600, 64, seed=22, lens=(200, 600), dtype="bf16"))
    ref_s = _run(small, 0.125, False)
    ref_b = _run(big, 0.125, True)
    for i in range(65):
        out_s, _ = gqa.gqa_fwd(small["q"], small["k"], small["v"], seqlens_k=small["seqlens_k"], scale=0.125)
        out_b, _ = gqa.gqa_fwd(big["q"], big["k"], big["v"], causal=True, seqlens_k=big["seqlens_k"], scale=0.125)
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0
    assert torch.equal(out_s, ref_s[0]) and torch.equal(out_b, ref_b[0])
