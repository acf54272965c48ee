"""GPU parity of gqa_decode_fp8 (FP8 e4m3 KV cache) against the fp64 oracle
on the dequantised cache, through the C ABI.  Held to the bf16 decode's
tolerance: the kernel's products are exact on the e4m3 values (f16
operands, fp32 accumulation), so only P's rounding and the bf16 output add
error.
"""
import numpy as np
import pytest
import torch

import grouped_query_attention_08_b300 as gqa
import oracle
from grouped_query_attention_08_b300 import build, inputs
from parity import compare, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    gqa.load_library()


def _ref(d, scale):
    return oracle.decode_fp8(d["q"], d["kcache"], d["vcache"], d["k_scale"], d["v_scale"], d["cache_seqlens"],
                             scale=scale)


def _run(d, scale, ns):
    out = gqa.gqa_decode_fp8(d["q"], d["kcache"], d["vcache"], d["cache_seqlens"], d["k_scale"], d["v_scale"],
                             scale=scale, num_splits=ns)
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0
    return out.float().cpu().numpy()


# (B, Hq, Hkv, Smax, lengths)
SHAPES = [
    (4, 64, 8, 700, (1, 700)),     # G=8, ragged blocks
    (3, 16, 16, 300, (0, 300)),    # G=1, an empty cache possible
    (2, 12, 3, 129, (100, 129)),   # G=4
    (5, 8, 4, 33, (1, 33)),        # G=2, one 16-key block and a ragged tail
    (2, 40, 8, 1000, (990, 1000)), # G=5
    (2, 24, 6, 400, (1, 400)),     # G=4, six K/V heads: a CTA's last two warps have no head
]


@pytest.mark.parametrize("ns", [1, 0, 7])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dS%d" % s[:4])
def test_fp8_decode_matches_oracle(shape, ns):
    B, Hq, Hkv, Smax, lens = shape
    inp = inputs.make_decode_fp8(B, Hq, Hkv, 128, Smax, seed=B + Hq + Smax, lens=lens)
    scale = 1.0 / np.sqrt(128)
    ref, _ = _ref(inp, scale)
    got = _run(to_dev(inp), scale, ns)
    compare(got, ref, torch.bfloat16, what="fp8 decode ns=%d" % ns)


@pytest.mark.parametrize("q_mult", [3.0e4, 1.0e-5])
def test_fp8_decode_q_magnitudes_outside_f16(q_mult):
    # q far above f16's largest value or far below its normal range: the
    # kernel's power-of-two scaling of q keeps the products exact
    inp = inputs.make_decode_fp8(2, 16, 2, 128, 200, seed=9, lens=(150, 200), q_mult=q_mult)
    scale = 1.0 / np.sqrt(128)
    ref, _ = _ref(inp, scale / q_mult)
    d = to_dev(inp)
    got = gqa.gqa_decode_fp8(d["q"], d["kcache"], d["vcache"], d["cache_seqlens"], d["k_scale"], d["v_scale"],
                             scale=scale / q_mult).float().cpu().numpy()
    assert gqa.gqa_device_status() == 0
    compare(got, ref, torch.bfloat16, what="q x %g" % q_mult)


def test_llama_decode_fp8_workload_full():
    w = inputs.WORKLOADS["llama_decode_fp8"]
    inp = inputs.make_workload(w)
    ref, _ = _ref(inp, w.scale)
    d = to_dev(inp)
    for ns in (0, 8):
        compare(_run(d, w.scale, ns), ref, torch.bfloat16, what="llama_decode_fp8 ns=%d" % ns)


def test_fp8_decode_out_of_range_length_reports_bounds():
    inp = to_dev(inputs.make_decode_fp8(2, 8, 2, 128, 64, seed=2, lens=(10, 64)))
    inp["cache_seqlens"][1] = 65
    gqa.gqa_decode_fp8(inp["q"], inp["kcache"], inp["vcache"], inp["cache_seqlens"], inp["k_scale"],
                       inp["v_scale"], num_splits=1)
    assert gqa.gqa_device_status() == gqa.GQA_ERR_DEVICE_BOUNDS
