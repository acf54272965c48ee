"""GPU parity of gqa_decode (split-KV decode + log-sum-exp combine) against the
fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import grouped_query_attention_08_b300 as gqa
from grouped_query_attention_08_b300 import build, inputs
from parity import compare, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    gqa.load_library()


def _decode(d, scale, ns):
    out = gqa.gqa_decode(d["q"], d["kcache"], d["vcache"], d["cache_seqlens"], scale=scale, num_splits=ns)
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0
    return out


def _ref(inp, scale):
    return oracle.decode(inp["q"], inp["kcache"], inp["vcache"], inp["cache_seqlens"], scale=scale)


# (B, Hq, Hkv, D, Smax, lens)
SMALL = [
    (3, 16, 2, 128, 300, (0, 300)),
    (4, 8, 8, 64, 129, (1, 129)),        # G=1
    (2, 8, 1, 128, 1000, (900, 1000)),   # G=8 MQA
    (5, 12, 2, 64, 77, (1, 77)),         # G=6
    (2, 64, 8, 128, 520, (500, 520)),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("ns", [1, 2, 5, 0])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B%dHq%dHkv%dD%dS%d" % s[:5])
def test_small_decode_matches_oracle(shape, ns, dtype):
    B, Hq, Hkv, D, Smax, lens = shape
    inp = inputs.make_decode(B, Hq, Hkv, D, Smax, seed=B + Hq + D, lens=lens, dtype=dtype)
    if shape == SMALL[0]:
        inp["cache_seqlens"][0] = 0           # an empty cache
        inp["cache_seqlens"][1] = Smax        # a full one
    scale = 1.0 / np.sqrt(D)
    ref, _ = _ref(inp, scale)
    out = _decode(to_dev(inp), scale, ns)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    compare(out.float().cpu().numpy(), ref, tdt)
    if shape == SMALL[0]:
        assert torch.all(out[0] == 0)


def test_llama_decode_workload_full():
    w = inputs.WORKLOADS["llama_decode"]
    inp = inputs.make_workload(w)
    ref, _ = _ref(inp, w.scale)
    d = to_dev(inp)
    for ns in (0, 1, 16):
        out = _decode(d, w.scale, ns)
        compare(out.float().cpu().numpy(), ref, torch.bfloat16, what="llama_decode ns=%d" % ns)


def test_split_count_does_not_change_the_fp32_result():
    inp = to_dev(inputs.make_decode(4, 16, 4, 128, 2000, seed=7, lens=(1, 2000), dtype="fp32"))
    outs = [_decode(inp, 0.09, ns) for ns in (1, 2, 4, 8, 0)]
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 1e-6


def test_decode_equals_prefill_with_one_query():
    inp = inputs.make_decode(4, 32, 8, 128, 700, seed=11, lens=(1, 700), dtype="bf16")
    d = to_dev(inp)
    out_d = _decode(d, 0.088, 0)
    q = d["q"].view(4, 1, 32, 128)
    out_p, _ = gqa.gqa_fwd(q, d["kcache"], d["vcache"], seqlens_k=d["cache_seqlens"], scale=0.088)
    torch.cuda.synchronize()
    compare(out_d.float().cpu().numpy(), out_p.view(4, 32, 128).float().cpu().numpy(), torch.bfloat16,
            max_tol=1e-2, mean_tol=1e-3)


def test_decode_runs_are_bitwise_deterministic():
    d = to_dev(inputs.make_decode(8, 64, 8, 128, 3000, seed=2, lens=(1, 3000), dtype="bf16"))
    a = _decode(d, 0.088, 0)
    b = _decode(d, 0.088, 0)
    assert torch.equal(a, b)


def test_keys_past_the_length_are_never_read_into_the_result():
    inp = inputs.make_decode(3, 16, 2, 128, 400, seed=5, lens=(10, 390), dtype="bf16")
    d = to_dev(inp)
    a = _decode(d, 0.088, 3)
    kc, vc = d["kcache"].clone(), d["vcache"].clone()
    for b, L in enumerate(inp["cache_seqlens"].tolist()):
        kc[b, L:] = float("nan")
        vc[b, L:] = float("nan")
    b_ = gqa.gqa_decode(d["q"], kc, vc, d["cache_seqlens"], scale=0.088, num_splits=3)
    torch.cuda.synchronize()
    assert torch.equal(a, b_)


def test_out_of_range_cache_length_reports_bounds_error():
    d = to_dev(inputs.make_decode(2, 8, 1, 128, 64, seed=1, lens=(1, 64), dtype="bf16"))
    d["cache_seqlens"] = torch.tensor([64, 65], dtype=torch.int32, device="cuda")
    out = gqa.gqa_decode(d["q"], d["kcache"], d["vcache"], d["cache_seqlens"], scale=0.1, num_splits=2)
    assert gqa.gqa_device_status() == gqa.GQA_ERR_DEVICE_BOUNDS
    assert torch.all(out[1] == 0)
