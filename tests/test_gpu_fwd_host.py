"""gqa_fwd_host (inputs and outputs in host memory, copies pipelined with the
computation by batch chunks) against gqa_fwd on the device, through the C
ABI.  Each chunk is one gqa_fwd launch over the same inputs, so the outputs
must agree bit for bit, for every chunking of the batch; and against the
oracle at the forward's tolerance.
"""
import numpy as np
import pytest
import torch

import grouped_query_attention_08_b300 as gqa
from grouped_query_attention_08_b300 import build, inputs
from parity import compare, compare_lse, oracle_fwd, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    gqa.load_library()


def _pinned(d):
    return {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


# (B, Hq, Hkv, Sq, Sk, D, causal, lens, dtype, chunk_b)
CASES = [
    (7, 12, 3, 300, 300, 64, False, (100, 300), "bf16", 0),    # automatic chunks (1 per entry)
    (7, 12, 3, 300, 300, 64, False, (100, 300), "bf16", 3),    # ragged last chunk
    (5, 8, 2, 257, 333, 128, True, None, "bf16", 2),           # causal, no key lengths
    (4, 24, 4, 129, 200, 64, False, (0, 200), "bf16", 4),      # one chunk, an empty key set possible
    (3, 4, 2, 70, 90, 64, True, (1, 90), "fp32", 1),           # fp32 check path
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dHq%dHkv%dSq%dSk%dD%d%s_%s_cb%d" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n", c[8], c[9]))
def test_host_pipeline_equals_device_call(case):
    B, Hq, Hkv, Sq, Sk, D, causal, lens, dtype, cb = case
    inp = inputs.make_prefill(B, Hq, Hkv, Sq, Sk, D, seed=B + Sq, lens=lens, dtype=dtype)
    d = to_dev(inp)
    ref_o, ref_l = gqa.gqa_fwd(d["q"], d["k"], d["v"], causal=causal, seqlens_k=d["seqlens_k"], scale=0.1)
    h = _pinned(inp)
    out, lse = gqa.gqa_fwd_host(h["q"], h["k"], h["v"], causal=causal, seqlens_k=h["seqlens_k"], scale=0.1,
                                chunk_b=cb)
    torch.cuda.current_stream().synchronize()
    assert gqa.gqa_device_status() == 0
    assert torch.equal(out, ref_o.cpu()) and torch.equal(lse, ref_l.cpu())
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    ro, rl = oracle_fwd(inp, 0.1, causal)
    compare(out.float().numpy(), ro, tdt)
    compare_lse(lse.numpy(), rl, tdt)


def test_host_pipeline_without_lse_and_reused_staging():
    inp = inputs.make_prefill(6, 12, 3, 200, 200, 64, seed=3, lens=(50, 200), dtype="bf16")
    h = _pinned(inp)
    staging = {}
    outs = []
    for _ in range(2):        # the second call reuses the staging buffers the first allocated
        out, lse = gqa.gqa_fwd_host(h["q"], h["k"], h["v"], seqlens_k=h["seqlens_k"], scale=0.125,
                                    return_lse=False, staging=staging, chunk_b=2)
        assert lse is None
        outs.append(out)
    torch.cuda.current_stream().synchronize()
    d = to_dev(inp)
    ref, _ = gqa.gqa_fwd(d["q"], d["k"], d["v"], seqlens_k=d["seqlens_k"], scale=0.125)
    for out in outs:
        assert torch.equal(out, ref.cpu())
    assert set(staging) == {"q", "k", "v", "out", "seqlens"}
