"""GPU parity of gqa_fwd_sparse (block-sparse attention) against the fp64
oracle, through the C ABI.

The oracle applies the block mask to every (query, key) pair; the kernel
skips whole 128-key tiles that no query of a unit keeps and masks the rest
per row, so masks with a mix of kept and dropped blocks inside a unit are
the interesting cases.
"""
import numpy as np
import pytest
import torch

import grouped_query_attention_08_b300 as gqa
import oracle
from grouped_query_attention_08_b300 import build, inputs
from parity import compare, compare_lse, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    gqa.load_library()


def _ref(inp, bm, bs, scale, causal):
    return oracle.attention_blockmask(inp["q"], inp["k"], inp["v"], bm, bs, scale=scale, causal=causal,
                                      seqlens_k=inp.get("seqlens_k"))


def _run(d, bm, bs, scale, causal):
    out, lse = gqa.gqa_fwd_sparse(d["q"], d["k"], d["v"], bm, bs, causal=causal, seqlens_k=d["seqlens_k"],
                                  scale=scale)
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0
    return out, lse


# (B, Hq, Hkv, Sq, Sk, D, causal, lens, block size, pattern)
CASES = [
    (2, 8, 2, 500, 700, 64, False, (1, 700), 64, "random"),     # G=4, half-tile blocks, padding
    (2, 12, 3, 640, 640, 64, False, None, 128, "band"),         # BERT grouping, band
    (1, 24, 4, 384, 512, 64, False, None, 64, "random"),        # G=6: units straddle query blocks
    (2, 8, 8, 300, 300, 128, True, None, 128, "random"),        # MHA, causal, D=128
    (1, 16, 2, 256, 1000, 128, True, None, 64, "band"),         # G=8, causal with Sq < Sk
    (2, 4, 2, 129, 130, 64, False, (0, 130), 128, "random"),    # an empty key set possible
]


def _ids(c):
    return "B%dHq%dHkv%dSq%dSk%dD%d%s_bs%d_%s" % (c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n",
                                                 c[8], c[9])


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_sparse_matches_oracle(case, dtype):
    B, Hq, Hkv, Sq, Sk, D, causal, lens, bs, pattern = case
    inp = inputs.make_prefill(B, Hq, Hkv, Sq, Sk, D, seed=Sq + Sk + D, lens=lens, dtype=dtype)
    bm = inputs.make_block_mask((Sq + bs - 1) // bs, (Sk + bs - 1) // bs, pattern, window=1, density=0.45,
                                seed=Sq)
    scale = 1.0 / np.sqrt(D)
    ref_out, ref_lse = _ref(inp, bm, bs, scale, causal)
    out, lse = _run(to_dev(inp), bm.cuda(), bs, scale, causal)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    compare(out.float().cpu().numpy(), ref_out, tdt)
    compare_lse(lse.cpu().numpy(), ref_lse, tdt)


@pytest.mark.parametrize("bs,causal", [(64, False), (128, True)])
def test_all_ones_mask_is_the_dense_kernel_bitwise(bs, causal):
    d = to_dev(inputs.make_prefill(2, 12, 3, 500, 600, 64, seed=3, lens=(300, 600), dtype="bf16"))
    bm = torch.ones(((500 + bs - 1) // bs, (600 + bs - 1) // bs), dtype=torch.uint8, device="cuda")
    a, la = _run(d, bm, bs, 0.125, causal)
    b, lb = gqa.gqa_fwd(d["q"], d["k"], d["v"], causal=causal, seqlens_k=d["seqlens_k"], scale=0.125)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_empty_mask_gives_zeros_and_minus_inf():
    d = to_dev(inputs.make_prefill(1, 8, 2, 200, 300, 64, seed=4, dtype="bf16"))
    bm = torch.zeros((2, 3), dtype=torch.uint8, device="cuda")
    out, lse = _run(d, bm, 128, 0.125, False)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_sparse_workload_matches_oracle():
    w = inputs.WORKLOADS["bert_large_long_sparse"]
    inp = inputs.make_workload(w)
    base = inputs.WORKLOADS[w.base]
    ref_out, ref_lse = _ref(inp, inp["block_mask"], w.block_size, base.scale, base.causal)
    d = to_dev(inp)
    out, lse = _run(d, d["block_mask"], w.block_size, base.scale, base.causal)
    compare(out.float().cpu().numpy(), ref_out, torch.bfloat16, what="bert_large_long_sparse")
    compare_lse(lse.cpu().numpy(), ref_lse, torch.bfloat16)
