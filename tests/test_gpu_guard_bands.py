"""Out-of-range write checks on every output of every entry point.

compute-sanitizer is not available on the GPU pool these tests run on, so
each output buffer (out, lse, dq/dk/dv, dsum, the decode workspace) is handed
to the library as a slice in the middle of a larger allocation whose guard
bands -- 4 KiB before and after -- are filled with a byte pattern.  After the
call the guard bands must be bitwise unchanged: a kernel that wrote one
element past either end of a tensor (a raw store of lse, dsum or the split
partials, or a TMA store box not clipped at the tensor's edge) would change
them.  The shapes are ragged on purpose: group sizes that do not divide 128
(G = 6: 21 tokens per Q tile), Sq not a multiple of the tile, Sk not a
multiple of 128 keys, packed rows after the last sequence, odd split counts.
"""
import pytest
import torch

import grouped_query_attention_08_b300 as gqa
from grouped_query_attention_08_b300 import build, inputs
from parity import to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096            # bytes of guard band on each side (keeps 16-byte alignment)
PATTERN = 0x5A          # guard byte; as bf16 0x5A5A and fp32 0x5A5A5A5A it is a finite number


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    gqa.load_library()


class Guarded:
    """A tensor of `shape` / `dtype` inside a byte buffer with guard bands."""

    def __init__(self, shape, dtype, fill=None):
        n = 1
        for s in shape:
            n *= int(s)
        esz = torch.empty((), dtype=dtype).element_size()
        self.nbytes = n * esz
        self.buf = torch.full((GUARD + self.nbytes + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)
        if fill is not None:
            self.t.fill_(fill)
        assert self.t.is_contiguous() and self.t.data_ptr() % 256 == 0

    def check(self, what):
        torch.cuda.synchronize()
        lo = self.buf[:GUARD]
        hi = self.buf[GUARD + self.nbytes:]
        bad_lo = int((lo != PATTERN).sum())
        bad_hi = int((hi != PATTERN).sum())
        assert bad_lo == 0 and bad_hi == 0, "%s: %d guard bytes changed before, %d after" % (what, bad_lo, bad_hi)


# (B, Hq, Hkv, Sq, Sk, D, causal, lens)
PREFILL = [
    (2, 24, 4, 257, 301, 64, False, (1, 301)),    # G=6: 21 tokens x 6 heads, ragged everything
    (3, 12, 3, 100, 200, 64, True, (0, 200)),     # an empty key set, causal with Sq < Sk
    (2, 8, 8, 130, 129, 128, False, None),        # MHA, D=128, one key past a tile
    (1, 48, 1, 37, 190, 64, False, None),         # G=48: 2 tokens per tile
    (2, 32, 8, 515, 515, 128, True, None),        # long-causal grouping, ragged
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("shape", PREFILL, ids=lambda s: "B%dHq%dHkv%dSq%dSk%dD%d%s" % (
    s[0], s[1], s[2], s[3], s[4], s[5], "c" if s[6] else "n"))
def test_prefill_writes_stay_inside_out_and_lse(shape, dtype):
    B, Hq, Hkv, Sq, Sk, D, causal, lens = shape
    d = to_dev(inputs.make_prefill(B, Hq, Hkv, Sq, Sk, D, seed=sum(shape[:6]), lens=lens, dtype=dtype))
    out = Guarded(d["q"].shape, d["q"].dtype)
    lse = Guarded((B, Hq, Sq), torch.float32)
    gqa.gqa_fwd(d["q"], d["k"], d["v"], causal=causal, seqlens_k=d["seqlens_k"], scale=0.1, out=out.t, lse=lse.t)
    assert gqa.gqa_device_status() == 0
    out.check("out")
    lse.check("lse")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_varlen_writes_stay_inside_out_and_lse(dtype):
    # G = 6, ragged lengths, an empty sequence; three spare packed rows after the last sequence
    vin = inputs.make_varlen(4, 24, 4, 64, seed=7, lens=[257, 0, 33, 100], lens_k=[120, 5, 257, 1], dtype=dtype)
    d = to_dev(vin)
    spare = 3
    total_q = d["q"].shape[0]
    q = torch.cat([d["q"], torch.zeros((spare,) + tuple(d["q"].shape[1:]), dtype=d["q"].dtype, device="cuda")])
    out = Guarded(q.shape, q.dtype, fill=7.0)
    lse = Guarded((24, total_q + spare), torch.float32, fill=7.0)
    gqa.gqa_fwd_varlen(q, d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], max_seqlen_q=257,
                       max_seqlen_k=257, causal=False, out=out.t, lse=lse.t)
    assert gqa.gqa_device_status() == 0
    out.check("out")
    lse.check("lse")
    # the spare rows belong to no sequence and keep the caller's values
    assert torch.all(out.t[total_q:].float() == 7.0)
    assert torch.all(lse.t[:, total_q:] == 7.0)


@pytest.mark.parametrize("bs", [64, 128])
def test_sparse_writes_stay_inside_out_and_lse(bs):
    B, Hq, Hkv, Sq, Sk, D = 2, 24, 4, 301, 333, 64
    d = to_dev(inputs.make_prefill(B, Hq, Hkv, Sq, Sk, D, seed=11, lens=(100, 333), dtype="bf16"))
    bm = inputs.make_block_mask((Sq + bs - 1) // bs, (Sk + bs - 1) // bs, "random", density=0.5, seed=5).cuda()
    out = Guarded(d["q"].shape, d["q"].dtype)
    lse = Guarded((B, Hq, Sq), torch.float32)
    gqa.gqa_fwd_sparse(d["q"], d["k"], d["v"], bm, bs, seqlens_k=d["seqlens_k"], out=out.t, lse=lse.t)
    assert gqa.gqa_device_status() == 0
    out.check("out")
    lse.check("lse")


@pytest.mark.parametrize("shape", [(2, 24, 4, 257, 301, 64, False, (1, 301)),
                                   (2, 8, 2, 130, 130, 128, True, None)],
                         ids=["G6_D64_ragged", "G4_D128_causal"])
def test_backward_writes_stay_inside_dq_dk_dv_dsum(shape):
    B, Hq, Hkv, Sq, Sk, D, causal, lens = shape
    d = to_dev(inputs.make_backward(B, Hq, Hkv, Sq, Sk, D, seed=3, lens=lens))
    out, lse = gqa.gqa_fwd(d["q"], d["k"], d["v"], causal=causal, seqlens_k=d["seqlens_k"], scale=0.1)
    dq = Guarded(d["q"].shape, torch.bfloat16)
    dk = Guarded(d["k"].shape, torch.bfloat16)
    dv = Guarded(d["v"].shape, torch.bfloat16)
    dsum = Guarded((B, Hq, Sq), torch.float32)
    gqa.gqa_bwd(d["q"], d["k"], d["v"], out, d["dout"], lse, causal=causal, seqlens_k=d["seqlens_k"], scale=0.1,
                dq=dq.t, dk=dk.t, dv=dv.t, dsum=dsum.t)
    assert gqa.gqa_device_status() == 0
    for g, what in ((dq, "dq"), (dk, "dk"), (dv, "dv"), (dsum, "dsum")):
        g.check(what)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("ns", [1, 3, 0])
def test_decode_writes_stay_inside_out_and_workspace(ns, dtype):
    B, Hq, Hkv, D, Smax = 5, 12, 2, 64, 333          # G = 6, ragged cache
    d = to_dev(inputs.make_decode(B, Hq, Hkv, D, Smax, seed=13, lens=(0, Smax), dtype=dtype))
    out = Guarded(d["q"].shape, d["q"].dtype)
    wsb = gqa.gqa_decode_workspace_bytes(B, Hq, Hkv, D, ns, Smax)
    work = Guarded((max(wsb, 16),), torch.uint8)
    gqa.gqa_decode(d["q"], d["kcache"], d["vcache"], d["cache_seqlens"], num_splits=ns, out=out.t, workspace=work.t)
    assert gqa.gqa_device_status() == 0
    out.check("out")
    work.check("workspace")


@pytest.mark.parametrize("ns", [1, 5, 0])
def test_fp8_decode_writes_stay_inside_out_and_workspace(ns):
    B, Hq, Hkv, D, Smax = 3, 16, 2, 128, 301
    d = to_dev(inputs.make_decode_fp8(B, Hq, Hkv, D, Smax, seed=17, lens=(0, Smax)))
    out = Guarded(d["q"].shape, d["q"].dtype)
    wsb = gqa.gqa_decode_fp8_workspace_bytes(B, Hq, Hkv, D, ns, Smax)
    work = Guarded((max(wsb, 16),), torch.uint8)
    gqa.gqa_decode_fp8(d["q"], d["kcache"], d["vcache"], d["cache_seqlens"], d["k_scale"], d["v_scale"],
                       num_splits=ns, out=out.t, workspace=work.t)
    assert gqa.gqa_device_status() == 0
    out.check("out")
    work.check("workspace")
