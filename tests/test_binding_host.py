"""The Python binding's argument checks, on CPU tensors (no GPU needed).

The C ABI receives bare pointers, so a caller-provided output buffer of the
wrong shape or dtype would be written out of bounds; the binding must refuse
it before any pointer reaches the library.  Each case below fails on the
buffer check itself (matched by its message), ahead of the check that every
tensor is on a CUDA device.
"""
import pytest
import torch

import grouped_query_attention_08_b300 as gqa

bf = torch.bfloat16


def _qkv(B=2, Sq=5, Sk=7, Hq=4, Hkv=2, D=64, dtype=bf):
    return (torch.zeros(B, Sq, Hq, D, dtype=dtype), torch.zeros(B, Sk, Hkv, D, dtype=dtype),
            torch.zeros(B, Sk, Hkv, D, dtype=dtype))


@pytest.mark.parametrize("kw,msg", [
    (dict(out=torch.zeros(2, 5, 4, 32, dtype=bf)), "out must be"),
    (dict(out=torch.zeros(2, 5, 4, 64, dtype=torch.float32)), "out must be"),
    (dict(lse=torch.zeros(2, 5, 4)), "lse must be"),
    (dict(lse=torch.zeros(2, 4, 5, dtype=torch.float64)), "lse must be"),
])
def test_fwd_refuses_wrong_output_buffers(kw, msg):
    q, k, v = _qkv()
    with pytest.raises(ValueError, match=msg):
        gqa.gqa_fwd(q, k, v, **kw)


def test_fwd_sparse_refuses_wrong_output_buffers():
    q, k, v = _qkv()
    bm = torch.ones(1, 1, dtype=torch.uint8)
    with pytest.raises(ValueError, match="out must be"):
        gqa.gqa_fwd_sparse(q, k, v, bm, 64, out=torch.zeros(2, 5, 4, 65, dtype=bf))
    with pytest.raises(ValueError, match="lse must be"):
        gqa.gqa_fwd_sparse(q, k, v, bm, 64, lse=torch.zeros(2, 4, 6))


def test_fwd_varlen_refuses_wrong_output_buffers():
    q, k, v = torch.zeros(9, 4, 64, dtype=bf), torch.zeros(11, 2, 64, dtype=bf), torch.zeros(11, 2, 64, dtype=bf)
    cu_q = torch.tensor([0, 4, 9], dtype=torch.int32)
    cu_k = torch.tensor([0, 5, 11], dtype=torch.int32)
    with pytest.raises(ValueError, match="out must be"):
        gqa.gqa_fwd_varlen(q, k, v, cu_q, cu_k, out=torch.zeros(8, 4, 64, dtype=bf))
    with pytest.raises(ValueError, match="lse must be"):
        gqa.gqa_fwd_varlen(q, k, v, cu_q, cu_k, lse=torch.zeros(9, 4))


def test_decode_entry_points_refuse_wrong_out():
    q = torch.zeros(2, 8, 128, dtype=bf)
    kc = torch.zeros(2, 16, 2, 128, dtype=bf)
    lens = torch.tensor([3, 16], dtype=torch.int32)
    bad = torch.zeros(2, 8, 64, dtype=bf)
    with pytest.raises(ValueError, match="out must be"):
        gqa.gqa_decode(q, kc, kc, lens, out=bad)
    with pytest.raises(ValueError, match="out must be"):
        gqa.gqa_decode_noalloc(q, kc, kc, lens, out=bad)
    k8 = torch.zeros(2, 16, 2, 128, dtype=torch.uint8)
    with pytest.raises(ValueError, match="out must be"):
        gqa.gqa_decode_fp8(q, k8, k8, lens, 1.0, 1.0, out=bad)


def test_decode_noalloc_checks_its_inputs():
    q = torch.zeros(2, 8, 128, dtype=bf)
    with pytest.raises(ValueError, match="shape mismatch"):
        gqa.gqa_decode_noalloc(q, torch.zeros(3, 16, 2, 128, dtype=bf), torch.zeros(3, 16, 2, 128, dtype=bf),
                               torch.tensor([1, 2], dtype=torch.int32))
    with pytest.raises(ValueError, match="cache_seqlens"):
        gqa.gqa_decode_noalloc(q, torch.zeros(2, 16, 2, 128, dtype=bf), torch.zeros(2, 16, 2, 128, dtype=bf),
                               torch.tensor([1, 2, 3], dtype=torch.int32))


@pytest.mark.parametrize("name,shape,dtype", [
    ("dq", (2, 5, 4, 32), bf), ("dk", (2, 7, 4, 64), bf), ("dv", (2, 7, 2, 64), torch.float32),
    ("dsum", (2, 5, 4), torch.float32),
])
def test_bwd_refuses_wrong_gradient_buffers(name, shape, dtype):
    q, k, v = _qkv()
    lse = torch.zeros(2, 4, 5)
    with pytest.raises(ValueError, match="%s must be" % name):
        gqa.gqa_bwd(q, k, v, q, q, lse, **{name: torch.zeros(shape, dtype=dtype)})


def test_correct_buffers_pass_the_checks_and_stop_at_the_device_check():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="CUDA"):
        gqa.gqa_fwd(q, k, v, out=torch.zeros_like(q), lse=torch.zeros(2, 4, 5))
    with pytest.raises(ValueError, match="CUDA"):
        gqa.gqa_bwd(q, k, v, q, q, torch.zeros(2, 4, 5), dq=torch.zeros_like(q), dk=torch.zeros_like(k),
                    dv=torch.zeros_like(v), dsum=torch.zeros(2, 4, 5))
