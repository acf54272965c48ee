"""gqa_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (for example an operator interface that only hands
over input and output buffers, or a decode loop that must never call
cudaMalloc).  Its split partials live in the library's fixed 32 MiB device
scratch array instead of a caller workspace.

This file is collected last on purpose: the GPU test checks the entry point
through the C ABI against gqa_decode on two calls in a row, and it must pass
both alone in a fresh process and after every other test.
"""
import ctypes

import pytest
import torch

import grouped_query_attention_08_b300 as gqa
from grouped_query_attention_08_b300 import build, inputs

SCRATCH = gqa.GQA_DECODE_NOALLOC_SCRATCH_BYTES


def _lib():
    build.build()
    lib = gqa.load_library()
    fn = lib.gqa_decode_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.restype = i32
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, i32, i32, vp]
    return lib


def _call(lib, d, out, scale, ns, dtype):
    B, Hq, D = d["q"].shape
    _, Smax, Hkv, _ = d["kcache"].shape
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.gqa_decode_noalloc(P(d["q"]), P(d["kcache"]), P(d["vcache"]), P(d["cache_seqlens"]), P(out),
                                  B, Hq, Hkv, D, scale, ns, Smax, dtype, st)


def test_rejects_calls_beyond_the_scratch_size():
    lib = _lib()
    # B=512, Hq=64, D=128 with 8 splits needs > 32 MiB of partials
    need = lib.gqa_decode_workspace_bytes(512, 64, 8, 128, 8, 8192)
    assert need > SCRATCH
    fake = ctypes.c_void_p(0x10000)
    rc = lib.gqa_decode_noalloc(fake, fake, fake, fake, fake, 512, 64, 8, 128, 0.1, 8, 8192, 0, None)
    assert rc == gqa.GQA_ERR_UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_noalloc_decode_matches_gqa_decode_on_two_calls_in_a_row(dtype):
    lib = _lib()
    code = gqa.GQA_DTYPE_BF16 if dtype == "bf16" else gqa.GQA_DTYPE_FP32
    for call, seed in enumerate((21, 22)):       # different inputs: stale scratch contents cannot pass
        inp = inputs.make_decode(16, 64, 8, 128, 4096, seed=seed, lens=(1, 4096), dtype=dtype)
        d = {k: v.cuda() for k, v in inp.items()}
        ns = 8
        assert 0 < lib.gqa_decode_workspace_bytes(16, 64, 8, 128, ns, 4096) <= SCRATCH
        ref = gqa.gqa_decode(d["q"], d["kcache"], d["vcache"], d["cache_seqlens"], scale=0.088, num_splits=ns)
        out = torch.full_like(d["q"], float("nan"))
        rc = _call(lib, d, out, 0.088, ns, code)
        assert rc == gqa.GQA_OK, gqa.gqa_status_string(rc)
        torch.cuda.synchronize()
        assert gqa.gqa_device_status() == 0
        # the same kernels on the same inputs, so the outputs agree bit for bit
        # (a scratch corrupted by an earlier call cannot hide inside a tolerance)
        assert torch.equal(out, ref), "noalloc call %d differs from gqa_decode" % call
