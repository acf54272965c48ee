"""Host-side checks of the C ABI that need no GPU.

The library must load, export every function include/gqa.h declares, and
reject bad arguments before touching the device (argument validation runs
before any CUDA call, so fake device pointers are safe here).
"""
import ctypes
import os
import re

import pytest

import grouped_query_attention_08_b300 as gqa
from grouped_query_attention_08_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gqa.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "gqa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["gqa_fwd", "gqa_decode", "gqa_decode_workspace_bytes", "gqa_decode_num_splits",
              "gqa_device_status", "gqa_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert gqa.gqa_status_string(0) == "GQA_OK"
    assert gqa.gqa_status_string(1) == "GQA_ERR_INVALID_ARG"
    assert gqa.gqa_status_string(5) == "GQA_ERR_DEVICE_BOUNDS"
    assert gqa.gqa_status_string(99) == "GQA_ERR_UNKNOWN"


FAKE = 0x10000   # 16-byte aligned, never dereferenced: validation fails first


def _fwd(lib, B=1, Hq=4, Hkv=2, Sq=8, Sk=8, D=64, scale=0.125, causal=0, dtype=0, q=FAKE, k=FAKE,
         v=FAKE, out=FAKE, lse=None, seqlens=None):
    P = ctypes.c_void_p
    return lib.gqa_fwd(P(q), P(k), P(v), P(out), P(lse) if lse else None, B, Hq, Hkv, Sq, Sk, D, scale,
                       causal, P(seqlens) if seqlens else None, dtype, None)


def test_fwd_rejects_indivisible_heads(lib):
    assert _fwd(lib, Hq=6, Hkv=4) == gqa.GQA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(B=0), dict(Sq=0), dict(Sk=-1), dict(D=0), dict(Hkv=0),
                                dict(q=0), dict(out=0), dict(scale=float("nan")),
                                dict(scale=float("inf")), dict(causal=2), dict(dtype=7),
                                dict(q=FAKE + 8), dict(lse=FAKE + 2), dict(seqlens=FAKE + 1)])
def test_fwd_rejects_invalid_arguments(lib, kw):
    assert _fwd(lib, **kw) == gqa.GQA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(D=96), dict(D=32), dict(D=256), dict(Hq=129, Hkv=1)])
def test_fwd_bf16_unsupported_shapes(lib, kw):
    assert _fwd(lib, **kw) == gqa.GQA_ERR_UNSUPPORTED


def test_fwd_fp32_head_dim_limit(lib):
    assert _fwd(lib, D=257, dtype=1) == gqa.GQA_ERR_UNSUPPORTED


def _fwd_host(lib, B=2, Hq=4, Hkv=2, Sq=8, Sk=8, D=64, scale=0.125, causal=0, dtype=0, qh=FAKE, oh=FAKE,
              lse_h=None, lse_d=None, sl_h=None, sl_d=None, qd=FAKE, chunk_b=0):
    P = ctypes.c_void_p
    opt = lambda x: P(x) if x else None  # noqa: E731
    return lib.gqa_fwd_host(P(qh), P(FAKE), P(FAKE), P(oh), opt(lse_h), B, Hq, Hkv, Sq, Sk, D, scale, causal,
                            opt(sl_h), dtype, P(qd), P(FAKE), P(FAKE), P(FAKE), opt(lse_d), opt(sl_d), chunk_b, None)


@pytest.mark.parametrize("kw", [dict(B=0), dict(Hq=6, Hkv=4), dict(qh=0), dict(oh=0), dict(qd=0),
                                dict(lse_h=FAKE), dict(lse_d=FAKE), dict(sl_h=FAKE), dict(sl_d=FAKE),
                                dict(qd=FAKE + 8), dict(scale=float("nan")), dict(causal=3), dict(dtype=5)])
def test_fwd_host_rejects_invalid_arguments_before_any_copy(lib, kw):
    # every rejection happens before a copy is enqueued (fake pointers are never touched)
    assert _fwd_host(lib, **kw) == gqa.GQA_ERR_INVALID_ARG


def test_fwd_host_unsupported_head_dim(lib):
    assert _fwd_host(lib, D=96) == gqa.GQA_ERR_UNSUPPORTED


def test_fwd_host_binding_refuses_device_tensors():
    import torch
    q = torch.zeros((1, 4, 4, 64), dtype=torch.bfloat16)
    k = torch.zeros((1, 4, 2, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gqa.gqa_fwd_host(q, k, k.clone(), seqlens_k=torch.zeros((2,), dtype=torch.int32))
    with pytest.raises(ValueError):
        gqa.gqa_fwd_host(q, k[:, :, :1], k)


def _fwd_varlen(lib, B=2, Hq=4, Hkv=2, msq=8, msk=8, tq=12, tk=12, D=64, scale=0.125, causal=0, dtype=0,
                q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=None, cuq=FAKE, cuk=FAKE):
    P = ctypes.c_void_p
    return lib.gqa_fwd_varlen(P(q), P(k), P(v), P(out), P(lse) if lse else None, P(cuq) if cuq else None,
                              P(cuk) if cuk else None, B, Hq, Hkv, msq, msk, tq, tk, D, scale, causal, dtype,
                              None)


@pytest.mark.parametrize("kw", [dict(B=0), dict(msq=0), dict(msk=0), dict(tq=0), dict(tk=-1), dict(D=0),
                                dict(Hq=6, Hkv=4), dict(cuq=0), dict(cuk=0), dict(cuq=FAKE + 2),
                                dict(q=0), dict(out=0), dict(scale=float("nan")), dict(causal=2),
                                dict(dtype=7), dict(k=FAKE + 8), dict(lse=FAKE + 1)])
def test_fwd_varlen_rejects_invalid_arguments(lib, kw):
    assert _fwd_varlen(lib, **kw) == gqa.GQA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(D=96), dict(Hq=129, Hkv=1), dict(D=300, dtype=1)])
def test_fwd_varlen_unsupported_shapes(lib, kw):
    assert _fwd_varlen(lib, **kw) == gqa.GQA_ERR_UNSUPPORTED


def _dec(lib, B=2, Hq=8, Hkv=2, D=128, scale=0.1, ns=1, smax=64, dtype=0, ws=None, wsb=0, q=FAKE,
         lens=FAKE):
    P = ctypes.c_void_p
    return lib.gqa_decode(P(q), P(FAKE), P(FAKE), P(lens) if lens else None, P(FAKE), B, Hq, Hkv, D,
                          scale, ns, smax, dtype, P(ws) if ws else None, wsb, None)


def test_decode_validation(lib):
    assert _dec(lib, Hq=6, Hkv=4) == gqa.GQA_ERR_INVALID_ARG
    assert _dec(lib, lens=0) == gqa.GQA_ERR_INVALID_ARG
    assert _dec(lib, smax=0) == gqa.GQA_ERR_INVALID_ARG
    assert _dec(lib, ns=129) == gqa.GQA_ERR_INVALID_ARG
    assert _dec(lib, D=96) == gqa.GQA_ERR_UNSUPPORTED
    assert _dec(lib, Hq=32, Hkv=2) == gqa.GQA_ERR_UNSUPPORTED          # G = 16 > 8 on bf16
    # two splits need a workspace
    assert _dec(lib, ns=2) == gqa.GQA_ERR_INVALID_ARG
    need = lib.gqa_decode_workspace_bytes(2, 8, 2, 128, 2, 64)
    assert need > 0
    assert _dec(lib, ns=2, ws=FAKE, wsb=need - 1) == gqa.GQA_ERR_INVALID_ARG
    assert _dec(lib, ns=2, ws=FAKE + 4, wsb=need) == gqa.GQA_ERR_INVALID_ARG


def test_split_planning(lib):
    # explicit counts: split length = ceil(Smax / n) rounded up to 16 keys
    assert gqa.gqa_decode_num_splits(4, 8, 8192, 1) == 1
    assert gqa.gqa_decode_num_splits(4, 8, 8192, 8) == 8
    assert gqa.gqa_decode_num_splits(4, 8, 100, 3) == 3          # ceil(100/3)=34 -> 48 -> 3 splits
    assert gqa.gqa_decode_num_splits(4, 8, 100, 7) == 7          # 15 -> 16 -> 7 splits
    assert gqa.gqa_decode_num_splits(4, 8, 40, 100) == 3         # at most one split per 16 keys
    n = gqa.gqa_decode_num_splits(64, 8, 8192, 0)
    assert 1 <= n <= 128
    assert gqa.gqa_decode_workspace_bytes(64, 64, 8, 128, 1, 8192) == 0
    ws = gqa.gqa_decode_workspace_bytes(64, 64, 8, 128, 8, 8192)
    assert ws >= 64 * 64 * 8 * 129 * 4


def test_fp8_split_planning(lib):
    # explicit counts plan exactly as the bf16 decode's
    for args in ((4, 8, 8192, 1), (4, 8, 8192, 8), (4, 8, 100, 3), (4, 8, 100, 7), (4, 8, 40, 100)):
        assert gqa.gqa_decode_fp8_num_splits(*args) == gqa.gqa_decode_num_splits(*args)
        B, Hkv, smax, ns = args
        assert (gqa.gqa_decode_fp8_workspace_bytes(B, 4 * Hkv, Hkv, 128, ns, smax)
                == gqa.gqa_decode_workspace_bytes(B, 4 * Hkv, Hkv, 128, ns, smax))
    # automatic: about 512 keys per split (148 SMs when no GPU is present)
    n8 = gqa.gqa_decode_fp8_num_splits(64, 8, 8192, 0)
    assert n8 == 16 and gqa.gqa_decode_num_splits(64, 8, 8192, 0) == 8
    assert gqa.gqa_decode_fp8_workspace_bytes(64, 64, 8, 128, 0, 8192) >= 64 * 64 * 16 * 129 * 4
    with pytest.raises(gqa.GQAError):
        gqa.gqa_decode_fp8_num_splits(64, 8, 8192, 129)
    assert gqa.gqa_decode_fp8_workspace_bytes(0, 64, 8, 128, 0, 8192) == 0


def _dec8(lib, B=2, Hq=8, Hkv=2, D=128, scale=0.1, ks=0.01, vs=0.02, ns=1, smax=64, ws=None, wsb=0, q=FAKE,
          kc=FAKE, lens=FAKE):
    P = ctypes.c_void_p
    return lib.gqa_decode_fp8(P(q), P(kc), P(FAKE), P(lens) if lens else None, P(FAKE), B, Hq, Hkv, D, scale,
                              ks, vs, ns, smax, P(ws) if ws else None, wsb, None)


def test_decode_fp8_validation(lib):
    assert _dec8(lib, Hq=6, Hkv=4) == gqa.GQA_ERR_INVALID_ARG
    assert _dec8(lib, lens=0) == gqa.GQA_ERR_INVALID_ARG
    assert _dec8(lib, kc=FAKE + 8) == gqa.GQA_ERR_INVALID_ARG          # caches 16-byte aligned
    assert _dec8(lib, ks=float("inf")) == gqa.GQA_ERR_INVALID_ARG
    assert _dec8(lib, vs=float("nan")) == gqa.GQA_ERR_INVALID_ARG
    assert _dec8(lib, ns=129) == gqa.GQA_ERR_INVALID_ARG
    assert _dec8(lib, D=64) == gqa.GQA_ERR_UNSUPPORTED                 # head dimension 128 only
    assert _dec8(lib, Hq=32, Hkv=2) == gqa.GQA_ERR_UNSUPPORTED         # G = 16 > 8
    assert _dec8(lib, ns=2) == gqa.GQA_ERR_INVALID_ARG                 # two splits need a workspace


def _sparse(lib, B=1, Hq=4, Hkv=2, Sq=8, Sk=8, D=64, bs=64, scale=0.125, causal=0, dtype=0, q=FAKE, bm=FAKE):
    P = ctypes.c_void_p
    return lib.gqa_fwd_sparse(P(q), P(FAKE), P(FAKE), P(FAKE), None, P(bm) if bm else None, bs, B, Hq, Hkv, Sq,
                              Sk, D, scale, causal, None, dtype, None)


@pytest.mark.parametrize("kw", [dict(bm=0), dict(bs=32), dict(bs=100), dict(Hq=6, Hkv=4), dict(B=0),
                                dict(scale=float("nan")), dict(causal=3), dict(q=FAKE + 8)])
def test_fwd_sparse_rejects_invalid_arguments(lib, kw):
    assert _sparse(lib, **kw) == gqa.GQA_ERR_INVALID_ARG


def test_fwd_sparse_unsupported_shapes(lib):
    assert _sparse(lib, Sk=8193) == gqa.GQA_ERR_UNSUPPORTED      # more than 64 key tiles of 128
    assert _sparse(lib, D=96) == gqa.GQA_ERR_UNSUPPORTED


def _bwd(lib, B=1, Hq=4, Hkv=2, Sq=8, Sk=8, D=64, scale=0.125, causal=0, dtype=0, q=FAKE, lse=FAKE, dsum=FAKE,
         dk=FAKE):
    P = ctypes.c_void_p
    return lib.gqa_bwd(P(q), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(lse) if lse else None, P(dsum) if dsum else None,
                       P(FAKE), P(dk), P(FAKE), B, Hq, Hkv, Sq, Sk, D, scale, causal, None, dtype, None)


@pytest.mark.parametrize("kw", [dict(lse=0), dict(dsum=0), dict(Hq=6, Hkv=4), dict(B=0), dict(Sk=0),
                                dict(scale=float("inf")), dict(causal=2), dict(q=FAKE + 8), dict(dk=FAKE + 2),
                                dict(lse=FAKE + 2), dict(dtype=7)])
def test_bwd_rejects_invalid_arguments(lib, kw):
    assert _bwd(lib, **kw) == gqa.GQA_ERR_INVALID_ARG


def test_bwd_unsupported(lib):
    assert _bwd(lib, dtype=gqa.GQA_DTYPE_FP32) == gqa.GQA_ERR_UNSUPPORTED   # bf16 only
    assert _bwd(lib, D=96) == gqa.GQA_ERR_UNSUPPORTED
    assert _bwd(lib, B=70000) == gqa.GQA_ERR_UNSUPPORTED                   # grid z limit


@pytest.mark.parametrize("causal,lens", [(False, None), (True, None), (False, [3, 0, 7]), (True, [5, 2, 7])])
def test_backward_flops_counts_admissible_pairs(causal, lens):
    # 10 * D flops per admissible (b, h, i, j), counted here by brute force
    from grouped_query_attention_08_b300 import roofline
    B, Hq, Sq, Sk, D = 3, 4, 5, 7, 16
    pairs = 0
    for b in range(B):
        L = Sk if lens is None else lens[b]
        for i in range(Sq):
            for j in range(Sk):
                if j < L and (not causal or j <= i + Sk - Sq):
                    pairs += Hq
    assert roofline.backward_flops(B, Hq, Sq, Sk, D, causal, lens) == 10 * D * pairs


def test_bwd_rejects_groups_wider_than_a_tile(lib):
    assert _bwd(lib, Hq=130, Hkv=1) == gqa.GQA_ERR_UNSUPPORTED    # 128 rows hold one token of each head


def test_product_code_does_not_touch_the_oracle():
    # the oracle is test infrastructure: nothing in the package (binding,
    # build script, inputs, roofline, CUDA sources) imports, loads or names it
    import pathlib
    pkg = pathlib.Path(gqa.__file__).parent
    files = [p for p in pkg.rglob("*") if p.suffix in (".py", ".cu", ".cuh", ".h", ".c")]
    assert files
    for p in files:
        text = p.read_text()
        assert "import oracle" not in text and "from oracle" not in text, p
        assert "liboracle" not in text and "oracle/" not in text, p
