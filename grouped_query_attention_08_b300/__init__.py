"""grouped_query_attention_08_b300 -- Python binding of libgqa (B300 / sm_103a).

Thin ctypes layer over the C ABI declared in ``include/gqa.h``: it checks
shapes and dtypes, allocates outputs with torch (device memory and streams
are the only things torch is used for) and passes raw device pointers and the
current CUDA stream.  Every step of the attention runs in libgqa's kernels;
there is no CPU or PyTorch fallback -- if the library is missing the calls
raise.

Functions keep the C names:
  gqa_fwd(q, k, v, *, causal=False, seqlens_k=None, scale=None, out=None, lse=None, return_lse=True)
  gqa_fwd_host(q, k, v, *, causal=False, seqlens_k=None, scale=None, ..., staging=None, chunk_b=0)
  gqa_decode(q, kcache, vcache, cache_seqlens, *, scale=None, num_splits=0, out=None, workspace=None)
  gqa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, *, causal=False, ...)
  gqa_fwd_sparse(q, k, v, block_mask, block_size, *, causal=False, seqlens_k=None, ...)
  gqa_bwd(q, k, v, out, dout, lse, *, causal=False, seqlens_k=None, scale=None, dq=None, dk=None, dv=None)
  gqa_decode_fp8(q, kcache, vcache, cache_seqlens, *, k_scale, v_scale, ...)
  gqa_decode_num_splits(B, Hkv, max_seqlen_k, num_splits)
  gqa_decode_workspace_bytes(B, Hq, Hkv, D, num_splits, max_seqlen_k)
  gqa_decode_fp8_num_splits(B, Hkv, max_seqlen_k, num_splits)
  gqa_decode_fp8_workspace_bytes(B, Hq, Hkv, D, num_splits, max_seqlen_k)
  gqa_device_status(stream=None)
  gqa_status_string(status)
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

GQA_OK = 0
GQA_ERR_INVALID_ARG = 1
GQA_ERR_UNSUPPORTED = 2
GQA_ERR_CUDA = 3
GQA_ERR_DEVICE_TIMEOUT = 4
GQA_ERR_DEVICE_BOUNDS = 5
GQA_DTYPE_BF16 = 0
GQA_DTYPE_FP32 = 1
# size of gqa_decode_noalloc's library-owned scratch (GQA_DECODE_NOALLOC_SCRATCH_BYTES in gqa.h)
GQA_DECODE_NOALLOC_SCRATCH_BYTES = 32 << 20

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libgqa.so")
_lock = threading.Lock()
_lib = None


class GQAError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        super().__init__("%s%s" % (gqa_status_string(status), (": " + what) if what else ""))


def lib_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libgqa.so (built in-tree by ``build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("libgqa.so is not built (%s); run grouped_query_attention_08_b300.build.build()"
                               % _LIB_PATH)
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.gqa_fwd.restype = i32
        lib.gqa_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp, i32, vp]
        lib.gqa_fwd_host.restype = i32
        lib.gqa_fwd_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp, i32, vp, vp, vp,
                                     vp, vp, vp, i32, vp]
        lib.gqa_fwd_varlen.restype = i32
        lib.gqa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                       f32, i32, i32, vp]
        lib.gqa_decode_fp8.restype = i32
        lib.gqa_decode_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, f32, i32, i32, vp, sz,
                                       vp]
        lib.gqa_fwd_sparse.restype = i32
        lib.gqa_fwd_sparse.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32, vp,
                                       i32, vp]
        lib.gqa_bwd.restype = i32
        lib.gqa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32,
                                vp, i32, vp]
        lib.gqa_decode.restype = i32
        lib.gqa_decode.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, i32, i32, vp, sz, vp]
        lib.gqa_decode_num_splits.restype = i32
        lib.gqa_decode_num_splits.argtypes = [i32, i32, i32, i32]
        lib.gqa_decode_workspace_bytes.restype = sz
        lib.gqa_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.gqa_decode_fp8_num_splits.restype = i32
        lib.gqa_decode_fp8_num_splits.argtypes = [i32, i32, i32, i32]
        lib.gqa_decode_fp8_workspace_bytes.restype = sz
        lib.gqa_decode_fp8_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.gqa_device_status.restype = i32
        lib.gqa_device_status.argtypes = [vp]
        lib.gqa_status_string.restype = ctypes.c_char_p
        lib.gqa_status_string.argtypes = [i32]
        _lib = lib
        return lib


def gqa_status_string(status: int) -> str:
    try:
        return load_library().gqa_status_string(int(status)).decode()
    except RuntimeError:
        return "status %d" % int(status)


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return GQA_DTYPE_BF16
    if t.dtype == torch.float32:
        return GQA_DTYPE_FP32
    raise TypeError("q/k/v must be bfloat16 or float32, got %s" % t.dtype)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device, stream=None):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _expect(t, shape, dtype, name):
    """A caller-provided buffer must have exactly the shape and dtype the
    library writes (the C ABI sees only a pointer)."""
    if t is not None and (tuple(t.shape) != tuple(shape) or t.dtype != dtype):
        raise ValueError("%s must be %s %s, got %s %s" % (name, dtype, list(shape), t.dtype, list(t.shape)))


def _check_cuda(*ts):
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (libgqa has no CPU path)")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("all tensors must be on the same device")
    return dev


def _on(dev):
    """Makes the tensors' device current for a library call: libgqa reads the
    current device for its per-device state and the stream's device."""
    return _torch().cuda.device(dev)


def gqa_fwd(q, k, v, *, causal=False, seqlens_k=None, scale=None, out=None, lse=None,
            return_lse=True, stream=None):
    """Prefill / encoder GQA attention.  q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D] (bf16 or fp32, CUDA).

    Returns (out [B,Sq,Hq,D], lse [B,Hq,Sq] fp32 or None).  ``scale`` defaults to
    1/sqrt(D); ``seqlens_k`` is an int32 CUDA tensor [B] of key lengths.
    """
    torch = _torch()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, S, H, D]")
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch between q, k and v")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share a dtype")
    code = _dtype_code(q)
    if seqlens_k is not None and (seqlens_k.dtype != torch.int32 or tuple(seqlens_k.shape) != (B,)):
        raise ValueError("seqlens_k must be int32 [B]")
    _expect(out, q.shape, q.dtype, "out")
    _expect(lse, (B, Hq, Sq), torch.float32, "lse")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    dev = _check_cuda(q, k, v, out, lse, seqlens_k)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on(dev):
        rc = load_library().gqa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D,
                                    float(scale), int(bool(causal)), _ptr(seqlens_k), code,
                                    _stream(dev, stream))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_fwd")
    return out, lse


def gqa_fwd_host(q, k, v, *, causal=False, seqlens_k=None, scale=None, out=None, lse=None, return_lse=True,
                 staging=None, chunk_b=0, device=None, stream=None):
    """gqa_fwd for host-resident tensors: q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D] CPU tensors (bf16 or
    fp32; page-locked for the copies to overlap), optional int32 CPU seqlens_k [B].  The batch
    is cut into chunks whose copies in, attention and copies out overlap on three streams.

    Returns (out, lse) CPU tensors (allocated page-locked when not given).  The call only
    enqueues work: the outputs are complete once the stream has completed
    (torch.cuda.current_stream(device).synchronize()).  ``staging`` is an optional dict of
    device tensors ``q, k, v, out, lse, seqlens`` of the full sizes, reused across calls;
    missing ones are allocated on ``device`` (default: the current CUDA device).
    """
    torch = _torch()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, S, H, D]")
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch between q, k and v")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share a dtype")
    code = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("seqlens_k", seqlens_k), ("out", out), ("lse", lse)):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("%s must be a contiguous CPU tensor" % name)
    if seqlens_k is not None and (seqlens_k.dtype != torch.int32 or tuple(seqlens_k.shape) != (B,)):
        raise ValueError("seqlens_k must be int32 [B]")
    _expect(out, q.shape, q.dtype, "out")
    _expect(lse, (B, Hq, Sq), torch.float32, "lse")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32).pin_memory()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    st = {} if staging is None else staging
    need = {"q": (q.shape, q.dtype), "k": (k.shape, k.dtype), "v": (v.shape, v.dtype), "out": (q.shape, q.dtype)}
    if lse is not None:
        need["lse"] = ((B, Hq, Sq), torch.float32)
    if seqlens_k is not None:
        need["seqlens"] = ((B,), torch.int32)
    for name, (shape, dtype) in need.items():
        if st.get(name) is None:
            st[name] = torch.empty(tuple(shape), dtype=dtype, device=dev)
        _expect(st[name], shape, dtype, "staging[%r]" % name)
    _check_cuda(*[st[n] for n in need])
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on(dev):
        rc = load_library().gqa_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D,
                                         float(scale), int(bool(causal)), _ptr(seqlens_k), code, _ptr(st["q"]),
                                         _ptr(st["k"]), _ptr(st["v"]), _ptr(st["out"]), _ptr(st.get("lse")),
                                         _ptr(st.get("seqlens")), int(chunk_b), _stream(dev, stream))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_fwd_host")
    return out, lse


def gqa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, *, max_seqlen_q=None, max_seqlen_k=None,
                   causal=False, scale=None, out=None, lse=None, return_lse=True, stream=None):
    """GQA attention over sequences packed without padding.

    q [total_q,Hq,D], k/v [total_k,Hkv,D] (bf16 or fp32, CUDA); cu_seqlens_q/k int32
    CUDA tensors [B+1] of row offsets.  Returns (out [total_q,Hq,D], lse [Hq,total_q]
    fp32 or None).  ``max_seqlen_q/k`` bound the sequence lengths; when None they are
    read from the offsets (a device-to-host copy that synchronises the stream).
    """
    torch = _torch()
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be 3-D [total, H, D]")
    total_q, Hq, D = q.shape
    total_k, Hkv, Dk = k.shape
    if Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch between q, k and v")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share a dtype")
    code = _dtype_code(q)
    for name, cu in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if cu.dtype != torch.int32 or cu.dim() != 1 or cu.shape[0] < 2:
            raise ValueError("%s must be int32 [B+1]" % name)
    if cu_seqlens_k.shape != cu_seqlens_q.shape:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both be [B+1]")
    B = cu_seqlens_q.shape[0] - 1
    if max_seqlen_q is None:
        max_seqlen_q = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item())
    if max_seqlen_k is None:
        max_seqlen_k = int((cu_seqlens_k[1:] - cu_seqlens_k[:-1]).max().item())
    _expect(out, q.shape, q.dtype, "out")
    _expect(lse, (Hq, total_q), torch.float32, "lse")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    dev = _check_cuda(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on(dev):
        rc = load_library().gqa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
                                           _ptr(cu_seqlens_k), B, Hq, Hkv, max(int(max_seqlen_q), 1),
                                           max(int(max_seqlen_k), 1), total_q, total_k, D, float(scale),
                                           int(bool(causal)), code, _stream(dev, stream))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_fwd_varlen")
    return out, lse


def gqa_fwd_sparse(q, k, v, block_mask, block_size, *, causal=False, seqlens_k=None, scale=None, out=None,
                   lse=None, return_lse=True, stream=None):
    """Block-sparse GQA attention.  q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D] (bf16 or fp32, CUDA);
    block_mask uint8/bool CUDA tensor [ceil(Sq/bs), ceil(Sk/bs)] (nonzero = attend), shared
    by all batch entries and heads; block_size 64 or 128.  Returns (out, lse) as gqa_fwd.
    """
    torch = _torch()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, S, H, D]")
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch between q, k and v")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share a dtype")
    code = _dtype_code(q)
    bs = int(block_size)
    if block_mask.dtype == torch.bool:
        block_mask = block_mask.to(torch.uint8)
    if block_mask.dtype != torch.uint8 or tuple(block_mask.shape) != ((Sq + bs - 1) // bs, (Sk + bs - 1) // bs):
        raise ValueError("block_mask must be uint8 [ceil(Sq/bs), ceil(Sk/bs)]")
    if seqlens_k is not None and (seqlens_k.dtype != torch.int32 or tuple(seqlens_k.shape) != (B,)):
        raise ValueError("seqlens_k must be int32 [B]")
    _expect(out, q.shape, q.dtype, "out")
    _expect(lse, (B, Hq, Sq), torch.float32, "lse")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    dev = _check_cuda(q, k, v, out, lse, seqlens_k, block_mask)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on(dev):
        rc = load_library().gqa_fwd_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(block_mask), bs,
                                           B, Hq, Hkv, Sq, Sk, D, float(scale), int(bool(causal)), _ptr(seqlens_k),
                                           code, _stream(dev, stream))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_fwd_sparse")
    return out, lse


def gqa_bwd(q, k, v, out, dout, lse, *, causal=False, seqlens_k=None, scale=None, dq=None, dk=None, dv=None,
            dsum=None, stream=None):
    """Gradients of gqa_fwd.  q/out/dout [B,Sq,Hq,D], k/v [B,Sk,Hkv,D] bf16 CUDA; lse fp32
    [B,Hq,Sq] from the forward (same causal / seqlens_k / scale).  Returns (dq, dk, dv) bf16;
    ``dsum`` (fp32 [B,Hq,Sq] scratch) is allocated when not given.
    """
    torch = _torch()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, S, H, D]")
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch between q, k and v")
    if tuple(out.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("out and dout must have q's shape")
    if any(t.dtype != torch.bfloat16 for t in (q, k, v, out, dout)):
        raise TypeError("gqa_bwd takes bf16 q, k, v, out, dout")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Sq):
        raise ValueError("lse must be float32 [B, Hq, Sq]")
    if seqlens_k is not None and (seqlens_k.dtype != torch.int32 or tuple(seqlens_k.shape) != (B,)):
        raise ValueError("seqlens_k must be int32 [B]")
    _expect(dq, q.shape, torch.bfloat16, "dq")
    _expect(dk, k.shape, torch.bfloat16, "dk")
    _expect(dv, k.shape, torch.bfloat16, "dv")
    _expect(dsum, (B, Hq, Sq), torch.float32, "dsum")
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    if dsum is None:
        dsum = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    dev = _check_cuda(q, k, v, out, dout, lse, dsum, dq, dk, dv, seqlens_k)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on(dev):
        rc = load_library().gqa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dsum), _ptr(dq),
                                    _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Sk, D, float(scale), int(bool(causal)),
                                    _ptr(seqlens_k), GQA_DTYPE_BF16, _stream(dev, stream))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_bwd")
    return dq, dk, dv


def gqa_decode_num_splits(B, Hkv, max_seqlen_k, num_splits=0) -> int:
    n = load_library().gqa_decode_num_splits(int(B), int(Hkv), int(max_seqlen_k), int(num_splits))
    if n < 0:
        raise GQAError(-n, "gqa_decode_num_splits")
    return n


def gqa_decode_workspace_bytes(B, Hq, Hkv, D, num_splits, max_seqlen_k) -> int:
    return int(load_library().gqa_decode_workspace_bytes(int(B), int(Hq), int(Hkv), int(D),
                                                         int(num_splits), int(max_seqlen_k)))


def gqa_decode_fp8_num_splits(B, Hkv, max_seqlen_k, num_splits=0) -> int:
    n = load_library().gqa_decode_fp8_num_splits(int(B), int(Hkv), int(max_seqlen_k), int(num_splits))
    if n < 0:
        raise GQAError(-n, "gqa_decode_fp8_num_splits")
    return n


def gqa_decode_fp8_workspace_bytes(B, Hq, Hkv, D, num_splits, max_seqlen_k) -> int:
    return int(load_library().gqa_decode_fp8_workspace_bytes(int(B), int(Hq), int(Hkv), int(D),
                                                             int(num_splits), int(max_seqlen_k)))


def gqa_decode(q, kcache, vcache, cache_seqlens, *, scale=None, num_splits=0, out=None,
               workspace=None, stream=None):
    """Single-token decode.  q [B,Hq,D]; caches [B,Smax,Hkv,D]; cache_seqlens int32 [B].

    Returns out [B,Hq,D].  ``workspace`` (uint8 CUDA tensor) is allocated when not given.
    """
    torch = _torch()
    if q.dim() != 3 or kcache.dim() != 4 or vcache.dim() != 4:
        raise ValueError("q must be [B,Hq,D] and caches [B,Smax,Hkv,D]")
    B, Hq, D = q.shape
    Bk, Smax, Hkv, Dk = kcache.shape
    if Bk != B or Dk != D or tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("shape mismatch between q and the caches")
    if q.dtype != kcache.dtype or q.dtype != vcache.dtype:
        raise TypeError("q and the caches must share a dtype")
    code = _dtype_code(q)
    if cache_seqlens.dtype != torch.int32 or tuple(cache_seqlens.shape) != (B,):
        raise ValueError("cache_seqlens must be int32 [B]")
    _expect(out, q.shape, q.dtype, "out")
    if out is None:
        out = torch.empty_like(q)
    dev = _check_cuda(q, kcache, vcache, cache_seqlens, out)
    with _on(dev):      # the automatic split count depends on the device's SM count
        need = gqa_decode_workspace_bytes(B, Hq, Hkv, D, num_splits, Smax)
    if workspace is None and need > 0:
        workspace = torch.empty((need,), dtype=torch.uint8, device=q.device)
    dev = _check_cuda(q, kcache, vcache, cache_seqlens, out, workspace)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on(dev):
        rc = load_library().gqa_decode(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(cache_seqlens), _ptr(out),
                                       B, Hq, Hkv, D, float(scale), int(num_splits), Smax, code,
                                       _ptr(workspace), wbytes, _stream(dev, stream))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_decode")
    return out


def gqa_decode_fp8(q, kcache, vcache, cache_seqlens, k_scale, v_scale, *, scale=None, num_splits=0, out=None,
                   workspace=None, stream=None):
    """Single-token decode over an FP8 (e4m3) cache.  q [B,Hq,128] bf16; caches
    [B,Smax,Hkv,128] torch.float8_e4m3fn (or uint8 holding e4m3 bytes); the cached
    key is k_scale * kcache and the value v_scale * vcache.  Returns out [B,Hq,128] bf16.
    """
    torch = _torch()
    if q.dim() != 3 or kcache.dim() != 4 or vcache.dim() != 4:
        raise ValueError("q must be [B,Hq,D] and caches [B,Smax,Hkv,D]")
    B, Hq, D = q.shape
    Bk, Smax, Hkv, Dk = kcache.shape
    if Bk != B or Dk != D or tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("shape mismatch between q and the caches")
    if q.dtype != torch.bfloat16:
        raise TypeError("q must be bfloat16")
    f8 = getattr(torch, "float8_e4m3fn", None)
    for c in (kcache, vcache):
        if c.dtype not in (torch.uint8, f8):
            raise TypeError("the caches must be float8_e4m3fn (or uint8 e4m3 bytes)")
    if cache_seqlens.dtype != torch.int32 or tuple(cache_seqlens.shape) != (B,):
        raise ValueError("cache_seqlens must be int32 [B]")
    _expect(out, q.shape, q.dtype, "out")
    if out is None:
        out = torch.empty_like(q)
    dev = _check_cuda(q, kcache, vcache, cache_seqlens, out)
    with _on(dev):      # the automatic split count depends on the device's SM count
        need = gqa_decode_fp8_workspace_bytes(B, Hq, Hkv, D, num_splits, Smax)
    if workspace is None and need > 0:
        workspace = torch.empty((need,), dtype=torch.uint8, device=q.device)
    dev = _check_cuda(q, kcache, vcache, cache_seqlens, out, workspace)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on(dev):
        rc = load_library().gqa_decode_fp8(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(cache_seqlens), _ptr(out),
                                           B, Hq, Hkv, D, float(scale), float(k_scale), float(v_scale),
                                           int(num_splits), Smax, _ptr(workspace), wbytes, _stream(dev, stream))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_decode_fp8")
    return out


def gqa_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    torch = _torch()
    st = stream if stream is not None else torch.cuda.current_stream()
    return int(load_library().gqa_device_status(ctypes.c_void_p(st.cuda_stream)))


def gqa_decode_noalloc(q, kcache, vcache, cache_seqlens, *, scale=None, num_splits=0, out=None, stream=None):
    """gqa_decode without a workspace argument, for callers that cannot allocate
    device memory: the split partials go to the library's own fixed 32 MiB
    device scratch array (see include/gqa.h).  Calls on one device share that
    array, so calls that overlap on the GPU must be serialised by the caller.
    Only ``out`` is allocated here when it is not given."""
    torch = _torch()
    lib = load_library()
    fn = lib.gqa_decode_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.restype = i32
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, i32, i32, vp]
    if q.dim() != 3 or kcache.dim() != 4 or vcache.dim() != 4:
        raise ValueError("q must be [B,Hq,D] and caches [B,Smax,Hkv,D]")
    B, Hq, D = q.shape
    Bk, Smax, Hkv, Dk = kcache.shape
    if Bk != B or Dk != D or tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("shape mismatch between q and the caches")
    if q.dtype != kcache.dtype or q.dtype != vcache.dtype:
        raise TypeError("q and the caches must share a dtype")
    if cache_seqlens.dtype != torch.int32 or tuple(cache_seqlens.shape) != (B,):
        raise ValueError("cache_seqlens must be int32 [B]")
    code = _dtype_code(q)
    _expect(out, q.shape, q.dtype, "out")
    if out is None:
        out = torch.empty_like(q)
    dev = _check_cuda(q, kcache, vcache, cache_seqlens, out)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on(dev):
        rc = fn(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(cache_seqlens), _ptr(out), B, Hq, Hkv, D, float(scale),
                int(num_splits), Smax, code, _stream(dev, stream))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_decode_noalloc")
    return out
