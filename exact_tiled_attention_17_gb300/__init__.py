"""Exact tiled attention forward for one NVIDIA GB300 (sm_103a).

A thin Python binding over the C ABI of ``libattn.so`` (declared in
``include/attn.h``): the functions here only check and marshal arguments;
every step of the computation runs in the library's CUDA kernels.  PyTorch
provides device memory and streams.  If the library has not been built the
import fails loudly; there is no CPU or PyTorch fallback.

    attn_fwd(q, k, v, causal=False, scale=None, Br=0, Bc=0, key_mask=None)
        -> (o, lse)          tiled exact forward (bf16 on tcgen05, or fp32 SIMT)
    attn_naive_fwd(...)      materialising baseline (S and P in the input dtype)
    attn_deviation(a, b)     max-abs, Wasserstein-1 (via sort), mean/std |a-b|
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")

ATTN_F32, ATTN_BF16, ATTN_F64 = 0, 1, 2
ATTN_OK = 0
ATTN_ERR_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_WORKSPACE = -3
ATTN_ERR_CUDA = -4
ATTN_ERR_DEVICE_TIMEOUT = -5

# Every symbol include/attn.h declares.
EXPORTS = ("attn_fwd", "attn_fwd_host_workspace_size", "attn_fwd_host", "attn_fwd_block_sparse", "attn_naive_workspace_size", "attn_naive_fwd", "attn_deviation_workspace_size",
           "attn_deviation", "attn_deviation_noalloc", "attn_decode_workspace_size", "attn_decode_fwd",
           "attn_bwd_workspace_size", "attn_bwd", "attn_emul_fwd", "attn_emul_round", "attn_status",
           "attn_strerror", "attn_last_variant", "attn_debug_wait_timeout")
DEVIATION_NOALLOC_MAX_N = 1 << 20

_DTYPE = {torch.float32: ATTN_F32, torch.bfloat16: ATTN_BF16, torch.float64: ATTN_F64}


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {strerror(status)} ({status})")
        self.status = status


class DevT(ctypes.Structure):
    _fields_ = [("max_abs", ctypes.c_double), ("w1", ctypes.c_double), ("mean_abs", ctypes.c_double),
                ("std_abs", ctypes.c_double), ("mean_signed", ctypes.c_double), ("n", ctypes.c_longlong)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
                          "(the CUDA library is required; there is no fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_longlong
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, i, vp, vp]
    lib.attn_fwd_block_sparse.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, vp]
    lib.attn_fwd_block_sparse.restype = i
    lib.attn_fwd.restype = i
    lib.attn_fwd_host_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.attn_fwd_host_workspace_size.restype = sz
    lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, i, vp, vp, sz, vp]
    lib.attn_fwd_host.restype = i
    lib.attn_naive_workspace_size.argtypes = [i, i, i, i]
    lib.attn_naive_workspace_size.restype = sz
    lib.attn_naive_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, sz, vp]
    lib.attn_naive_fwd.restype = i
    lib.attn_deviation_workspace_size.argtypes = [ll]
    lib.attn_deviation_workspace_size.restype = sz
    lib.attn_deviation.argtypes = [vp, i, vp, i, ll, vp, sz, vp, ctypes.POINTER(DevT)]
    lib.attn_deviation.restype = i
    lib.attn_deviation_noalloc.argtypes = [vp, i, vp, i, ll, vp, ctypes.POINTER(DevT)]
    lib.attn_deviation_noalloc.restype = i
    lib.attn_decode_workspace_size.argtypes = [i, i, i, i]
    lib.attn_decode_workspace_size.restype = sz
    lib.attn_decode_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, vp, sz, vp]
    lib.attn_decode_fwd.restype = i
    lib.attn_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.attn_bwd_workspace_size.restype = sz
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, sz, vp]
    lib.attn_bwd.restype = i
    lib.attn_emul_fwd.argtypes = [vp, vp, vp, i, vp, i, i, i, i, i, f, vp, i, i, i, i, vp, ll, vp]
    lib.attn_emul_fwd.restype = i
    lib.attn_emul_round.argtypes = [vp, vp, ll, i, i, vp]
    lib.attn_emul_round.restype = i
    lib.attn_status.argtypes = [vp]
    lib.attn_status.restype = i
    lib.attn_strerror.argtypes = [i]
    lib.attn_strerror.restype = ctypes.c_char_p
    lib.attn_last_variant.argtypes = [ctypes.c_char_p, i]
    lib.attn_last_variant.restype = i
    lib.attn_debug_wait_timeout.argtypes = [ctypes.c_uint, vp]
    lib.attn_debug_wait_timeout.restype = i
    return lib


lib = _load()


def strerror(status: int) -> str:
    return lib.attn_strerror(int(status)).decode()


def _check(rc: int, what: str) -> None:
    if rc != ATTN_OK:
        raise AttnError(rc, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _shape4(q):
    if q.dim() == 4:
        return q.shape
    if q.dim() == 3:
        return (1,) + tuple(q.shape)
    raise ValueError("q, k, v must be [B, H, N, d] or [H, N, d]")


BLOCK_SPARSE_BLOCK = 128
BLOCK_SPARSE_MAX_N = 131072


def attn_fwd_block_sparse(q, k, v, block_mask, causal: bool = False, scale: float | None = None, key_mask=None,
                          out=None, lse=None, stream=None, want_lse: bool = True):
    """Forward restricted to the marked 128 x 128 blocks.  block_mask: [B, H,
    nb, nb] uint8 (or bool) device tensor, nb = ceil(N / 128), non-zero = the
    block takes part.  Returns (o, lse)."""
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous device tensors")
    if not (q.shape == k.shape == v.shape and q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share shape and dtype")
    B, H, N, d = _shape4(q)
    nb = -(-N // BLOCK_SPARSE_BLOCK)
    if block_mask.dtype == torch.bool:
        block_mask = block_mask.to(torch.uint8)
    if (block_mask.dtype != torch.uint8 or not block_mask.is_cuda or not block_mask.is_contiguous()
            or block_mask.numel() != B * H * nb * nb):
        raise ValueError("block_mask must be a contiguous uint8 device tensor with B*H*nb*nb elements")
    if q.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {q.dtype}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = out if out is not None else torch.empty_like(q)
    l = lse if lse is not None else (torch.empty((B, H, N), dtype=torch.float32, device=q.device)
                                     if want_lse else None)
    m = None
    if key_mask is not None:
        m = key_mask
        if m.dtype != torch.float32 or not m.is_contiguous() or m.numel() != B * H * N or not m.is_cuda:
            raise ValueError("key_mask must be a contiguous float32 device tensor with B*H*N elements")
    rc = lib.attn_fwd_block_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, N, d, int(bool(causal)),
                                   float(scale), _DTYPE[q.dtype], _ptr(block_mask), _ptr(m),
                                   ctypes.c_void_p(_stream(stream)))
    _check(rc, "attn_fwd_block_sparse")
    return o, l


def attn_fwd_host_workspace_size(B: int, H: int, N: int, d: int, dtype, with_mask: bool = False) -> int:
    return int(lib.attn_fwd_host_workspace_size(B, H, N, d, _DTYPE[dtype] if not isinstance(dtype, int) else dtype,
                                                int(bool(with_mask))))


def _attn_fwd_host(q, k, v, causal, scale, Br, Bc, key_mask, out, lse, stream, want_lse, sync, workspace):
    """attn_fwd on host tensors through the C ABI's attn_fwd_host: the library
    copies the inputs into a device workspace, runs the forward and copies O
    and LSE back, all on `stream`."""
    for t in (q, k, v):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous host tensors")
    if not (q.shape == k.shape == v.shape and q.dtype == k.dtype == v.dtype) or q.dtype not in _DTYPE:
        raise ValueError("q, k, v must share shape and a supported dtype")
    B, H, N, d = _shape4(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = stream if stream is not None else torch.cuda.current_stream()
    if not isinstance(st, torch.cuda.Stream):
        st = torch.cuda.ExternalStream(int(st))
    m = None
    if key_mask is not None:
        m = key_mask
        if m.device.type != "cpu" or m.dtype != torch.float32 or not m.is_contiguous() or m.numel() != B * H * N:
            raise ValueError("key_mask must be a contiguous float32 host tensor with B*H*N elements")
    need = attn_fwd_host_workspace_size(B, H, N, d, q.dtype, m is not None)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=torch.device("cuda", torch.cuda.current_device()))
        workspace.record_stream(st)
    ho = out if out is not None else torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    hl = lse if lse is not None else (torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
                                      if want_lse else None)
    for t in (ho,) + ((hl,) if hl is not None else ()):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError("out / lse must be contiguous host tensors")
    rc = lib.attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(ho), _ptr(hl), B, H, N, d, int(bool(causal)), float(scale),
                           int(Br), int(Bc), _DTYPE[q.dtype], _ptr(m), _ptr(workspace), workspace.numel(),
                           ctypes.c_void_p(st.cuda_stream))
    _check(rc, "attn_fwd_host")
    if sync:
        st.synchronize()
    return ho, hl


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, Br: int = 0, Bc: int = 0,
             key_mask=None, out=None, lse=None, stream=None, want_lse: bool = True, sync: bool = True,
             workspace=None):
    """Tiled exact attention forward.  Returns (o, lse).

    Device tensors: the call is enqueued on `stream` (default: torch's current
    stream) and returns immediately.  Host tensors (pinned or not): the C ABI's
    attn_fwd_host copies the inputs into a device workspace (``workspace``, a
    uint8 device tensor of attn_fwd_host_workspace_size bytes, allocated here
    if not given), runs the kernel and copies o / lse back into host tensors,
    all on `stream`; with sync=False the call returns once that work is
    enqueued (o / lse are valid after the stream is synchronised), so calls on
    two streams overlap one's copies with the other's kernel.
    """
    if q.device.type == "cpu":
        return _attn_fwd_host(q, k, v, causal, scale, Br, Bc, key_mask, out, lse, stream, want_lse, sync, workspace)
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous tensors on one device")
    if not (q.shape == k.shape == v.shape and q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share shape and dtype")
    B, H, N, d = _shape4(q)
    if q.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {q.dtype}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = out if out is not None else torch.empty_like(q)
    l = lse if lse is not None else (torch.empty((B, H, N), dtype=torch.float32, device=q.device)
                                     if want_lse else None)
    m = None
    if key_mask is not None:
        m = key_mask
        if m.dtype != torch.float32 or not m.is_contiguous() or m.numel() != B * H * N or not m.is_cuda:
            raise ValueError("key_mask must be a contiguous float32 device tensor with B*H*N elements")
    rc = lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, N, d, int(bool(causal)),
                      float(scale), int(Br), int(Bc), _DTYPE[q.dtype], _ptr(m), ctypes.c_void_p(_stream(stream)))
    _check(rc, "attn_fwd")
    return o, l


def attn_naive_workspace_size(B: int, H: int, N: int, dtype) -> int:
    return int(lib.attn_naive_workspace_size(B, H, N, _DTYPE[dtype] if not isinstance(dtype, int) else dtype))


def attn_naive_fwd(q, k, v, causal: bool = False, scale: float | None = None, key_mask=None, workspace=None,
                   stream=None, out=None, lse=None):
    """Materialising baseline.  Returns (o, lse).  Allocates its workspace
    (uint8 device tensor) and outputs with torch unless they are passed."""
    B, H, N, d = _shape4(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = attn_naive_workspace_size(B, H, N, q.dtype)
    ws = workspace if workspace is not None else torch.empty(need, dtype=torch.uint8, device=q.device)
    o = out if out is not None else torch.empty_like(q)
    l = lse if lse is not None else torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    rc = lib.attn_naive_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, N, d, int(bool(causal)),
                            float(scale), _DTYPE[q.dtype], _ptr(key_mask), _ptr(ws), ws.numel(),
                            ctypes.c_void_p(_stream(stream)))
    _check(rc, "attn_naive_fwd")
    return o, l


def attn_deviation_workspace_size(n: int) -> int:
    return int(lib.attn_deviation_workspace_size(int(n)))


def _same_device(a, b):
    if a.numel() != b.numel():
        raise ValueError("a and b must have the same number of elements")
    if not (a.is_cuda and b.is_cuda) or a.device != b.device:
        raise ValueError("a and b must be tensors on one CUDA device")


def attn_deviation(a, b, workspace=None, stream=None) -> dict:
    """Deviation between two device tensors of equal size (synchronous)."""
    _same_device(a, b)
    a = a.contiguous()
    b = b.contiguous()
    n = a.numel()
    with torch.cuda.device(a.device):   # the library launches on the current device
        ws = workspace if workspace is not None else torch.empty(attn_deviation_workspace_size(n),
                                                                 dtype=torch.uint8, device=a.device)
        if not ws.is_cuda or ws.device != a.device:
            raise ValueError("workspace must be on the tensors' device")
        res = DevT()
        rc = lib.attn_deviation(_ptr(a), _DTYPE[a.dtype], _ptr(b), _DTYPE[b.dtype], n, _ptr(ws), ws.numel(),
                                ctypes.c_void_p(_stream(stream)), ctypes.byref(res))
    _check(rc, "attn_deviation")
    return {"max_abs": res.max_abs, "w1": res.w1, "mean_abs": res.mean_abs, "std_abs": res.std_abs,
            "mean_signed": res.mean_signed, "n": res.n}


def attn_deviation_noalloc(a, b, stream=None) -> dict:
    """attn_deviation without a workspace, for callers that cannot allocate
    device memory (the library's own fixed scratch array is used instead;
    n <= DEVIATION_NOALLOC_MAX_N; calls that overlap on the GPU race)."""
    _same_device(a, b)
    a = a.contiguous()
    b = b.contiguous()
    res = DevT()
    with torch.cuda.device(a.device):   # the scratch array and the launch follow the current device
        rc = lib.attn_deviation_noalloc(_ptr(a), _DTYPE[a.dtype], _ptr(b), _DTYPE[b.dtype], a.numel(),
                                        ctypes.c_void_p(_stream(stream)), ctypes.byref(res))
    _check(rc, "attn_deviation_noalloc")
    return {"max_abs": res.max_abs, "w1": res.w1, "mean_abs": res.mean_abs, "std_abs": res.std_abs,
            "mean_signed": res.mean_signed, "n": res.n}


DECODE_MAX_NQ = 8


def attn_decode_workspace_size(B: int, H: int, Nq: int, d: int) -> int:
    return int(lib.attn_decode_workspace_size(B, H, Nq, d))


def attn_decode_fwd(q, k, v, causal: bool = False, scale: float | None = None, key_mask=None, out=None, lse=None,
                    workspace=None, stream=None, want_lse: bool = True):
    """Decode with a key/value cache.  q: [B, H, Nq, d]; k, v: [B, H, Nk, d]
    contiguous device tensors of one dtype (bfloat16 or float32).  Causal:
    query row i is the token at position Nk - Nq + i.  Returns (o, lse)."""
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous device tensors")
    if k.shape != v.shape or q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("k and v must share a shape, and q, k, v a dtype")
    B, H, Nq, d = _shape4(q)
    Bk, Hk, Nk, dk = _shape4(k)
    if (Bk, Hk, dk) != (B, H, d):
        raise ValueError("q and k/v disagree on B, H or d")
    if q.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {q.dtype}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = out if out is not None else torch.empty_like(q)
    l = lse if lse is not None else (torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
                                     if want_lse else None)
    need = attn_decode_workspace_size(B, H, Nq, d)
    ws = workspace if workspace is not None else torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    m = None
    if key_mask is not None:
        m = key_mask
        if m.dtype != torch.float32 or not m.is_contiguous() or m.numel() != B * H * Nk or not m.is_cuda:
            raise ValueError("key_mask must be a contiguous float32 device tensor with B*H*Nk elements")
    rc = lib.attn_decode_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, Nq, Nk, d, int(bool(causal)),
                             float(scale), _DTYPE[q.dtype], _ptr(m), _ptr(ws), ws.numel(),
                             ctypes.c_void_p(_stream(stream)))
    _check(rc, "attn_decode_fwd")
    return o, l


def attn_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(lib.attn_bwd_workspace_size(B, H, N, d))


def attn_bwd(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None, key_mask=None,
             dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients of attention.  q, k, v, o, do: [B, H, N, d] contiguous
    bfloat16 device tensors (o and lse from attn_fwd on the same inputs);
    lse: [B, H, N] float32.  Returns (dq, dk, dv)."""
    ts = (q, k, v, o, do)
    for t in ts:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v, o, do must be contiguous device tensors")
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError("q, k, v, o, do must share one shape and dtype")
    B, H, N, d = _shape4(q)
    if q.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {q.dtype}")
    if (lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or lse.numel() != B * H * N):
        raise ValueError("lse must be a contiguous float32 device tensor with B*H*N elements")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = dq if dq is not None else torch.empty_like(q)
    dk = dk if dk is not None else torch.empty_like(q)
    dv = dv if dv is not None else torch.empty_like(q)
    need = attn_bwd_workspace_size(B, H, N, d)
    ws = workspace if workspace is not None else torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    m = None
    if key_mask is not None:
        m = key_mask
        if m.dtype != torch.float32 or not m.is_contiguous() or m.numel() != B * H * N or not m.is_cuda:
            raise ValueError("key_mask must be a contiguous float32 device tensor with B*H*N elements")
    rc = lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                      B, H, N, d, int(bool(causal)), float(scale), _DTYPE[q.dtype], _ptr(m), _ptr(ws), ws.numel(),
                      ctypes.c_void_p(_stream(stream)))
    _check(rc, "attn_bwd")
    return dq, dk, dv


# Number formats of the emulation (fraction bits, exponent bits).
EMUL_FORMATS = {"bf16": (7, 8), "fp16": (10, 5), "tf32": (10, 8), "fp32": (23, 8), "fp64": (52, 11)}
EMUL_BASELINE, EMUL_TILED = 0, 1


def attn_emul_fwd(q, k, v, causal: bool, scale: float, algo: int, Bc: int, mbits: int, ebits: int,
                  key_mask=None, rows=None, stream=None):
    """Attention with every tensor op rounded to a number format (the
    paper's numerical re-implementation; see include/attn.h).  q, k, v:
    contiguous device tensors [B, H, N, d] (float32, bfloat16 or float64).
    rows: None or a device int64 tensor of flat row ids.  Returns a float64
    device tensor [B, H, N, d] (all rows) or [nrows, d]."""
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous device tensors")
    B, H, N, d = _shape4(q)
    if rows is None:
        o = torch.empty((B, H, N, d), dtype=torch.float64, device=q.device)
        nrows = 0
    else:
        if rows.dtype != torch.int64 or not rows.is_cuda or not rows.is_contiguous():
            raise ValueError("rows must be a contiguous int64 device tensor")
        nrows = rows.numel()
        o = torch.empty((nrows, d), dtype=torch.float64, device=q.device)
    m = None
    if key_mask is not None:
        m = key_mask
        if m.dtype != torch.float32 or not m.is_contiguous() or m.numel() != B * H * N or not m.is_cuda:
            raise ValueError("key_mask must be a contiguous float32 device tensor with B*H*N elements")
    rc = lib.attn_emul_fwd(_ptr(q), _ptr(k), _ptr(v), _DTYPE[q.dtype], _ptr(o), B, H, N, d, int(bool(causal)),
                           float(scale), _ptr(m), int(algo), int(Bc), int(mbits), int(ebits), _ptr(rows), nrows,
                           ctypes.c_void_p(_stream(stream)))
    _check(rc, "attn_emul_fwd")
    return o


def attn_emul_round(x, mbits: int, ebits: int, stream=None):
    """fl(x) for a contiguous float64 device tensor (new tensor)."""
    if x.dtype != torch.float64 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float64 device tensor")
    y = torch.empty_like(x)
    rc = lib.attn_emul_round(_ptr(x), _ptr(y), x.numel(), int(mbits), int(ebits), ctypes.c_void_p(_stream(stream)))
    _check(rc, "attn_emul_round")
    return y


def attn_status(stream=None) -> int:
    return int(lib.attn_status(ctypes.c_void_p(_stream(stream))))


def attn_last_variant() -> str:
    buf = ctypes.create_string_buffer(128)
    lib.attn_last_variant(buf, 128)
    return buf.value.decode()


def attn_debug_wait_timeout(timeout_us: int, stream=None) -> int:
    return int(lib.attn_debug_wait_timeout(int(timeout_us), ctypes.c_void_p(_stream(stream))))
