"""FP64 CPU oracle for exact attention — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product package never imports it
and shares no code with it: the arithmetic lives in ``oracle_attn.c``, a
plain C file compiled here with gcc, and this module only marshals numpy
arrays into it.

Functions
---------
attn(q, k, v, causal, scale, key_mask=None, rows=None, block_mask=None, block=(128, 128))
    The definition of attention, softmax(Q K^T * scale + mask) V, one row at
    a time in binary64 ("Is Flash Attention Stable?" §II-A, the
    Attention(Q,K,V) equation).  Fully masked rows give O = 0, LSE = -inf.
    ``block_mask`` ([..., ceil(N/bq), ceil(N/bk)], non-zero = take part) sets
    every score outside the marked blocks to -inf: the block-sparse reading.
blocked_row(scores, values, width, block_order=None, no_rescale=False)
    The online merge of one row of scores, block by block, with the running
    maximum / denominator / unnormalised-vector state of the yadro-code.ru
    FlashAttention tutorial (the paragraph on merging a new block with a
    larger maximum).  ``no_rescale`` plants the tutorial exercise's mistake.
deviation(a, b)
    Max-abs difference, 1-D Wasserstein-1 via sorting, mean/std of |a-b| and
    the signed mean (the paper's §IV-A and §V measures).
round_fmt(x, mbits, ebits)
    Rounding of binary64 values to an IEEE-style format with ``mbits``
    fraction and ``ebits`` exponent bits (round to nearest even, subnormals,
    overflow to infinity), from the definition (``oracle_emul.c``).
emul(q, k, v, causal, scale, algo, Bc, mbits, ebits, key_mask=None, rows=None, plant=0)
    The paper's numerical re-implementation (§III, §IV-A Fig. 3): baseline
    (algo 0) or tiled (algo 1, key blocks of width Bc) attention with every
    tensor operation's result rounded to that format (``oracle_emul.c``).
attn_bwd(q, k, v, do, causal, scale, key_mask=None, heads=None)
    dL/dQ, dL/dK, dL/dV of the same definition for an upstream gradient dO,
    by the chain rule through the softmax, row by row in binary64
    (``oracle_bwd.c``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_attn.c")
_SRC_EMUL = os.path.join(_HERE, "oracle_emul.c")
_SRC_BWD = os.path.join(_HERE, "oracle_bwd.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ORACLE_NO_RESCALE = 1


def build(force: bool = False) -> str:
    """Compile the oracle's C files into liboracle.so next to them (gcc, -O2, no fast-math)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_SRC_EMUL), os.path.getmtime(_SRC_BWD))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRC, _SRC_EMUL, _SRC_BWD, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_longlong)
            lib.oracle_attn_rows_f64.argtypes = [dp, dp, dp, dp, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                 lp, ctypes.c_longlong, dp, dp, ctypes.c_int]
            lib.oracle_attn_rows_f64.restype = ctypes.c_int
            ubp = ctypes.POINTER(ctypes.c_ubyte)
            lib.oracle_attn_rows_bs_f64.argtypes = [dp, dp, dp, dp, ubp, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_double, lp, ctypes.c_longlong, dp, dp, ctypes.c_int]
            lib.oracle_attn_rows_bs_f64.restype = ctypes.c_int
            ip = ctypes.POINTER(ctypes.c_int)
            lib.oracle_blocked_row_f64.argtypes = [dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ip, ctypes.c_int, dp, dp]
            lib.oracle_blocked_row_f64.restype = ctypes.c_int
            lib.oracle_deviation_f64.argtypes = [dp, dp, ctypes.c_longlong, dp]
            lib.oracle_deviation_f64.restype = ctypes.c_int
            lib.oracle_round_array.argtypes = [dp, dp, ctypes.c_longlong, ctypes.c_int, ctypes.c_int]
            lib.oracle_round_array.restype = None
            lib.oracle_emul_rows.argtypes = [dp, dp, dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, lp, ctypes.c_longlong, dp,
                                             ctypes.c_int]
            lib.oracle_emul_rows.restype = ctypes.c_int
            lib.oracle_emul_rows_planted.argtypes = lib.oracle_emul_rows.argtypes + [ctypes.c_int]
            lib.oracle_emul_rows_planted.restype = ctypes.c_int
            lib.oracle_attn_bwd_f64.argtypes = [dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_double, lp, ctypes.c_longlong,
                                                dp, dp, dp, ctypes.c_int, ctypes.c_int]
            lib.oracle_attn_bwd_f64.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact upcast of a numpy array or CPU torch tensor (any float dtype) to float64."""
    if hasattr(x, "detach"):  # torch tensor: go through float32, exact for bf16/fp16/fp32
        import torch
        t = x.detach().cpu()
        if t.dtype != torch.float64:
            t = t.to(torch.float32).to(torch.float64)
        x = t.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray, ctype=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def attn(q, k, v, causal: bool, scale: float, key_mask=None, rows=None, nthreads: int | None = None,
         block_mask=None, block=(128, 128)):
    """Binary64 attention.

    q, k, v: [..., N, d] (leading dims flattened to BH); key_mask: None or
    [..., N] additive (finite or -inf).  rows: None for every row, else an
    integer array of flat row ids ``bh * N + i``.
    Returns (O, LSE): O [..., N, d] / LSE [..., N] for all rows, or
    O [nrows, d] / LSE [nrows] for a row subset.
    """
    lib = _load()
    Q, K, V = _f64(q), _f64(k), _f64(v)
    if Q.shape != K.shape or Q.shape != V.shape or Q.ndim < 2:
        raise ValueError("q, k, v must share one shape [..., N, d]")
    lead = Q.shape[:-2]
    N, d = Q.shape[-2], Q.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    M = None
    if key_mask is not None:
        M = _f64(key_mask)
        if M.size != BH * N:
            raise ValueError("key_mask must have BH*N elements")
    if rows is None:
        nrows = BH * N
        R = None
    else:
        R = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = R.size
    BM = None
    bq, bk = int(block[0]), int(block[1])
    if block_mask is not None:
        bm = block_mask.detach().cpu().numpy() if hasattr(block_mask, "detach") else np.asarray(block_mask)
        BM = np.ascontiguousarray((bm != 0).astype(np.uint8))
        if BM.size != BH * ((N + bq - 1) // bq) * ((N + bk - 1) // bk):
            raise ValueError("block_mask must have BH * ceil(N/bq) * ceil(N/bk) elements")
    O = np.zeros((nrows, d), dtype=np.float64)
    L = np.zeros((nrows,), dtype=np.float64)
    rc = lib.oracle_attn_rows_bs_f64(_ptr(Q), _ptr(K), _ptr(V), _ptr(M) if M is not None else None,
                                     _ptr(BM, ctypes.c_ubyte) if BM is not None else None, bq, bk,
                                     BH, N, d, 1 if causal else 0, float(scale),
                                     _ptr(R, ctypes.c_longlong) if R is not None else None, nrows,
                                     _ptr(O), _ptr(L), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_attn_rows_f64 failed")
    if rows is None:
        return O.reshape(*lead, N, d), L.reshape(*lead, N)
    return O, L


def blocked_row(scores, values, width: int, block_order=None, no_rescale: bool = False):
    """Online merge of one row (see module docstring).  Returns (out[dv], lse)."""
    lib = _load()
    S = _f64(scores).reshape(-1)
    Vv = _f64(values)
    if Vv.ndim == 1:
        Vv = Vv.reshape(-1, 1)
    n, dv = Vv.shape
    if S.size != n:
        raise ValueError("scores and values disagree on n")
    order = None
    nb = (n + width - 1) // width
    if block_order is not None:
        order = np.ascontiguousarray(np.asarray(block_order, dtype=np.int32))
        if order.size != nb:
            raise ValueError("block_order must list every block once")
    out = np.zeros(dv, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    rc = lib.oracle_blocked_row_f64(_ptr(S), _ptr(Vv), n, dv, int(width),
                                    _ptr(order, ctypes.c_int) if order is not None else None,
                                    ORACLE_NO_RESCALE if no_rescale else 0, _ptr(out), _ptr(lse))
    if rc != 0:
        raise RuntimeError("oracle_blocked_row_f64 failed")
    return out, float(lse[0])


def deviation(a, b) -> dict:
    """max_abs, w1, mean_abs, std_abs, mean_signed and n, in binary64."""
    lib = _load()
    A = _f64(a).reshape(-1)
    B = _f64(b).reshape(-1)
    if A.size != B.size or A.size == 0:
        raise ValueError("a and b must be non-empty and the same size")
    out = np.zeros(5, dtype=np.float64)
    if lib.oracle_deviation_f64(_ptr(A), _ptr(B), A.size, _ptr(out)) != 0:
        raise RuntimeError("oracle_deviation_f64 failed")
    return {"max_abs": out[0], "w1": out[1], "mean_abs": out[2], "std_abs": out[3],
            "mean_signed": out[4], "n": int(A.size)}


# Number formats of the precision sweep (fraction bits, exponent bits).
FORMATS = {"bf16": (7, 8), "fp16": (10, 5), "tf32": (10, 8), "fp32": (23, 8), "fp64": (52, 11)}


def round_fmt(x, mbits: int, ebits: int) -> np.ndarray:
    """fl(x) in the format with ``mbits`` fraction and ``ebits`` exponent bits."""
    lib = _load()
    X = _f64(x)
    Y = np.empty_like(X)
    lib.oracle_round_array(_ptr(X), _ptr(Y), X.size, int(mbits), int(ebits))
    return Y


# Planted mistakes of the emulation (oracle_emul.c), for the oracle's own tests:
# each names the rounding site that is left out, moved or duplicated.
EMUL_PLANTS = {
    "q_in": 1, "k_in": 2, "v_in": 3, "score": 4, "mask_add": 5, "m_diff": 6, "a_exp": 7, "s_diff": 8,
    "p_exp": 9, "a_times_l": 10, "rowsum": 11, "l_add": 12, "a_times_o": 13, "pv": 14, "o_add": 15,
    "div": 16, "l_late": 17, "pv_per_key": 18, "dot_per_term": 19, "softmax": 20, "base_pv": 21,
    "softmax_ops": 22,
}


def emul(q, k, v, causal: bool, scale: float, algo: int, Bc: int, mbits: int, ebits: int,
         key_mask=None, rows=None, nthreads: int | None = None, plant: int = 0) -> np.ndarray:
    """Attention with every tensor op rounded to a format (see oracle_emul.c).

    algo 0: baseline (softmax, then P V); algo 1: tiled online merge over key
    blocks of width Bc.  Returns O [..., N, d] for all rows, or [nrows, d].
    ``plant`` (a value of EMUL_PLANTS) is for the oracle's own tests.
    """
    lib = _load()
    Q, K, V = _f64(q), _f64(k), _f64(v)
    if Q.shape != K.shape or Q.shape != V.shape or Q.ndim < 2:
        raise ValueError("q, k, v must share one shape [..., N, d]")
    lead = Q.shape[:-2]
    N, d = Q.shape[-2], Q.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    M = None
    if key_mask is not None:
        M = _f64(key_mask)
        if M.size != BH * N:
            raise ValueError("key_mask must have BH*N elements")
    R = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nrows = BH * N if R is None else R.size
    O = np.zeros((nrows, d), dtype=np.float64)
    rc = lib.oracle_emul_rows_planted(_ptr(Q), _ptr(K), _ptr(V), _ptr(M) if M is not None else None, BH, N, d,
                                      1 if causal else 0, float(scale), int(algo), int(Bc), int(mbits),
                                      int(ebits), _ptr(R, ctypes.c_longlong) if R is not None else None, nrows,
                                      _ptr(O), nthreads or default_threads(), int(plant))
    if rc != 0:
        raise RuntimeError("oracle_emul_rows failed")
    return O.reshape(*lead, N, d) if R is None else O


ORACLE_BWD_PLANT_NO_CENTER = 1   # drop the softmax Jacobian's rank-one term (planted mistake)
ORACLE_BWD_PLANT_NO_SCALE = 2    # leave `scale` out of dQ and dK (planted mistake)


def attn_bwd(q, k, v, do, causal: bool, scale: float, key_mask=None, heads=None, plant: int = 0,
             nthreads: int | None = None):
    """Binary64 gradients of attention for the upstream gradient ``do``.

    q, k, v, do: [..., N, d] (leading dims flattened to BH); key_mask: None
    or [..., N] additive.  heads: None for every head, else integer head ids
    bh.  Returns (dQ, dK, dV), each [..., N, d] for all heads or
    [nheads, N, d] for a subset.  ``plant`` is for the oracle's own tests.
    """
    lib = _load()
    Q, K, V, dO = _f64(q), _f64(k), _f64(v), _f64(do)
    if not (Q.shape == K.shape == V.shape == dO.shape) or Q.ndim < 2:
        raise ValueError("q, k, v, do must share one shape [..., N, d]")
    lead = Q.shape[:-2]
    N, d = Q.shape[-2], Q.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    M = None
    if key_mask is not None:
        M = _f64(key_mask)
        if M.size != BH * N:
            raise ValueError("key_mask must have BH*N elements")
    Hs = None if heads is None else np.ascontiguousarray(np.asarray(heads, dtype=np.int64))
    nh = BH if Hs is None else Hs.size
    dQ = np.zeros((nh, N, d), dtype=np.float64)
    dK = np.zeros((nh, N, d), dtype=np.float64)
    dV = np.zeros((nh, N, d), dtype=np.float64)
    rc = lib.oracle_attn_bwd_f64(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(M) if M is not None else None,
                                 BH, N, d, 1 if causal else 0, float(scale),
                                 _ptr(Hs, ctypes.c_longlong) if Hs is not None else None, nh,
                                 _ptr(dQ), _ptr(dK), _ptr(dV), int(plant), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_attn_bwd_f64 failed")
    if heads is None:
        return dQ.reshape(*lead, N, d), dK.reshape(*lead, N, d), dV.reshape(*lead, N, d)
    return dQ, dK, dV
