"""Host-side checks of the C ABI: the library builds, loads without a GPU,
exports every symbol include/attn.h declares, and rejects bad arguments
synchronously without launching anything."""
import ctypes
import importlib.util
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    spec = importlib.util.spec_from_file_location(
        "_eta_build", os.path.join(ROOT, "exact_tiled_attention_17_gb300", "_build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    path = mod.build()
    return ctypes.CDLL(path)


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*(attn_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("attn_fwd", "attn_naive_fwd", "attn_deviation"):
        assert must in names
    assert len(names) >= 9


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_binding_exports_match_header():
    import exact_tiled_attention_17_gb300 as eta
    assert sorted(eta.EXPORTS) == _declared_functions()


def test_sizes_and_strings(lib):
    lib.attn_naive_workspace_size.restype = ctypes.c_size_t
    lib.attn_naive_workspace_size.argtypes = [ctypes.c_int] * 4
    # the tutorial's arithmetic: 8192 tokens, 2-byte scores: 128 MiB per head, 4 GiB for 32 heads
    assert lib.attn_naive_workspace_size(1, 1, 8192, 1) == 128 * 2 ** 20
    assert lib.attn_naive_workspace_size(1, 32, 8192, 1) == 4 * 2 ** 30
    assert lib.attn_naive_workspace_size(1, 1, 100, 0) == 100 * 100 * 4
    assert lib.attn_naive_workspace_size(0, 1, 100, 0) == 0
    assert lib.attn_naive_workspace_size(1, 1, 100, 7) == 0
    lib.attn_deviation_workspace_size.restype = ctypes.c_size_t
    lib.attn_deviation_workspace_size.argtypes = [ctypes.c_longlong]
    assert lib.attn_deviation_workspace_size(0) == 0
    assert lib.attn_deviation_workspace_size(1000) >= 3 * 8 * 1000
    lib.attn_strerror.restype = ctypes.c_char_p
    lib.attn_strerror.argtypes = [ctypes.c_int]
    for code in range(-5, 1):
        assert lib.attn_strerror(code)
    assert b"timed out" in lib.attn_strerror(-5)


def _fwd(lib, **kw):
    args = dict(Q=16, K=16, V=16, O=16, LSE=0, B=1, H=1, N=8, d=64, causal=0, scale=0.125, Br=0, Bc=0,
                dtype=1, mask=0, stream=0)
    args.update(kw)
    vp = ctypes.c_void_p
    f = lib.attn_fwd
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp] + [ctypes.c_int] * 5 + [ctypes.c_float] + [ctypes.c_int] * 3 + [vp, vp]
    return f(vp(args["Q"]) if args["Q"] else None, vp(args["K"]) if args["K"] else None,
             vp(args["V"]) if args["V"] else None, vp(args["O"]) if args["O"] else None,
             vp(args["LSE"]) if args["LSE"] else None, args["B"], args["H"], args["N"], args["d"],
             args["causal"], args["scale"], args["Br"], args["Bc"], args["dtype"],
             vp(args["mask"]) if args["mask"] else None, None)


def test_argument_rejection_without_launch(lib):
    # fake, never dereferenced pointers: every call must be rejected on the host
    assert _fwd(lib, Q=0) == -1
    assert _fwd(lib, N=0) == -1
    assert _fwd(lib, B=-1) == -1
    assert _fwd(lib, scale=0.0) == -1
    assert _fwd(lib, scale=float("nan")) == -1
    assert _fwd(lib, scale=-1.0) == -1
    assert _fwd(lib, Q=24) == -1                  # not 16-byte aligned
    assert _fwd(lib, causal=2) == -1
    assert _fwd(lib, mask=18) == -1               # mask not 4-byte aligned
    assert _fwd(lib, dtype=9) == -1
    assert _fwd(lib, d=96) == -2                  # bf16 supports d in {64, 128}
    assert _fwd(lib, Br=32, Bc=64) == -2
    assert _fwd(lib, Br=128, Bc=96) == -2
    assert _fwd(lib, dtype=0, d=129) == -2
    assert _fwd(lib, dtype=0, Br=128, Bc=128) == -2
    assert _fwd(lib, dtype=2) == -2


def test_naive_and_deviation_rejection(lib):
    vp = ctypes.c_void_p
    f = lib.attn_naive_fwd
    f.restype = ctypes.c_int
    f.argtypes = [vp] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int, vp, vp, ctypes.c_size_t, vp]
    p = vp(16)
    assert f(p, p, p, p, None, 1, 1, 8, 64, 0, 0.125, 1, None, None, 0, None) == -3      # no workspace
    assert f(p, p, p, p, None, 1, 1, 8, 64, 0, 0.125, 1, None, p, 100, None) == -3       # too small
    assert f(p, p, p, p, None, 1, 1, 8, 200, 0, 0.125, 1, None, p, 1 << 20, None) == -2  # d > 128
    g = lib.attn_deviation
    g.restype = ctypes.c_int
    g.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, ctypes.c_longlong, vp, ctypes.c_size_t, vp, vp]
    out = ctypes.create_string_buffer(64)
    assert g(p, 0, p, 0, 0, p, 1 << 20, None, out) == -1                                 # n = 0
    assert g(p, 0, p, 5, 10, p, 1 << 20, None, out) == -1                                # bad dtype
    assert g(p, 0, p, 0, 10, None, 0, None, out) == -3                                   # no workspace
    assert g(p, 0, p, 0, 10, vp(16 + 256), 1 << 20, None, out) == -3                     # misaligned


def test_debug_timeout_rejects_bad_limit(lib):
    f = lib.attn_debug_wait_timeout
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_uint, ctypes.c_void_p]
    assert f(0, None) == -1
    assert f(2_000_000, None) == -1


def test_backward_and_block_sparse_rejection(lib):
    vp = ctypes.c_void_p
    ws_size = lib.attn_bwd_workspace_size
    ws_size.restype = ctypes.c_size_t
    ws_size.argtypes = [ctypes.c_int] * 4
    # LSE and D vectors padded to 64 rows (256-byte aligned each), plus the f32 dQ accumulator
    assert ws_size(1, 1, 100, 64) == 2 * 512 + 100 * 64 * 4
    assert ws_size(2, 16, 4096, 128) == 2 * 32 * 4096 * 4 + 32 * 4096 * 128 * 4
    assert ws_size(0, 1, 100, 64) == 0
    f = lib.attn_bwd
    f.restype = ctypes.c_int
    f.argtypes = [vp] * 9 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int, vp, vp, ctypes.c_size_t, vp]
    p, big = vp(256), 1 << 30

    def bwd(**kw):
        a = dict(Q=p, K=p, V=p, O=p, dO=p, LSE=p, dQ=p, dK=p, dV=p, B=1, H=1, N=8, d=64, causal=0, scale=0.125,
                 dtype=1, mask=None, ws=p, ws_bytes=big)
        a.update(kw)
        return f(a["Q"], a["K"], a["V"], a["O"], a["dO"], a["LSE"], a["dQ"], a["dK"], a["dV"], a["B"], a["H"],
                 a["N"], a["d"], a["causal"], a["scale"], a["dtype"], a["mask"], a["ws"], a["ws_bytes"], None)

    assert bwd(dO=None) == -1
    assert bwd(LSE=None) == -1
    assert bwd(dQ=vp(264)) == -1                 # not 16-byte aligned
    assert bwd(LSE=vp(258)) == -1                # not 4-byte aligned
    assert bwd(causal=3) == -1
    assert bwd(dtype=2) == -2                    # float64: bf16 or float32 only
    assert bwd(dtype=0, d=200) == -2             # float32: d <= 128
    assert bwd(dtype=0, ws=None) == -3
    assert bwd(d=96) == -2                       # bf16: d in {64, 128}
    assert bwd(ws=None) == -3
    assert bwd(ws_bytes=100) == -3
    assert bwd(ws=vp(256 + 16)) == -3            # not 256-byte aligned
    g = lib.attn_fwd_block_sparse
    g.restype = ctypes.c_int
    g.argtypes = [vp] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int, vp, vp, vp]

    def bs(**kw):
        a = dict(N=8, d=64, dtype=1, bm=p)
        a.update(kw)
        return g(p, p, p, p, None, 1, 1, a["N"], a["d"], 0, 0.125, a["dtype"], a["bm"], None, None)

    assert bs(bm=None) == -1
    assert bs(dtype=0) == -2
    assert bs(d=96) == -2
    assert bs(N=131073) == -2


def test_host_entry_sizes_and_rejection(lib):
    """attn_fwd_host: workspace arithmetic, and argument errors returned
    before any copy is enqueued (fake, never dereferenced pointers)."""
    vp = ctypes.c_void_p
    ws_size = lib.attn_fwd_host_workspace_size
    ws_size.restype = ctypes.c_size_t
    ws_size.argtypes = [ctypes.c_int] * 6
    t = 2 * 16 * 4096 * 128 * 2                       # one bf16 tensor of the bench shape
    r = 2 * 16 * 4096 * 4                             # one float32 row vector
    assert ws_size(2, 16, 4096, 128, 1, 0) == 4 * t + r
    assert ws_size(2, 16, 4096, 128, 1, 1) == 4 * t + 2 * r
    assert ws_size(1, 1, 3, 5, 0, 0) == 4 * 256 + 256  # every part on a 256-byte boundary
    assert ws_size(1, 1, 8, 64, 2, 0) == 0             # float64 is not a forward dtype
    assert ws_size(0, 1, 8, 64, 1, 0) == 0
    f = lib.attn_fwd_host
    f.restype = ctypes.c_int
    f.argtypes = [vp] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float] + [ctypes.c_int] * 3 + [vp, vp, ctypes.c_size_t, vp]
    p, big = vp(256), 1 << 30

    def host(**kw):
        a = dict(Q=p, O=p, N=8, d=64, causal=0, scale=0.125, Br=0, Bc=0, dtype=1, ws=p, ws_bytes=big)
        a.update(kw)
        return f(a["Q"], p, p, a["O"], None, 1, 1, a["N"], a["d"], a["causal"], a["scale"], a["Br"], a["Bc"],
                 a["dtype"], None, a["ws"], a["ws_bytes"], None)

    assert host(Q=None) == -1
    assert host(O=None) == -1
    assert host(N=0) == -1
    assert host(scale=0.0) == -1
    assert host(causal=2) == -1
    assert host(ws=None) == -3
    assert host(ws_bytes=1000) == -3
    assert host(ws=vp(256 + 16)) == -3               # not 256-byte aligned
    assert host(d=96) == -2                          # bf16: d in {64, 128}
    assert host(Bc=96) == -2
    assert host(dtype=2) == -2
    assert host(dtype=0, Br=128) == -2


def test_decode_sizes_and_rejection(lib):
    """attn_decode_fwd: the workspace holds the partial results of up to 128
    key splits; argument errors are returned before anything is launched
    (fake, never dereferenced pointers)."""
    vp = ctypes.c_void_p
    ws_size = lib.attn_decode_workspace_size
    ws_size.restype = ctypes.c_size_t
    ws_size.argtypes = [ctypes.c_int] * 4
    # per split and row: m, l and d partial sums, float32
    assert ws_size(1, 32, 1, 128) == 128 * 32 * 1 * (2 + 128) * 4
    assert ws_size(2, 8, 4, 64) == 128 * 16 * 4 * (2 + 64) * 4
    assert ws_size(0, 1, 1, 64) == 0
    f = lib.attn_decode_fwd
    f.restype = ctypes.c_int
    f.argtypes = [vp] * 5 + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_int, vp, vp, ctypes.c_size_t, vp]
    p, big = vp(256), 1 << 30

    def dec(**kw):
        a = dict(Q=p, K=p, V=p, O=p, B=1, H=1, Nq=1, Nk=64, d=64, causal=0, scale=0.125, dtype=1, mask=None,
                 ws=p, ws_bytes=big)
        a.update(kw)
        return f(a["Q"], a["K"], a["V"], a["O"], None, a["B"], a["H"], a["Nq"], a["Nk"], a["d"], a["causal"],
                 a["scale"], a["dtype"], a["mask"], a["ws"], a["ws_bytes"], None)

    assert dec(Q=None) == -1
    assert dec(Nq=0) == -1
    assert dec(Nk=-1) == -1
    assert dec(scale=0.0) == -1
    assert dec(scale=float("inf")) == -1
    assert dec(causal=2) == -1
    assert dec(causal=1, Nq=8, Nk=4) == -1          # causal needs Nq <= Nk
    assert dec(dtype=7) == -1
    assert dec(dtype=2) == -2                       # float64: bf16 or float32 only
    assert dec(Nq=9) == -2                          # at most 8 new rows
    assert dec(d=48) == -2                          # d a multiple of 32, at most 128
    assert dec(d=160) == -2
    assert dec(K=vp(264)) == -1                     # not 16-byte aligned
    assert dec(mask=vp(258)) == -1                  # not 4-byte aligned
    assert dec(ws=None) == -3
    assert dec(ws_bytes=100) == -3
    assert dec(ws=vp(264)) == -3                    # not 16-byte aligned


def test_emulation_rejection(lib):
    """attn_emul_fwd / attn_emul_round: argument errors are returned before
    anything is launched (fake, never dereferenced pointers); n = 0 rounds
    nothing and returns ATTN_OK."""
    vp = ctypes.c_void_p
    f = lib.attn_emul_fwd
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, vp, ctypes.c_int, vp] + [ctypes.c_int] * 5 + [ctypes.c_float, vp] + [ctypes.c_int] * 4 + \
                 [vp, ctypes.c_longlong, vp]
    p = vp(256)
    BASELINE, TILED = 0, 1

    def emul(**kw):
        a = dict(Q=p, dtype=1, O=p, N=8, d=64, causal=0, scale=0.125, mask=None, algo=TILED, Bc=4, mb=7, eb=8,
                 rows=None, nrows=0)
        a.update(kw)
        return f(a["Q"], p, p, a["dtype"], a["O"], 1, 1, a["N"], a["d"], a["causal"], a["scale"], a["mask"],
                 a["algo"], a["Bc"], a["mb"], a["eb"], a["rows"], a["nrows"], None)

    assert emul(Q=None) == -1
    assert emul(N=0) == -1
    assert emul(scale=-1.0) == -1
    assert emul(causal=5) == -1
    assert emul(dtype=9) == -1
    assert emul(algo=4) == -1
    assert emul(mb=0) == -1 and emul(mb=53) == -1
    assert emul(eb=1) == -1 and emul(eb=12) == -1
    assert emul(rows=p, nrows=-1) == -1
    assert emul(Bc=0) == -1
    assert emul(d=129) == -2
    assert emul(mask=vp(258)) == -1                 # not 4-byte aligned
    assert emul(O=vp(260)) == -1                    # not 8-byte aligned
    g = lib.attn_emul_round
    g.restype = ctypes.c_int
    g.argtypes = [vp, vp, ctypes.c_longlong, ctypes.c_int, ctypes.c_int, vp]
    assert g(None, p, 4, 7, 8, None) == -1
    assert g(p, p, -1, 7, 8, None) == -1
    assert g(p, p, 4, 0, 8, None) == -1
    assert g(p, vp(260), 4, 7, 8, None) == -1
    assert g(p, p, 0, 7, 8, None) == 0               # nothing to round
