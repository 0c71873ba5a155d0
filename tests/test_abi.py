"""The C ABI loads, exports every symbol include/gdr.h declares, and rejects bad
arguments synchronously -- host-only checks, no GPU and no kernel launch."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import gated_delta_rule_gdr_gb300 as gdr
from gated_delta_rule_gdr_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdr.h")


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdr.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdr_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("gdr_chunk_fwd", "gdr_decode_step", "gdr_chunk_decay", "gdr_chunk_wy",
                 "gdr_chunk_state", "gdr_chunk_output", "gdr_last_device_error",
                 "gdr_status_string", "gdr_version"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_status_strings(lib):
    assert gdr.version().startswith("gdr ")
    assert "sm_103a" in gdr.version()
    for code in range(6):
        s = gdr.status_string(code)
        assert s and s != "unknown status"
    assert gdr.status_string(99) == "unknown status"


P = ctypes.c_void_p(0x1000)   # never dereferenced: every case fails validation first


def fwd(lib, **kw):
    a = dict(q=P, k=P, v=P, g=P, beta=P, a_min=0.95, init=None, out=P, fin=None, B=1, H=1,
             T=64, dk=128, dv=128, chunk=64, dtype=1, stream=None)
    a.update(kw)
    return lib.gdr_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["a_min"], a["init"],
                             a["out"], a["fin"], a["B"], a["H"], a["T"], a["dk"], a["dv"],
                             a["chunk"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), 1), (dict(H=-2), 1), (dict(T=-1), 1),
    (dict(a_min=0.0), 1), (dict(a_min=-0.5), 1), (dict(a_min=1.5), 1),
    (dict(a_min=float("nan")), 1),
    (dict(dk=96), 2), (dict(dv=256), 2), (dict(chunk=128), 2), (dict(chunk=8), 2),
    (dict(dtype=7), 2),
    (dict(a_min=0.2), 3),                 # 64 * -ln 0.2 = 103 > 80
    (dict(a_min=0.28), 3),                # 64 * -ln 0.28 = 81.5 > 80
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(g=None), 1),
    (dict(beta=None), 1), (dict(out=None), 1),
])
def test_chunk_fwd_rejects(lib, kw, code):
    assert fwd(lib, **kw) == code


def test_range_rule_boundary(lib):
    # chunk = 16 allows a_min down to e^-5 (the pages' own per-step floor)
    assert fwd(lib, chunk=16, a_min=0.00674, q=None) == 1     # e^-5 = 0.006738: in range
    assert fwd(lib, chunk=16, a_min=0.0067, q=None) == 3


def test_empty_inputs_are_a_no_op(lib):
    assert fwd(lib, B=0, q=None, k=None) == 0
    assert fwd(lib, H=0, q=None) == 0


def test_decode_rejects(lib):
    d = lib.gdr_decode_step
    assert d(P, P, P, P, P, 0.95, P, P, -1, 1, 128, 128, 1, None) == 1
    assert d(P, P, P, P, P, 0.0, P, P, 1, 1, 128, 128, 1, None) == 1
    assert d(P, P, P, P, P, 0.95, P, P, 1, 1, 100, 128, 1, None) == 2
    assert d(P, P, P, P, P, 0.95, None, P, 1, 1, 128, 128, 1, None) == 1
    assert d(P, P, P, P, P, 0.95, P, P, 0, 4, 128, 128, 1, None) == 0   # empty


def test_staged_steps_reject(lib):
    assert lib.gdr_chunk_decay(P, 0.0, P, 1, 64, 64, None) == 1
    assert lib.gdr_chunk_decay(P, 0.9, P, 1, 64, 48, None) == 2
    assert lib.gdr_chunk_decay(P, 0.1, P, 1, 64, 64, None) == 3
    assert lib.gdr_chunk_decay(None, 0.9, P, 1, 64, 64, None) == 1
    assert lib.gdr_chunk_wy(P, P, P, P, P, P, 1, 64, 48, 64, 64, 1, None) == 2
    assert lib.gdr_chunk_wy(P, P, None, P, P, P, 1, 64, 64, 64, 64, 1, None) == 1
    assert lib.gdr_chunk_state(P, P, P, P, None, None, None, None, 1, 64, 64, 64, 64, 0,
                               None) == 1
    assert lib.gdr_chunk_output(P, P, P, P, P, P, -1, 64, 64, 64, 64, 0, None) == 1


def test_binding_fails_loudly_without_cuda_tensors(lib):
    import torch
    q = torch.zeros(1, 1, 4, 16)
    with pytest.raises(ValueError):
        gdr.chunk_fwd(q, q, q, torch.zeros(1, 1, 4), torch.zeros(1, 1, 4), 0.9, chunk=16)


def test_path_query(lib):
    q = lib.gdr_chunk_fwd_path
    assert q(1, 2, 256, 64, 64, 64, 0.9, 0) == 6          # fp32: one-pass CUDA-core kernel
    assert q(1, 2, 0, 128, 128, 64, 0.95, 1) == 0         # empty: no kernel
    assert q(1, 2, 256, 48, 128, 64, 0.95, 1) == -1       # rejected
    with gdr.option(fused_variant=1):
        assert q(4, 16, 4096, 128, 128, 64, 0.95, 1) == 2
    with gdr.option(fused_variant=2):
        assert q(4, 16, 4096, 128, 128, 64, 0.95, 1) == 3
    assert lib.gdr_chunk_fwd_ws_path(1, 2, 256, 64, 64, 64, 0.9, 0) == 1   # staged, workspace
    assert lib.gdr_chunk_fwd_kernels(1, 2, 256, 64, 64, 64, 0.9, 0) == 1


def test_options(lib):
    assert gdr.get_option("wait_limit_ns") == 2_000_000_000
    for name in ("fused_variant", "chain_split", "segments"):
        assert gdr.get_option(name) == 0
    with gdr.option(chain_split=2, segments=5):
        assert gdr.get_option("chain_split") == 2 and gdr.get_option("segments") == 5
    assert gdr.get_option("chain_split") == 0 and gdr.get_option("segments") == 0
    assert lib.gdr_set_option(1, 3) == 1                  # fused_variant out of range
    assert lib.gdr_set_option(0, -1) == 1                 # negative wait limit
    assert lib.gdr_set_option(99, 0) == 1                 # unknown option
    assert lib.gdr_get_option(99) == -1


def test_workspace_sizes(lib):
    ws = lib.gdr_chunk_fwd_workspace_size
    # staged shapes: 4 (BH T (1 + dk + 2 dv) + BH ceil(T / C) dk dv) bytes
    assert ws(1, 2, 256, 64, 64, 64, 0) == 4 * (2 * 256 * (1 + 64 + 128) + 2 * 4 * 64 * 64)
    assert ws(1, 1, 100, 32, 16, 32, 1) == 4 * (100 * (1 + 32 + 32) + 4 * 32 * 16)
    # two-kernel path: 16 KB per chunk
    assert ws(4, 16, 4096, 128, 128, 64, 1) >= 64 * 64 * 16384
    assert ws(1, 2, 0, 64, 64, 64, 0) == 0 and ws(1, 2, 64, 48, 64, 64, 0) == 0


def test_varlen_rejects(lib):
    f = lib.gdr_chunk_fwd_varlen
    args = lambda **kw: [kw.get(n, d) for n, d in (
        ("q", P), ("k", P), ("v", P), ("g", P), ("beta", P), ("a_min", 0.95), ("init", None),
        ("out", P), ("fin", None), ("cu", P), ("S", 2), ("H", 2), ("tt", 100), ("dk", 128),
        ("dv", 128), ("chunk", 64), ("dtype", 1), ("stream", None))]
    assert f(*args(S=-1)) == 1                 # GDR_ERR_INVALID_ARG
    assert f(*args(dtype=2)) == 2              # unknown dtype
    assert f(*args(dk=48)) == 2                # dimensions 16, 32, 64, 128 only
    assert f(*args(chunk=48)) == 2             # chunks 16, 32, 64 only
    assert f(*args(a_min=0.2)) == 3            # range rule
    assert f(*args(cu=None)) == 1              # offsets required
    assert f(*args(q=None)) == 1
    assert f(*args(S=0)) == 0                  # no sequences: nothing to do


def ex(lib, **kw):
    a = dict(q=P, k=P, v=P, g=P, beta=P, decay=1, bound=-5.0, init=None, out=P, fin=None, B=1,
             H=1, T=64, dk=128, dv=128, chunk=16, dtype=1, ws=None, wsb=0, stream=None)
    a.update(kw)
    f = lib.gdr_chunk_fwd_ex
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_float] + [ctypes.c_void_p] * 3 + \
        [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f(a["q"], a["k"], a["v"], a["g"], a["beta"], a["decay"], a["bound"], a["init"],
             a["out"], a["fin"], a["B"], a["H"], a["T"], a["dk"], a["dv"], a["chunk"], a["dtype"],
             a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(decay=2), 1), (dict(decay=-1), 1),                  # no such decay mode
    (dict(bound=0.5), 1), (dict(bound=float("nan")), 1),      # log floor must be <= 0
    (dict(decay=0, bound=0.0), 1), (dict(decay=0, bound=1.5), 1),
    (dict(chunk=64), 3),                                       # 64 * 5 = 320 > 80
    (dict(bound=-5.01), 3),                                    # 16 * 5.01 > 80
    (dict(q=None), 1),                                         # in range: the pages' setting
    (dict(chunk=64, bound=-1.25, q=None), 1),                  # 64 * 1.25 = 80: in range
    (dict(chunk=64, bound=-1.26), 3),
    (dict(decay=0, bound=0.95, chunk=64, q=None), 1),          # the linear form through _ex
])
def test_chunk_fwd_ex_rejects(lib, kw, code):
    """The decay-mode entry point (the pages' log-domain form log alpha = g_min sigmoid(g)
    and the linear-domain floor) validates the mode, the bound and the range rule."""
    assert ex(lib, **kw) == code


def test_workspace_path_range_rule(lib):
    """The two-kernel workspace path applies the range rule over a 16-token tile (its
    preparation splits the decay at 16-row reference points), the other paths over the
    chunk: with a workspace, g_min = -5 and a floor of 0.05 pass at chunk 64 (the null q
    is then what fails), one step beyond the tile bound is GDR_ERR_RANGE."""
    big = 1 << 40
    assert ex(lib, chunk=64, bound=-5.0, ws=P, wsb=big, q=None) == 1
    assert ex(lib, chunk=64, bound=-5.01, ws=P, wsb=big) == 3
    assert ex(lib, chunk=64, bound=-5.0, ws=P, wsb=16) == 3      # too small: single-launch rule
    assert ex(lib, decay=0, bound=0.05, chunk=64, ws=P, wsb=big, q=None) == 1
    assert ex(lib, decay=0, bound=0.006, chunk=64, ws=P, wsb=big) == 3   # 16 * 5.12 > 80
    wp = lib.gdr_chunk_fwd_ws_path
    wp.argtypes = [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_int]
    wp.restype = ctypes.c_int
    fp = lib.gdr_chunk_fwd_path
    fp.argtypes = [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_int]
    fp.restype = ctypes.c_int
    assert wp(1, 2, 300, 128, 128, 64, 0.05, 1) in (4, 5)
    assert fp(1, 2, 300, 128, 128, 64, 0.05, 1) == -1
    assert wp(1, 2, 300, 128, 128, 64, 0.006, 1) == -1
    assert wp(1, 2, 300, 128, 128, 64, 0.95, 1) in (4, 5)


def test_decode_ex_rejects(lib):
    d = lib.gdr_decode_step_ex
    d.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_float] + [ctypes.c_void_p] * 2 + \
        [ctypes.c_int] * 5 + [ctypes.c_void_p]
    d.restype = ctypes.c_int
    assert d(P, P, P, P, P, 1, 0.5, P, P, 1, 1, 128, 128, 1, None) == 1      # log floor > 0
    assert d(P, P, P, P, P, 3, -5.0, P, P, 1, 1, 128, 128, 1, None) == 1     # unknown mode
    assert d(P, P, P, P, P, 1, -5.0, P, P, 0, 4, 128, 128, 1, None) == 0     # empty
    assert d(P, P, P, P, P, 1, -5.0, None, P, 1, 1, 128, 128, 1, None) == 1  # no state


def bwd(lib, **kw):
    a = dict(q=P, k=P, v=P, g=P, beta=P, decay=0, bound=0.9, init=None, dout=P, dfin=None,
             dq=P, dk_=P, dv_=P, dg=P, db=P, dinit=None, B=1, H=2, T=100, dk=64, dv=64,
             chunk=64, dtype=0, ws=P, wsb=1 << 40, stream=None)
    a.update(kw)
    f = lib.gdr_chunk_bwd
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_float] + \
        [ctypes.c_void_p] * 9 + [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_size_t,
                                                       ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f(*(a[n] for n in ("q", "k", "v", "g", "beta", "decay", "bound", "init", "dout",
                              "dfin", "dq", "dk_", "dv_", "dg", "db", "dinit", "B", "H", "T",
                              "dk", "dv", "chunk", "dtype", "ws", "wsb", "stream")))


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), 1), (dict(decay=5), 1), (dict(bound=0.0), 1),  # sizes, decay mode, floor
    (dict(dtype=7), 2), (dict(dk=16), 2), (dict(dv=8), 2), (dict(chunk=128), 2),
    (dict(bound=0.2), 3),                                        # 64 * -ln(0.2) > 80
    (dict(decay=1, bound=-5.0), 3), (dict(decay=1, bound=-5.0, chunk=16, q=None), 1),
    (dict(q=None), 1), (dict(dout=None), 1), (dict(dg=None), 1), (dict(db=None), 1),
    (dict(ws=None), 1), (dict(wsb=1024), 1),                     # workspace missing / small
    (dict(ws=ctypes.c_void_p(0x1008)), 1),                       # not 16-byte aligned
    (dict(k=ctypes.c_void_p(0x1004)), 1), (dict(dout=ctypes.c_void_p(0x1002)), 1),
    (dict(B=0), 0), (dict(H=0), 0),                              # no heads: nothing to do
])
def test_chunk_bwd_rejects(lib, kw, code):
    """The backward's entry point validates everything before it enqueues anything."""
    assert bwd(lib, **kw) == code


def test_chunk_bwd_workspace_size(lib):
    f = lib.gdr_chunk_bwd_workspace_size
    f.argtypes = [ctypes.c_int] * 7
    f.restype = ctypes.c_size_t
    n = f(2, 3, 100, 128, 64, 64, 1)
    # gamma, U, Wk, dR per token; W per token padded to whole chunks; M_n, dM' and the
    # P, T, DK tiles per chunk; fp32 words
    tok, pad, st, tiles = 2 * 3 * 100, 2 * 3 * 128, 2 * 3 * 2 * 128 * 64, 2 * 3 * 2 * 64 * 64
    assert n == 4 * (tok + 2 * tok * 64 + tok * 128 + pad * 64 + 2 * st + 3 * tiles)
    assert f(2, 3, 0, 128, 64, 64, 1) == 0 and f(0, 3, 10, 128, 64, 64, 1) == 0
    assert f(1, 1, 10, 16, 64, 64, 1) == 0   # unsupported dk


def test_chunk_fwd_host_rejects(lib):
    f = lib.gdr_chunk_fwd_host
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_float] + [ctypes.c_void_p] * 3 + \
        [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    f.restype = ctypes.c_int
    sz = lib.gdr_chunk_fwd_host_buffer_size
    sz.argtypes = [ctypes.c_int] * 7
    sz.restype = ctypes.c_size_t
    need = sz(1, 2, 100, 128, 128, 64, 1)
    assert need > 0 and need % 256 == 0
    buf = ctypes.c_void_p(0x100000)

    def call(**kw):
        a = dict(q=P, k=P, v=P, g=P, beta=P, a=0.95, init=None, out=P, fin=None, B=1, H=2, T=100,
                 dk=128, dv=128, chunk=64, dt=1, buf=buf, n=need)
        a.update(kw)
        return f(a["q"], a["k"], a["v"], a["g"], a["beta"], a["a"], a["init"], a["out"], a["fin"],
                 a["B"], a["H"], a["T"], a["dk"], a["dv"], a["chunk"], a["dt"], a["buf"], a["n"], None)
    assert call(n=need - 1) == 1                          # buffer too small
    assert call(buf=ctypes.c_void_p(0x100010)) == 1       # not 256-byte aligned
    assert call(buf=None) == 1
    assert call(q=None) == 1 and call(out=None) == 1
    assert call(a=0.0) == 1 and call(a=0.001) == 3        # floor; range over the 16-token tile
    assert call(dk=48) == 2 and call(dt=5) == 2
    assert call(B=0) == 0                                  # no heads: nothing to do
    assert sz(1, 2, 100, 48, 128, 64, 1) == 0


def test_static_entry_rejects_oversized_work_before_any_device_call(lib):
    """The allocation-free prefill checks its size limit on the host, in 64-bit
    arithmetic that cannot overflow, before it touches a device."""
    f = lib.gdr_chunk_fwd_static
    args = lambda B, H, T, d=128, C=64: (P, P, P, P, P, 0.95, None, P, None, B, H, T, d, d, C, 1,
                                         None)
    assert f(*args(65536, 65536, 1)) == 2                 # B H beyond int32
    assert f(*args(46340, 46340, 2**31 - 1)) == 2         # B H T far beyond the array
    assert f(*args(1, 2**20, 2**20)) == 2
    assert f(*args(4, 16, 4096)) == 2                     # the prefill workload: ~ 2.3 GB
    # 4 (B H T (1 + dk + 2 dv) + B H ceil(T / C) dk dv) against 32 MiB at d = 64, C = 64:
    # T = 16320 for two heads needs 512 bytes less than the array, T = 16321 more
    assert f(*args(1, 2, 16321, d=64)) == 2
    assert f(*args(1, 2, 16320, d=64, C=48)) == 2         # unsupported chunk
    assert f(*args(1, 2, 64, d=64)[:5] + (0.0,) + args(1, 2, 64, d=64)[6:]) == 1   # a_min


def test_mla_decode_rejects(lib):
    f = lib.gdr_mla_decode
    args = lambda **kw: [kw.get(n, d) for n, d in (
        ("q", P), ("c", P), ("lens", P), ("w", P), ("z", P), ("scale", 0.088), ("out", P),
        ("N", 2), ("H", 64), ("L", 100), ("dc", 512), ("dh", 128), ("ws", P), ("wsb", 1 << 40),
        ("stream", None))]
    assert f(*args(N=-1)) == 1
    assert f(*args(scale=0.0)) == 1
    assert f(*args(scale=float("nan"))) == 1
    assert f(*args(N=0)) == 0                              # nothing to do
    assert f(*args(dc=256)) == 2                           # latent width 512 only
    assert f(*args(H=48)) == 2                             # heads in groups of 64
    assert f(*args(dh=130)) == 2
    assert f(*args(L=0)) == 2
    assert f(*args(q=None)) == 1
    assert f(*args(q=ctypes.c_void_p(0x1008))) == 1        # not 16-byte aligned
    assert f(*args(ws=None)) == 1
    assert f(*args(wsb=16)) == 1                           # workspace too small
    ws = lib.gdr_mla_decode_workspace_size
    assert ws(2, 64, 100, 512, 128) > 0 and ws(2, 64, 100, 256, 128) == 0
    assert ws(0, 64, 100, 512, 128) == 0


def test_chunk_saved_size(lib):
    f = lib.gdr_chunk_saved_size
    f.argtypes = [ctypes.c_int] * 7
    f.restype = ctypes.c_size_t
    # per (b, h, chunk): the state transposed (128 x 128) and W transposed (128 x 64),
    # T and P (64 x 64 each), bf16; four rows of 64 fp32 scalars
    per = 128 * (128 + 64) * 2 + 2 * 64 * 64 * 2 + 4 * 64 * 4
    assert per == 66560
    assert f(2, 3, 100, 128, 128, 64, 1) == 2 * 3 * 2 * per
    assert f(1, 1, 64, 128, 128, 64, 1) == per
    assert f(1, 1, 0, 128, 128, 64, 1) == 0 and f(0, 1, 64, 128, 128, 64, 1) == 0
    assert f(1, 1, 64, 128, 128, 64, 0) == 0      # fp32: not the two-kernel path
    assert f(1, 1, 64, 64, 128, 64, 1) == 0 and f(1, 1, 64, 128, 128, 32, 1) == 0


def train(lib, **kw):
    a = dict(q=P, k=P, v=P, g=P, beta=P, decay=0, bound=0.95, init=None, out=P, fin=None, B=1,
             H=2, T=100, dk=128, dv=128, chunk=64, dtype=1, ws=P, wsb=1 << 40, sv=P,
             svb=1 << 40, stream=None)
    a.update(kw)
    f = lib.gdr_chunk_fwd_train
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_float] + \
        [ctypes.c_void_p] * 3 + [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_size_t] * 2 + \
        [ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f(*(a[n] for n in ("q", "k", "v", "g", "beta", "decay", "bound", "init", "out", "fin",
                              "B", "H", "T", "dk", "dv", "chunk", "dtype", "ws", "wsb", "sv",
                              "svb", "stream")))


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), 1), (dict(decay=5), 1), (dict(bound=0.0), 1),
    (dict(dtype=0), 2), (dict(dk=64), 2), (dict(chunk=32), 2),   # not the two-kernel shape
    (dict(bound=0.001), 3),                                      # 16 * -ln(0.001) > 80
    (dict(ws=None), 1), (dict(wsb=1024), 1), (dict(ws=ctypes.c_void_p(0x1008)), 1),
    (dict(sv=None), 1), (dict(svb=1024), 1), (dict(sv=ctypes.c_void_p(0x1004)), 1),
    (dict(q=None), 1), (dict(out=None), 1),
    (dict(B=0), 0),                                              # no heads: nothing to do
])
def test_chunk_fwd_train_rejects(lib, kw, code):
    assert train(lib, **kw) == code


def bwd_saved(lib, **kw):
    a = dict(q=P, k=P, v=P, g=P, beta=P, decay=0, bound=0.95, init=None, dout=P, dfin=None,
             dq=P, dk_=P, dv_=P, dg=P, db=P, dinit=None, B=1, H=2, T=100, dk=128, dv=128,
             chunk=64, dtype=1, sv=P, svb=1 << 40, ws=P, wsb=1 << 40, stream=None)
    a.update(kw)
    f = lib.gdr_chunk_bwd_saved
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_float] + \
        [ctypes.c_void_p] * 9 + [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_size_t] * 2 + \
        [ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f(*(a[n] for n in ("q", "k", "v", "g", "beta", "decay", "bound", "init", "dout",
                              "dfin", "dq", "dk_", "dv_", "dg", "db", "dinit", "B", "H", "T",
                              "dk", "dv", "chunk", "dtype", "sv", "svb", "ws", "wsb", "stream")))


@pytest.mark.parametrize("kw,code", [
    (dict(decay=5), 1), (dict(bound=0.0), 1),
    (dict(dtype=0), 2), (dict(dv=64), 2), (dict(chunk=16), 2),
    (dict(bound=0.2), 3),                                        # 64 * -ln(0.2) > 80
    (dict(sv=None), 1), (dict(svb=1024), 1), (dict(sv=ctypes.c_void_p(0x1008)), 1),
    (dict(ws=None), 1), (dict(wsb=1024), 1),
    (dict(dq=ctypes.c_void_p(0x1002)), 1), (dict(dv_=ctypes.c_void_p(0x1008)), 1),
    (dict(q=None), 1), (dict(dout=None), 1), (dict(dg=None), 1),
    (dict(B=0), 0),
])
def test_chunk_bwd_saved_rejects(lib, kw, code):
    assert bwd_saved(lib, **kw) == code
