"""fp64 CPU oracle for the gated delta rule with a lower-bounded decay.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It never imports the CUDA library package and shares no code with
it; the two meet only in the seeded input generator, which holds none of the
method's arithmetic.

Contents
--------
* ``fwd``      -- the token-by-token recurrence (C, fp64, ``gdr_oracle.c``):
                  alpha_t = a_min + (1 - a_min) sigmoid(g_t),
                  S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
                  o_t = S_t q_t.
* ``decode``   -- one step of the same recurrence, in place on the state.
* ``bwd``      -- the gradients of L = <d_out, out> + <d_final, final_state> with
                  respect to q, k, v, g, beta and the initial state: reverse-mode
                  differentiation of the token loop as written (C, fp64).
* ``alpha``    -- the lower-bounded decay itself: the linear-domain floor a_min, or
                  (decay="log") the pages' log-domain form alpha = exp(g_min sigmoid(g)).
* ``chunkwise`` (module) -- the chunked reformulation in numpy fp64, used to
                  check the token loop and to export per-stage intermediates.
* ``mla_decode`` -- one decode step of gated multi-head latent attention (C, fp64,
                  ``mla_oracle.c``): softmax attention of the absorbed query over the
                  latent cache, the value up-projection, the sigmoid output gate.

Every function is pinned by ``tests/test_oracle_pins.py`` (see the module
docstrings there for which mathematical fact pins which part).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgdr_oracle.so")
_lib = None
_lock = threading.Lock()
_MLA_SRC = os.path.join(_HERE, "mla_oracle.c")
_MLA_LIB_PATH = os.path.join(_HERE, "libmla_oracle.so")
_mla_lib = None


def _compile(src: str, out: str, force: bool) -> str:
    if (not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``gdr_oracle.c`` and ``mla_oracle.c`` with the host C compiler (fp64, no
    fast-math); returns the path of the recurrence's library."""
    _compile(_MLA_SRC, _MLA_LIB_PATH, force)
    return _compile(_SRC, _LIB_PATH, force)


def _load_mla():
    global _mla_lib
    with _lock:
        if _mla_lib is None:
            build()
            lib = ctypes.CDLL(_MLA_LIB_PATH)
            set_mla_signature(lib)
            _mla_lib = lib
    return _mla_lib


def set_mla_signature(lib):
    f32p = ctypes.POINTER(ctypes.c_float)
    lib.gdr_oracle_mla_decode.restype = ctypes.c_int
    lib.gdr_oracle_mla_decode.argtypes = [f32p, f32p, ctypes.POINTER(ctypes.c_int), f32p, f32p,
                                          ctypes.c_double, ctypes.POINTER(ctypes.c_double)] + \
        [ctypes.c_int] * 6


def mla_decode(q_abs, ckv, seqlens, w_uv, gate, scale: float, *, nthreads: int | None = None):
    """One decode step of gated multi-head latent attention, fp64.  q_abs [N,H,dc] (the
    query with the key up-projection absorbed), ckv [N,Lmax,dc] (latent cache),
    seqlens [N] (cache rows in use), w_uv [H,dh,dc], gate [N,H,dh] (the gate's
    pre-activation).  Returns out [N,H,dh] fp64:
    out[n,h] = sigmoid(gate[n,h]) * (w_uv[h] @ sum_t softmax_t(scale q_abs[n,h].ckv[n,t]) ckv[n,t])."""
    qa, c, w, z = (_f32(x) for x in (q_abs, ckv, w_uv, gate))
    N, H, dc = qa.shape
    Lmax = c.shape[1]
    dh = w.shape[1]
    if c.shape != (N, Lmax, dc) or w.shape != (H, dh, dc) or z.shape != (N, H, dh):
        raise ValueError("mla_decode shape mismatch")
    if hasattr(seqlens, "detach"):
        seqlens = seqlens.detach().cpu().numpy()
    lens = np.ascontiguousarray(np.asarray(seqlens), dtype=np.int32)
    if lens.shape != (N,):
        raise ValueError("seqlens must have N entries")
    out = np.empty((N, H, dh), np.float64)
    rc = _load_mla().gdr_oracle_mla_decode(
        _ptr(qa, ctypes.c_float), _ptr(c, ctypes.c_float), _ptr(lens, ctypes.c_int),
        _ptr(w, ctypes.c_float), _ptr(z, ctypes.c_float), float(scale), _ptr(out, ctypes.c_double),
        N, H, Lmax, dc, dh, int(nthreads or os.cpu_count() or 1))
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_mla_decode failed with code {rc}")
    return out


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            lib.gdr_oracle_alpha.restype = ctypes.c_double
            lib.gdr_oracle_alpha.argtypes = [ctypes.c_double, ctypes.c_double]
            lib.gdr_oracle_alpha_log.restype = ctypes.c_double
            lib.gdr_oracle_alpha_log.argtypes = [ctypes.c_double, ctypes.c_double]
            lib.gdr_oracle_fwd.restype = ctypes.c_int
            lib.gdr_oracle_fwd.argtypes = [f32p, f32p, f32p, f32p, f32p, ctypes.c_double,
                                           f32p, f64p, f64p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int]
            lib.gdr_oracle_bwd.restype = ctypes.c_int
            lib.gdr_oracle_bwd.argtypes = [f32p] * 5 + [ctypes.c_double] + [f32p] * 3 + \
                [f64p] * 6 + [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                              ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.gdr_oracle_decode.restype = ctypes.c_int
            lib.gdr_oracle_decode.argtypes = [f32p, f32p, f32p, f32p, f32p, ctypes.c_double,
                                              f64p, f64p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int]
            _lib = lib
    return _lib


def _f32(x) -> np.ndarray:
    """Widen to a contiguous float32 numpy array.

    Accepts numpy arrays or CPU torch tensors of bf16/fp32 (bf16 -> fp32 is
    exact).  Values are never rounded: fp64 input is refused.
    """
    if hasattr(x, "detach"):          # a torch tensor
        import torch
        t = x.detach()
        if t.dtype not in (torch.float32, torch.bfloat16, torch.float16):
            raise TypeError(f"oracle input dtype {t.dtype} is not a 16/32-bit float")
        x = t.to("cpu", torch.float32).contiguous().numpy()
    a = np.asarray(x)
    if a.dtype == np.float64:
        raise TypeError("oracle inputs are the kernel's fp32/bf16 values; got float64")
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


DECAY = {"affine": 0, "log": 1}


def alpha(g, a_min: float, decay: str = "affine"):
    """The lower-bounded decay, elementwise, fp64: decay "affine":
    alpha = a_min + (1 - a_min) sigmoid(g); decay "log": alpha = exp(g_min sigmoid(g))
    with g_min = the bound."""
    lib = _load()
    g = np.asarray(g, dtype=np.float64)
    fn = lib.gdr_oracle_alpha_log if decay == "log" else lib.gdr_oracle_alpha
    if decay not in DECAY:
        raise ValueError(f"unknown decay {decay!r}")
    return np.vectorize(lambda x: fn(float(x), float(a_min)), otypes=[np.float64])(g)


def fwd(q, k, v, g, beta, a_min: float, init_state=None, *, want_out: bool = True,
        want_final: bool = True, nthreads: int | None = None, decay: str = "affine"):
    """Token-by-token forward.  Shapes: q,k [B,H,T,dk], v [B,H,T,dv], g,beta [B,H,T],
    init_state [B,H,dk,dv] or None (zeros).  Returns (out [B,H,T,dv] fp64 or None,
    final_state [B,H,dk,dv] fp64 or None).  decay "log": a_min is g_min and
    alpha = exp(g_min sigmoid(g)).
    """
    q, k, v, g, beta = (_f32(x) for x in (q, k, v, g, beta))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if k.shape != (B, H, T, dk) or v.shape != (B, H, T, dv):
        raise ValueError("q/k/v shape mismatch")
    if g.shape != (B, H, T) or beta.shape != (B, H, T):
        raise ValueError("g/beta shape mismatch")
    init = None if init_state is None else _f32(init_state)
    if init is not None and init.shape != (B, H, dk, dv):
        raise ValueError("init_state shape mismatch")
    out = np.empty((B, H, T, dv), np.float64) if want_out else None
    fin = np.empty((B, H, dk, dv), np.float64) if want_final else None
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    lib = _load()
    f32, f64 = ctypes.c_float, ctypes.c_double
    rc = lib.gdr_oracle_fwd(_ptr(q, f32), _ptr(k, f32), _ptr(v, f32), _ptr(g, f32),
                            _ptr(beta, f32), float(a_min),
                            None if init is None else _ptr(init, f32),
                            None if out is None else _ptr(out, f64),
                            None if fin is None else _ptr(fin, f64),
                            B, H, T, dk, dv, int(nthreads), DECAY[decay])
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_fwd failed with code {rc}")
    return out, fin


def decode(q, k, v, g, beta, a_min: float, state: np.ndarray, *, nthreads: int | None = None,
           decay: str = "affine"):
    """One decode step in place on ``state`` ([N,H,dk,dv] float64).  q,k [N,H,dk],
    v [N,H,dv], g,beta [N,H].  Returns out [N,H,dv] fp64."""
    q, k, v, g, beta = (_f32(x) for x in (q, k, v, g, beta))
    N, H, dk = q.shape
    dv = v.shape[-1]
    if state.dtype != np.float64 or not state.flags["C_CONTIGUOUS"] \
            or state.shape != (N, H, dk, dv):
        raise ValueError("state must be a contiguous float64 [N,H,dk,dv] array")
    out = np.empty((N, H, dv), np.float64)
    lib = _load()
    f32, f64 = ctypes.c_float, ctypes.c_double
    rc = lib.gdr_oracle_decode(_ptr(q, f32), _ptr(k, f32), _ptr(v, f32), _ptr(g, f32),
                               _ptr(beta, f32), float(a_min), _ptr(state, f64),
                               _ptr(out, f64), N, H, dk, dv,
                               int(nthreads or os.cpu_count() or 1), DECAY[decay])
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_decode failed with code {rc}")
    return out


def bwd(q, k, v, g, beta, a_min: float, init_state=None, d_out=None, d_final=None, *,
        nthreads: int | None = None, decay: str = "affine"):
    """Gradients of L = sum <d_out, out> + <d_final, final_state> for the forward of
    ``fwd`` with the same arguments.  d_out [B,H,T,dv] and d_final [B,H,dk,dv] may be
    None (zero).  Returns (dq, dk, dv, dg, dbeta, dinit), fp64, shaped like q, k, v, g,
    beta and the initial state."""
    q, k, v, g, beta = (_f32(x) for x in (q, k, v, g, beta))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if k.shape != (B, H, T, dk) or v.shape != (B, H, T, dv):
        raise ValueError("q/k/v shape mismatch")
    if g.shape != (B, H, T) or beta.shape != (B, H, T):
        raise ValueError("g/beta shape mismatch")
    init = None if init_state is None else _f32(init_state)
    dout = None if d_out is None else _f32(d_out)
    dfin = None if d_final is None else _f32(d_final)
    if init is not None and init.shape != (B, H, dk, dv):
        raise ValueError("init_state shape mismatch")
    if dout is not None and dout.shape != (B, H, T, dv):
        raise ValueError("d_out shape mismatch")
    if dfin is not None and dfin.shape != (B, H, dk, dv):
        raise ValueError("d_final shape mismatch")
    gq = np.empty((B, H, T, dk), np.float64)
    gk = np.empty((B, H, T, dk), np.float64)
    gv = np.empty((B, H, T, dv), np.float64)
    gg = np.empty((B, H, T), np.float64)
    gb = np.empty((B, H, T), np.float64)
    gi = np.empty((B, H, dk, dv), np.float64)
    lib = _load()
    f32, f64 = ctypes.c_float, ctypes.c_double
    opt = lambda a: None if a is None else _ptr(a, f32)
    rc = lib.gdr_oracle_bwd(_ptr(q, f32), _ptr(k, f32), _ptr(v, f32), _ptr(g, f32),
                            _ptr(beta, f32), float(a_min), opt(init), opt(dout), opt(dfin),
                            _ptr(gq, f64), _ptr(gk, f64), _ptr(gv, f64), _ptr(gg, f64),
                            _ptr(gb, f64), _ptr(gi, f64), B, H, T, dk, dv,
                            int(nthreads or os.cpu_count() or 1), DECAY[decay])
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_bwd failed with code {rc}")
    return gq, gk, gv, gg, gb, gi


def rel_l2(x, ref) -> float:
    """||x - ref||_2 / ||ref||_2 over the whole tensor, in fp64."""
    x = np.asarray(_f64(x), np.float64)
    ref = np.asarray(_f64(ref), np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((x - ref).ravel())
    if den == 0.0:
        return float(num)
    return float(num / den)


def _f64(x):
    if hasattr(x, "detach"):
        import torch
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, np.float64)
