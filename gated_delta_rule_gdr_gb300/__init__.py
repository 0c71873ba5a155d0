"""GB300 gated delta rule: thin Python binding over libgdr.so (include/gdr.h).

Argument marshalling only -- every step of the computation runs in the CUDA
kernels behind the C ABI.  Tensors are torch CUDA tensors, contiguous, in the
layouts of the header; the current torch stream is passed as the stream.  If
the library is missing or fails to load, every call raises: there is no CPU
or PyTorch fallback.

    out, final = chunk_fwd(q, k, v, g, beta, a_min, init_state=None, chunk=64)
    out        = decode_step(q, k, v, g, beta, a_min, state)   # state in place

chunk_fwd and chunk_fwd_varlen take the two-kernel path (a parallel chunk
preparation into a workspace, then the state chain) when it applies, with the
workspace from torch's caching allocator; workspace=None selects the
single-launch path, a uint8 CUDA tensor supplies the workspace.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

from . import build as _build

__all__ = ["GdrError", "load", "chunk_fwd", "decode_step", "chunk_decay", "chunk_wy",
           "chunk_state", "chunk_output", "chunk_fwd_kernels", "chunk_fwd_path", "chunk_fwd_varlen",
           "chunk_fwd_workspace_size", "chunk_fwd_varlen_workspace_size", "last_device_error",
           "status_string", "version", "library_path", "STATUS", "PATHS", "OPTIONS",
           "set_option", "get_option", "option", "mla_decode", "mla_decode_workspace_size",
           "chunk_bwd", "chunk_bwd_workspace_size", "chunk_saved_size", "chunk_fwd_train",
           "chunk_bwd_saved"]

DECAY = {"affine": 0, "log": 1}   # gdr_decay_t
STATUS = {0: "GDR_OK", 1: "GDR_ERR_INVALID_ARG", 2: "GDR_ERR_UNSUPPORTED", 3: "GDR_ERR_RANGE",
          4: "GDR_ERR_CUDA", 5: "GDR_ERR_TIMEOUT"}
DTYPE = {torch.float32: 0, torch.bfloat16: 1}
# gdr_option_t
OPTIONS = {"wait_limit_ns": 0, "fused_variant": 1, "chain_split": 2, "segments": 3,
           "bwd_variant": 4}

_lib = None


class GdrError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        msg = status_string(code) if _lib is not None else self.name
        super().__init__(f"{where}: {self.name} ({msg})")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libgdr.so (optionally building it first).  Raises if unavailable."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libgdr.so not built ({path}); run __graft_entry__.build() or "
                               "python -m gated_delta_rule_gdr_gb300.build")
        _build.build()
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "gdr_chunk_fwd": [vp, vp, vp, vp, vp, f, vp, vp, vp, i, i, i, i, i, i, i, vp],
        "gdr_chunk_fwd_ws": [vp, vp, vp, vp, vp, f, vp, vp, vp, i, i, i, i, i, i, i, vp, sz, vp],
        "gdr_chunk_fwd_varlen_ws": [vp, vp, vp, vp, vp, f, vp, vp, vp, vp, i, i, i, i, i, i, i, vp,
                                    sz, vp],
        "gdr_chunk_fwd_ws_path": [i, i, i, i, i, i, f, i],
        "gdr_chunk_fwd_ex": [vp, vp, vp, vp, vp, i, f, vp, vp, vp, i, i, i, i, i, i, i, vp, sz, vp],
        "gdr_decode_step_ex": [vp, vp, vp, vp, vp, i, f, vp, vp, i, i, i, i, i, vp],
        "gdr_chunk_fwd_host": [vp, vp, vp, vp, vp, f, vp, vp, vp, i, i, i, i, i, i, i, vp, sz, vp],
        "gdr_chunk_bwd": [vp, vp, vp, vp, vp, i, f, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                          i, i, i, i, i, i, i, vp, sz, vp],
        "gdr_chunk_fwd_train": [vp, vp, vp, vp, vp, i, f, vp, vp, vp, i, i, i, i, i, i, i, vp, sz,
                                vp, sz, vp],
        "gdr_chunk_bwd_saved": [vp, vp, vp, vp, vp, i, f, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                i, i, i, i, i, i, i, vp, sz, vp, sz, vp],
        "gdr_chunk_fwd_varlen": [vp, vp, vp, vp, vp, f, vp, vp, vp, vp, i, i, i, i, i, i, i, vp],
        "gdr_chunk_fwd_static": [vp, vp, vp, vp, vp, f, vp, vp, vp, i, i, i, i, i, i, i, vp],
        "gdr_decode_step": [vp, vp, vp, vp, vp, f, vp, vp, i, i, i, i, i, vp],
        "gdr_chunk_decay": [vp, f, vp, i, i, i, vp],
        "gdr_chunk_wy": [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp],
        "gdr_chunk_state": [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp],
        "gdr_chunk_output": [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp],
        "gdr_last_device_error": [vp],
        "gdr_chunk_fwd_kernels": [i, i, i, i, i, i, f, i],
        "gdr_chunk_fwd_path": [i, i, i, i, i, i, f, i],
        "gdr_status_string": [i],
        "gdr_version": [],
        "gdr_set_option": [i, ctypes.c_int64],
        "gdr_mla_decode": [vp, vp, vp, vp, vp, f, vp, i, i, i, i, i, vp, sz, vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    for name in ("gdr_chunk_fwd_workspace_size", "gdr_chunk_fwd_varlen_workspace_size",
                 "gdr_chunk_bwd_workspace_size", "gdr_chunk_fwd_host_buffer_size",
                 "gdr_chunk_saved_size"):
        fn = getattr(lib, name)
        fn.argtypes = [i, i, i, i, i, i, i]
        fn.restype = sz
    lib.gdr_mla_decode_workspace_size.argtypes = [i, i, i, i, i]
    lib.gdr_mla_decode_workspace_size.restype = sz
    lib.gdr_get_option.argtypes = [i]
    lib.gdr_get_option.restype = ctypes.c_int64
    lib.gdr_status_string.restype = ctypes.c_char_p
    lib.gdr_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().gdr_status_string(int(code)).decode()


def version() -> str:
    return load().gdr_version().decode()


def set_option(name: str, value: int) -> None:
    """Set a process-wide option of the library (gdr_set_option): "wait_limit_ns"
    (0 = every device-side wait gives up at once), "fused_variant" (0 auto, 1 one CTA
    per head, 2 cluster pair), "chain_split" (0 auto, 1, 2), "segments" (0 auto, else
    the sequence segments of the two-kernel path)."""
    _check(load().gdr_set_option(OPTIONS[name], int(value)), "gdr_set_option")


def get_option(name: str) -> int:
    return int(load().gdr_get_option(OPTIONS[name]))


@contextlib.contextmanager
def option(**values):
    """Set options for the duration of a with-block, then restore them."""
    old = {n: get_option(n) for n in values}
    try:
        for n, val in values.items():
            set_option(n, val)
        yield
    finally:
        for n, val in old.items():
            set_option(n, val)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libgdr takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libgdr takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(code: int, where: str):
    if code != 0:
        raise GdrError(code, where)


def _f32(t, name):
    if t is not None and t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")
    return t


def _workspace(nbytes: int, workspace, device):
    """The workspace to pass: None for the single-launch path, else a uint8 CUDA
    tensor of at least nbytes ("auto": from torch's caching allocator)."""
    if workspace is None or nbytes == 0:
        return None
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError('workspace must be "auto", None or a uint8 CUDA tensor')
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace.dtype != torch.uint8 or workspace.numel() < nbytes:
        raise ValueError(f"workspace must be a uint8 tensor of at least {nbytes} bytes")
    return workspace


def chunk_fwd_workspace_size(B, H, T, dk, dv, chunk=64, dtype=torch.bfloat16) -> int:
    """Bytes of workspace the two-kernel path needs (0 where it does not apply)."""
    return int(load().gdr_chunk_fwd_workspace_size(B, H, T, dk, dv, chunk, DTYPE[dtype]))


def chunk_fwd_varlen_workspace_size(S, H, total_T, dk, dv, chunk=64, dtype=torch.bfloat16) -> int:
    """Bytes of workspace the packed two-kernel path needs (0 where it does not apply)."""
    return int(load().gdr_chunk_fwd_varlen_workspace_size(S, H, total_T, dk, dv, chunk, DTYPE[dtype]))


def chunk_fwd(q, k, v, g, beta, a_min: float, init_state=None, *, chunk: int = 64,
              out=None, final_state=None, want_final: bool = True, workspace="auto",
              decay: str = "affine"):
    """Chunked prefill.  q,k [B,H,T,dk], v [B,H,T,dv] (fp32 or bf16), g,beta [B,H,T]
    fp32, init_state [B,H,dk,dv] fp32 or None.  Returns (out, final_state).
    decay "log": a_min is the log-domain floor g_min <= 0, log alpha = g_min sigmoid(g)."""
    lib = load()
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if q.dtype not in DTYPE or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype, float32 or bfloat16")
    _f32(g, "g"), _f32(beta, "beta"), _f32(init_state, "init_state")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    if final_state is None and want_final:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    ws = _workspace(chunk_fwd_workspace_size(B, H, T, dk, dv, chunk, q.dtype), workspace, q.device)
    if decay != "affine":
        if decay not in DECAY:
            raise ValueError(f"unknown decay {decay!r}")
        _check(lib.gdr_chunk_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), DECAY[decay],
                                    float(a_min), _ptr(init_state), _ptr(out), _ptr(final_state),
                                    B, H, T, dk, dv, int(chunk), DTYPE[q.dtype], _ptr(ws),
                                    0 if ws is None else ws.numel(), _stream(q.device)),
               "gdr_chunk_fwd_ex")
    elif ws is None:
        _check(lib.gdr_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(a_min),
                                 _ptr(init_state), _ptr(out), _ptr(final_state), B, H, T, dk, dv,
                                 int(chunk), DTYPE[q.dtype], _stream(q.device)), "gdr_chunk_fwd")
    else:
        _check(lib.gdr_chunk_fwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(a_min),
                                    _ptr(init_state), _ptr(out), _ptr(final_state), B, H, T, dk,
                                    dv, int(chunk), DTYPE[q.dtype], _ptr(ws), ws.numel(),
                                    _stream(q.device)), "gdr_chunk_fwd_ws")
    return out, final_state


def chunk_fwd_varlen(q, k, v, g, beta, a_min: float, cu_seqlens, init_state=None, *,
                     chunk: int = 64, out=None, final_state=None, want_final: bool = True,
                     workspace="auto"):
    """Chunked prefill over packed sequences.  q,k [total_T,H,dk], v [total_T,H,dv] bf16,
    g,beta [total_T,H] fp32, cu_seqlens int32 [S+1] on the device, init_state [S,H,dk,dv]
    fp32 or None.  Returns (out [total_T,H,dv], final_state [S,H,dk,dv])."""
    lib = load()
    total_T, H, dk = q.shape
    dv = v.shape[-1]
    S = cu_seqlens.numel() - 1
    if q.dtype not in DTYPE or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_contiguous():
        raise TypeError("cu_seqlens must be a contiguous int32 tensor")
    _f32(g, "g"), _f32(beta, "beta"), _f32(init_state, "init_state")
    if out is None:
        out = torch.empty((total_T, H, dv), dtype=q.dtype, device=q.device)
    if final_state is None and want_final:
        final_state = torch.empty((S, H, dk, dv), dtype=torch.float32, device=q.device)
    ws = _workspace(chunk_fwd_varlen_workspace_size(S, H, total_T, dk, dv, chunk, q.dtype),
                    workspace, q.device)
    if ws is None:
        _check(lib.gdr_chunk_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                        float(a_min), _ptr(init_state), _ptr(out),
                                        _ptr(final_state), _ptr(cu_seqlens), S, H, total_T, dk, dv,
                                        int(chunk), DTYPE[q.dtype], _stream(q.device)),
               "gdr_chunk_fwd_varlen")
    else:
        _check(lib.gdr_chunk_fwd_varlen_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                           float(a_min), _ptr(init_state), _ptr(out),
                                           _ptr(final_state), _ptr(cu_seqlens), S, H, total_T, dk,
                                           dv, int(chunk), DTYPE[q.dtype], _ptr(ws), ws.numel(),
                                           _stream(q.device)), "gdr_chunk_fwd_varlen_ws")
    return out, final_state


def chunk_fwd_host_buffer_size(B, H, T, dk, dv, chunk=64, dtype=torch.bfloat16) -> int:
    """Bytes of device memory chunk_fwd_host needs (inputs, outputs, workspace)."""
    return int(load().gdr_chunk_fwd_host_buffer_size(B, H, T, dk, dv, chunk, DTYPE[dtype]))


def _host_ptr(t):
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise ValueError("chunk_fwd_host takes contiguous CPU tensors")
    return ctypes.c_void_p(t.data_ptr())


def chunk_fwd_host(q, k, v, g, beta, a_min: float, init_state, out, final_state, device_buffer,
                   *, chunk: int = 64, stream=None):
    """Prefill from host tensors to host tensors (pinned memory for overlap): copies in,
    computes and copies out on ``stream`` (default: the current stream of the buffer's
    device).  ``device_buffer`` is a uint8 CUDA tensor of chunk_fwd_host_buffer_size
    bytes; ``out`` [B,H,T,dv] and ``final_state`` [B,H,dk,dv] (or None) are CPU tensors
    written when the stream reaches the end of the call."""
    lib = load()
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if q.dtype not in DTYPE or k.dtype != q.dtype or v.dtype != q.dtype or out.dtype != q.dtype:
        raise TypeError("q, k, v, out must share one dtype, float32 or bfloat16")
    _f32(g, "g"), _f32(beta, "beta"), _f32(init_state, "init_state"), _f32(final_state, "final_state")
    if device_buffer.dtype != torch.uint8 or not device_buffer.is_cuda:
        raise ValueError("device_buffer must be a uint8 CUDA tensor")
    st = stream if stream is not None else torch.cuda.current_stream(device_buffer.device)
    _check(lib.gdr_chunk_fwd_host(_host_ptr(q), _host_ptr(k), _host_ptr(v), _host_ptr(g),
                                  _host_ptr(beta), float(a_min), _host_ptr(init_state),
                                  _host_ptr(out), _host_ptr(final_state), B, H, T, dk, dv,
                                  int(chunk), DTYPE[q.dtype], _ptr(device_buffer),
                                  device_buffer.numel(), ctypes.c_void_p(st.cuda_stream)),
           "gdr_chunk_fwd_host")
    return out, final_state


def chunk_bwd_workspace_size(B, H, T, dk, dv, chunk=64, dtype=torch.bfloat16) -> int:
    """Bytes of workspace the backward needs (0 for empty work or unsupported shapes)."""
    return int(load().gdr_chunk_bwd_workspace_size(B, H, T, dk, dv, chunk, DTYPE[dtype]))


def chunk_bwd(q, k, v, g, beta, a_min: float, init_state, d_out, d_final=None, *,
              chunk: int = 64, want_dinit: bool = True, workspace=None, decay: str = "affine"):
    """Gradients of a loss through chunk_fwd: given d_out [B,H,T,dv] (q's dtype) and
    d_final [B,H,dk,dv] fp32 or None, returns (dq, dk, dv, dg, dbeta, dinit) for the
    forward with the same arguments (dinit None unless want_dinit).  workspace: None
    (allocated here) or a uint8 CUDA tensor of at least chunk_bwd_workspace_size bytes."""
    lib = load()
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if q.dtype not in DTYPE or k.dtype != q.dtype or v.dtype != q.dtype or d_out.dtype != q.dtype:
        raise TypeError("q, k, v, d_out must share one dtype, float32 or bfloat16")
    _f32(g, "g"), _f32(beta, "beta"), _f32(init_state, "init_state"), _f32(d_final, "d_final")
    if decay not in DECAY:
        raise ValueError(f"unknown decay {decay!r}")
    dq, dk_, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg, db = torch.empty_like(g), torch.empty_like(beta)
    dinit = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device) if want_dinit else None
    need = chunk_bwd_workspace_size(B, H, T, dk, dv, chunk, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    elif workspace.dtype != torch.uint8 or workspace.numel() < need:
        raise ValueError(f"workspace must be a uint8 tensor of at least {need} bytes")
    _check(lib.gdr_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), DECAY[decay],
                             float(a_min), _ptr(init_state), _ptr(d_out), _ptr(d_final),
                             _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg), _ptr(db), _ptr(dinit),
                             B, H, T, dk, dv, int(chunk), DTYPE[q.dtype], _ptr(workspace),
                             workspace.numel(), _stream(q.device)), "gdr_chunk_bwd")
    return dq, dk_, dv_, dg, db, dinit


def chunk_saved_size(B, H, T, dk, dv, chunk=64, dtype=torch.bfloat16) -> int:
    """Bytes of the buffer chunk_fwd_train fills for chunk_bwd_saved (0: not supported)."""
    return int(load().gdr_chunk_saved_size(B, H, T, dk, dv, chunk, DTYPE[dtype]))


def chunk_fwd_train(q, k, v, g, beta, a_min: float, init_state=None, *, chunk: int = 64,
                    out=None, final_state=None, want_final: bool = True, workspace=None,
                    saved=None, decay: str = "affine"):
    """chunk_fwd (bf16, d = 128, chunk 64, two-kernel path) that also keeps every chunk's
    state and W tile for chunk_bwd_saved.  workspace / saved: None (allocated here) or
    uint8 CUDA tensors of at least chunk_fwd_workspace_size / chunk_saved_size bytes.
    Returns (out, final_state, saved)."""
    lib = load()
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if q.dtype not in DTYPE or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    _f32(g, "g"), _f32(beta, "beta"), _f32(init_state, "init_state")
    if decay not in DECAY:
        raise ValueError(f"unknown decay {decay!r}")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    if final_state is None and want_final:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    need_ws = chunk_fwd_workspace_size(B, H, T, dk, dv, chunk, q.dtype)
    need_sv = chunk_saved_size(B, H, T, dk, dv, chunk, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need_ws, 16), dtype=torch.uint8, device=q.device)
    if saved is None:
        saved = torch.empty(max(need_sv, 16), dtype=torch.uint8, device=q.device)
    for name, t, need in (("workspace", workspace, need_ws), ("saved", saved, need_sv)):
        if t.dtype != torch.uint8 or t.numel() < need:
            raise ValueError(f"{name} must be a uint8 tensor of at least {need} bytes")
    _check(lib.gdr_chunk_fwd_train(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), DECAY[decay],
                                   float(a_min), _ptr(init_state), _ptr(out), _ptr(final_state),
                                   B, H, T, dk, dv, int(chunk), DTYPE[q.dtype], _ptr(workspace),
                                   workspace.numel(), _ptr(saved), saved.numel(),
                                   _stream(q.device)), "gdr_chunk_fwd_train")
    return out, final_state, saved


def chunk_bwd_saved(q, k, v, g, beta, a_min: float, init_state, d_out, saved, d_final=None, *,
                    chunk: int = 64, want_dinit: bool = True, workspace=None,
                    decay: str = "affine"):
    """chunk_bwd reading the states chunk_fwd_train saved (same arguments as that
    forward) instead of recomputing them.  Returns (dq, dk, dv, dg, dbeta, dinit)."""
    lib = load()
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if q.dtype not in DTYPE or k.dtype != q.dtype or v.dtype != q.dtype or d_out.dtype != q.dtype:
        raise TypeError("q, k, v, d_out must share one dtype")
    _f32(g, "g"), _f32(beta, "beta"), _f32(init_state, "init_state"), _f32(d_final, "d_final")
    if decay not in DECAY:
        raise ValueError(f"unknown decay {decay!r}")
    if saved.dtype != torch.uint8 or not saved.is_cuda:
        raise ValueError("saved must be the uint8 CUDA tensor chunk_fwd_train filled")
    dq, dk_, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg, db = torch.empty_like(g), torch.empty_like(beta)
    dinit = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device) if want_dinit else None
    need = chunk_bwd_workspace_size(B, H, T, dk, dv, chunk, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    elif workspace.dtype != torch.uint8 or workspace.numel() < need:
        raise ValueError(f"workspace must be a uint8 tensor of at least {need} bytes")
    _check(lib.gdr_chunk_bwd_saved(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), DECAY[decay],
                                   float(a_min), _ptr(init_state), _ptr(d_out), _ptr(d_final),
                                   _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg), _ptr(db),
                                   _ptr(dinit), B, H, T, dk, dv, int(chunk), DTYPE[q.dtype],
                                   _ptr(saved), saved.numel(), _ptr(workspace), workspace.numel(),
                                   _stream(q.device)), "gdr_chunk_bwd_saved")
    return dq, dk_, dv_, dg, db, dinit


def decode_step(q, k, v, g, beta, a_min: float, state, *, out=None, decay: str = "affine"):
    """One token for N sequences.  q,k [N,H,dk], v [N,H,dv], g,beta [N,H] fp32,
    state [N,H,dk,dv] fp32 updated in place.  Returns out [N,H,dv]."""
    lib = load()
    N, H, dk = q.shape
    dv = v.shape[-1]
    if q.dtype not in DTYPE or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype, float32 or bfloat16")
    _f32(g, "g"), _f32(beta, "beta"), _f32(state, "state")
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    if decay != "affine":
        if decay not in DECAY:
            raise ValueError(f"unknown decay {decay!r}")
        _check(lib.gdr_decode_step_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), DECAY[decay],
                                      float(a_min), _ptr(state), _ptr(out), N, H, dk, dv,
                                      DTYPE[q.dtype], _stream(q.device)), "gdr_decode_step_ex")
        return out
    _check(lib.gdr_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(a_min),
                               _ptr(state), _ptr(out), N, H, dk, dv, DTYPE[q.dtype],
                               _stream(q.device)), "gdr_decode_step")
    return out


def chunk_decay(g, a_min: float, chunk: int = 64, *, gamma=None):
    """gamma [BH,T] = chunk-local cumulative product of alpha.  g [..., T] fp32."""
    lib = load()
    T = g.shape[-1]
    BH = g.numel() // max(T, 1) if T else 0
    _f32(g, "g")
    if gamma is None:
        gamma = torch.empty_like(g)
    _check(lib.gdr_chunk_decay(_ptr(g), float(a_min), _ptr(gamma), BH, T, int(chunk),
                               _stream(g.device)), "gdr_chunk_decay")
    return gamma


def chunk_wy(k, v, beta, gamma, chunk: int = 64):
    """U [BH,T,dv], Wk [BH,T,dk] (fp32) of the intra-chunk WY/UT transform."""
    lib = load()
    *lead, T, dk = k.shape
    dv = v.shape[-1]
    BH = k.numel() // max(T * dk, 1)
    U = torch.empty((*lead, T, dv), dtype=torch.float32, device=k.device)
    Wk = torch.empty((*lead, T, dk), dtype=torch.float32, device=k.device)
    _check(lib.gdr_chunk_wy(_ptr(k), _ptr(v), _ptr(beta), _ptr(gamma), _ptr(U), _ptr(Wk), BH, T,
                            dk, dv, int(chunk), DTYPE[k.dtype], _stream(k.device)),
           "gdr_chunk_wy")
    return U, Wk


def chunk_state(k, gamma, U, Wk, init_state=None, chunk: int = 64, want_mn: bool = True):
    """W [BH,T,dv], Mn [BH,NC,dk,dv] (or None), final [BH,dk,dv] of the state pass."""
    lib = load()
    *lead, T, dk = k.shape
    dv = U.shape[-1]
    BH = k.numel() // max(T * dk, 1)
    NC = (T + chunk - 1) // chunk
    W = torch.empty_like(U)
    Mn = (torch.empty((*lead, NC, dk, dv), dtype=torch.float32, device=k.device)
          if want_mn else None)
    fin = torch.empty((*lead, dk, dv), dtype=torch.float32, device=k.device)
    _check(lib.gdr_chunk_state(_ptr(k), _ptr(gamma), _ptr(U), _ptr(Wk), _ptr(init_state),
                               _ptr(W), _ptr(Mn), _ptr(fin), BH, T, dk, dv, int(chunk),
                               DTYPE[k.dtype], _stream(k.device)), "gdr_chunk_state")
    return W, Mn, fin


def chunk_output(q, k, gamma, Mn, W, chunk: int = 64):
    """out [BH,T,dv] in q's dtype from the per-chunk states and W."""
    lib = load()
    *lead, T, dk = q.shape
    dv = W.shape[-1]
    BH = q.numel() // max(T * dk, 1)
    out = torch.empty((*lead, T, dv), dtype=q.dtype, device=q.device)
    _check(lib.gdr_chunk_output(_ptr(q), _ptr(k), _ptr(gamma), _ptr(Mn), _ptr(W), _ptr(out), BH,
                                T, dk, dv, int(chunk), DTYPE[q.dtype], _stream(q.device)),
           "gdr_chunk_output")
    return out


def chunk_fwd_kernels(B, H, T, dk, dv, chunk=64, a_min=0.95, dtype=torch.bfloat16) -> int:
    """How many kernels one chunk_fwd call with these arguments launches."""
    return int(load().gdr_chunk_fwd_kernels(B, H, T, dk, dv, chunk, float(a_min), DTYPE[dtype]))


PATHS = {0: "none", 1: "staged (on the workspace)", 2: "fused one CTA per head",
         3: "fused two-CTA cluster per head", 4: "prep + chain, two CTAs per head",
         5: "prep + chain, one CTA per head", 6: "one-pass CUDA-core kernel",
         7: "prep + segment maps + scan + chain over sequence segments"}


def chunk_fwd_path(B, H, T, dk, dv, chunk=64, a_min=0.95, dtype=torch.bfloat16,
                   workspace: bool = True) -> int:
    """Which path one chunk_fwd call with these arguments takes on the current
    device (see PATHS; -1 = rejected); workspace=False: the single-launch path."""
    fn = load().gdr_chunk_fwd_ws_path if workspace else load().gdr_chunk_fwd_path
    return int(fn(B, H, T, dk, dv, chunk, float(a_min), DTYPE[dtype]))


def mla_decode_workspace_size(N, H, Lmax, dc=512, dh=128) -> int:
    """Bytes of workspace one latent-attention decode step needs (0 if unsupported)."""
    return int(load().gdr_mla_decode_workspace_size(N, H, Lmax, dc, dh))


def mla_decode(q_abs, ckv, seqlens, w_uv, gate, scale: float, *, out=None, workspace=None):
    """One decode step of gated multi-head latent attention.  q_abs [N,H,dc] bf16 (the
    query with the key up-projection absorbed), ckv [N,Lmax,dc] bf16 (latent cache),
    seqlens [N] int32 on the device, w_uv [H,dh,dc] bf16, gate [N,H,dh] fp32 (the gate's
    pre-activation).  Returns out [N,H,dh] bf16.  workspace: None (from torch's caching
    allocator) or a uint8 CUDA tensor of at least mla_decode_workspace_size bytes."""
    lib = load()
    N, H, dc = q_abs.shape
    Lmax = ckv.shape[1]
    dh = w_uv.shape[1]
    for t, name in ((q_abs, "q_abs"), (ckv, "ckv"), (w_uv, "w_uv")):
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16")
    _f32(gate, "gate")
    if seqlens.dtype != torch.int32:
        raise TypeError("seqlens must be int32")
    if out is None:
        out = torch.empty((N, H, dh), dtype=torch.bfloat16, device=q_abs.device)
    need = mla_decode_workspace_size(N, H, Lmax, dc, dh)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_abs.device)
    elif workspace.dtype != torch.uint8 or workspace.numel() < need:
        raise ValueError(f"workspace must be a uint8 tensor of at least {need} bytes")
    _check(lib.gdr_mla_decode(_ptr(q_abs), _ptr(ckv), _ptr(seqlens), _ptr(w_uv), _ptr(gate),
                              float(scale), _ptr(out), N, H, Lmax, dc, dh, _ptr(workspace),
                              workspace.numel(), _stream(q_abs.device)), "gdr_mla_decode")
    return out


def last_device_error(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device error word
    as a status code (0 = ok, 5 = a bounded wait timed out)."""
    lib = load()
    return int(lib.gdr_last_device_error(_stream(device)))
