"""gdr_chunk_fwd_static: prefill for callers that cannot allocate device memory
(for example a plugin whose host framework owns all device memory, or a
deployment that forbids allocation after start-up).  It must give the same
results as gdr_chunk_fwd, call after call, on its fixed library-owned scratch,
and refuse work that does not fit that scratch."""
from __future__ import annotations

import ctypes

import pytest
import torch

import oracle
import gated_delta_rule_gdr_gb300 as gdr
from gated_delta_rule_gdr_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 5e-3}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = gdr.load(build_if_missing=True)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.gdr_chunk_fwd_static.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp, i, i, i, i, i, i, i,
                                         vp]
    lib.gdr_chunk_fwd_static.restype = ctypes.c_int
    return lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def static_fwd(lib, x, w, out, fin):
    return lib.gdr_chunk_fwd_static(
        _p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["g"]), _p(x["beta"]), float(w.a_min),
        _p(x["init_state"]), _p(out), _p(fin), w.B, w.H, w.T, w.dk, w.dv, w.chunk,
        0 if w.dtype == "f32" else 1, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype,d,T,C", [("f32", 64, 256, 64), ("bf16", 64, 200, 32),
                                         ("f32", 128, 130, 16)])
def test_static_scratch_matches_chunk_fwd(lib, dtype, d, T, C):
    w = I.CORRECTNESS.with_(B=1, H=2, T=T, dk=d, dv=d, chunk=C, dtype=dtype, init_std=0.02)
    x = {n: (None if t is None else t.cuda()) for n, t in I.prefill_inputs(w).items()}
    ref_out, ref_fin = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min,
                                     x["init_state"], chunk=C)
    torch.cuda.synchronize()
    for _ in range(2):      # two calls in a row on the shared scratch
        out = torch.full_like(ref_out, float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        assert static_fwd(lib, x, w, out, fin) == 0
        torch.cuda.synchronize()
        assert oracle.rel_l2(out, ref_out) <= TOL[dtype]
        assert oracle.rel_l2(fin, ref_fin) <= TOL[dtype]
    assert gdr.last_device_error() == 0


def test_static_scratch_refuses_oversized_work(lib):
    w = I.PREFILL            # B4 H16 T4096 d128: far beyond 32 MiB of intermediates
    z = torch.empty(1, device="cuda")
    x = dict(q=z, k=z, v=z, g=z, beta=z, init_state=None)
    assert static_fwd(lib, x, w, z, None) == 2          # GDR_ERR_UNSUPPORTED
