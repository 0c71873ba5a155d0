"""gdr_chunk_fwd_static: prefill for callers that cannot allocate device memory
(for example a plugin whose host framework owns all device memory, or a
deployment that forbids allocation after start-up).  It must give the oracle's
results, the same as gdr_chunk_fwd, call after call on its fixed library-owned
scratch; refuse work that does not fit that scratch; and copy the initial state
for empty sequences."""
from __future__ import annotations

import ctypes

import pytest
import torch

import oracle
import gated_delta_rule_gdr_gb300 as gdr
from gated_delta_rule_gdr_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 5e-3}
LIMIT = 32 << 20     # bytes of the library's scratch array


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return gdr.load(build_if_missing=True)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def static_fwd(lib, x, w, out, fin):
    return lib.gdr_chunk_fwd_static(
        _p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["g"]), _p(x["beta"]), float(w.a_min),
        _p(x["init_state"]), _p(out), _p(fin), w.B, w.H, w.T, w.dk, w.dv, w.chunk,
        0 if w.dtype == "f32" else 1, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def scratch_bytes(w):
    nc = (w.T + w.chunk - 1) // w.chunk
    bh = w.B * w.H
    return 4 * (bh * w.T * (1 + w.dk + 2 * w.dv) + bh * nc * w.dk * w.dv)


@pytest.mark.parametrize("dtype,d,T,C", [("f32", 64, 256, 64), ("bf16", 64, 200, 32),
                                         ("f32", 128, 130, 16), ("f32", 64, 16320, 64)])
def test_static_scratch_matches_oracle_and_chunk_fwd(lib, dtype, d, T, C):
    w = I.CORRECTNESS.with_(B=1, H=2, T=T, dk=d, dv=d, chunk=C, dtype=dtype, init_std=0.02)
    assert scratch_bytes(w) <= LIMIT
    x = {n: (None if t is None else t.cuda()) for n, t in I.prefill_inputs(w).items()}
    ref_out, ref_fin = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min,
                                     x["init_state"], chunk=C)
    cpu = {n: t.cpu() for n, t in x.items()}
    ro, rf = oracle.fwd(cpu["q"], cpu["k"], cpu["v"], cpu["g"], cpu["beta"], w.a_min,
                        cpu["init_state"])
    torch.cuda.synchronize()
    for _ in range(2):      # two calls in a row on the shared scratch
        out = torch.full_like(ref_out, float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        assert static_fwd(lib, x, w, out, fin) == 0
        torch.cuda.synchronize()
        assert oracle.rel_l2(out, ro) <= TOL[dtype]
        assert oracle.rel_l2(fin, rf) <= TOL[dtype]
        assert oracle.rel_l2(out, ref_out) <= TOL[dtype]
        assert oracle.rel_l2(fin, ref_fin) <= TOL[dtype]
    assert gdr.last_device_error() == 0


def test_static_scratch_limit_boundary(lib):
    under = I.CORRECTNESS.with_(B=1, H=2, T=16320, dk=64, dv=64, chunk=64)
    over = under.with_(T=16321)
    assert scratch_bytes(under) <= LIMIT < scratch_bytes(over)
    z = torch.empty(1, device="cuda")
    x = dict(q=z, k=z, v=z, g=z, beta=z, init_state=None)
    assert static_fwd(lib, x, over, z, None) == 2           # GDR_ERR_UNSUPPORTED
    assert static_fwd(lib, x, I.PREFILL, z, None) == 2      # B4 H16 T4096 d128: ~2.3 GB
    assert gdr.last_device_error() == 0


def test_static_empty_sequence_copies_initial_state(lib):
    w = I.CORRECTNESS.with_(B=2, H=3, T=0, dk=64, dv=32, init_std=0.5)
    init = torch.randn(2, 3, 64, 32, device="cuda")
    fin = torch.full_like(init, float("nan"))
    z = torch.empty(1, device="cuda")
    x = dict(q=z, k=z, v=z, g=z, beta=z, init_state=init)
    assert static_fwd(lib, x, w, z, fin) == 0
    torch.cuda.synchronize()
    assert torch.equal(fin, init)
    x["init_state"] = None                                  # no initial state: zeros
    assert static_fwd(lib, x, w, z, fin) == 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(fin) == 0
    assert static_fwd(lib, x, w.with_(B=0), z, None) == 0   # no heads: nothing to do
