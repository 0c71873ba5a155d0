"""GPU parity of the backward (gdr_chunk_bwd, through the C ABI) against the fp64
oracle's reverse-mode gradients on the same seeded inputs and cotangents.

Tolerance (relative L2 per gradient tensor): the forward's, 1e-5 on the fp32
path (every gradient is formed in fp32; measured ~3e-7), and 5e-3 on the bf16
path.  There dq, dk, dv are rounded to bf16 (2^-9 relative per element), and the
reverse chain and the per-chunk products of the d = 128, chunk-64 shape run on
tensor cores with the fp32 intermediates (P, T, dW, dR, W, the chunk states M and
dM', the masked pair gradients) rounded to bf16 operands and fp32 accumulation
(the running dM stays fp32): dq, dk, dv and dbeta measure ~3e-3, dg ~2e-3 and the
initial state's gradient ~1.8e-3."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_gdr_gb300 as gdr
from gated_delta_rule_gdr_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 5e-3}
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dinit")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdr.load(build_if_missing=True)
    yield
    assert gdr.last_device_error() == 0


def run(w, *, init=True, final=True, bound=None, decay="affine"):
    x = I.prefill_inputs(w, device="cuda")
    ct = I.cotangents(w, device="cuda")
    bound = w.a_min if bound is None else bound
    init_state = x["init_state"] if init else None
    d_final = ct["d_final"] if final else None
    got = gdr.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], bound, init_state,
                        ct["d_out"], d_final, chunk=w.chunk, decay=decay)
    torch.cuda.synchronize()
    assert gdr.last_device_error() == 0
    cpu = lambda t: None if t is None else t.cpu()
    ref = oracle.bwd(*(cpu(x[n]) for n in ("q", "k", "v", "g", "beta")), bound, cpu(init_state),
                     cpu(ct["d_out"]), cpu(d_final), decay=decay)
    return got, ref


def check(got, ref, tol):
    errs = {}
    for n, a, b in zip(NAMES, got, ref):
        assert np.isfinite(a.float().cpu().numpy()).all(), n
        errs[n] = oracle.rel_l2(a, b)
    print(" ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    assert all(e <= tol for e in errs.values()), errs
    return errs


@pytest.mark.parametrize("T", [1, 63, 64, 200, 256])
def test_bwd_fp32_correctness_workload(T):
    """The correctness workload's shape (d = 64, chunk 64, fp32) with ragged tails."""
    w = I.CORRECTNESS.with_(T=T, init_std=0.3)
    check(*run(w), TOL["f32"])


@pytest.mark.parametrize("init,final", [(False, False), (True, False), (False, True)])
def test_bwd_optional_state_terms(init, final):
    """Zero initial state and / or no final-state cotangent."""
    w = I.CORRECTNESS.with_(T=150, init_std=0.3)
    check(*run(w, init=init, final=final), TOL["f32"])


@pytest.mark.parametrize("T", [1, 64, 65, 300])
def test_bwd_bf16_prefill_shape(T):
    """The prefill workload's head shape (bf16, d = 128, chunk 64, init N(0, 0.02))."""
    w = I.PREFILL.with_(B=1, H=2, T=T)
    check(*run(w), TOL["bf16"])


@pytest.mark.parametrize("segments", [3, 4])
def test_bwd_bf16_default_with_sequence_segments(segments):
    """The default backward recomputes through the training forward's kernels, which cut
    few heads' long sequences into segments (forced here on 2 heads of 32 chunks): the
    saved states then come from the segment chains."""
    w = I.PREFILL.with_(B=1, H=2, T=2048)
    with gdr.option(segments=segments):
        check(*run(w), TOL["bf16"])


@pytest.mark.parametrize("init,final", [(False, False), (True, False), (False, True)])
def test_bwd_bf16_prefill_shape_optional_state_terms(init, final):
    """The tensor-core kernels of the prefill shape without an initial state and / or a
    final-state cotangent."""
    w = I.PREFILL.with_(B=1, H=2, T=200)
    check(*run(w, init=init, final=final), TOL["bf16"])


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 300])
def test_bwd_bf16_per_chunk_kernels(variant, T):
    """Both per-chunk gradient kernels of the prefill shape after the backward's own
    recomputation: 1 warp-level MMAs, 2 the tensor cores (the default's per-chunk
    kernel), with ragged and single-chunk sequences, several heads (the persistent grid
    walks several tasks per CTA at B = 3, H = 64, T = 300)."""
    w = I.PREFILL.with_(B=1, H=2, T=T) if T != 300 else I.PREFILL.with_(B=3, H=64, T=300)
    with gdr.option(bwd_variant=variant):
        got, ref = run(w)
    if T == 300:   # the oracle on sampled heads: (0, 0), (1, 17), (2, 63)
        for b, h in ((0, 0), (1, 17), (2, 63)):
            check([t[b:b + 1, h:h + 1] for t in got], [t[b:b + 1, h:h + 1] for t in ref], TOL["bf16"])
    else:
        check(got, ref, TOL["bf16"])


def test_bwd_bf16_per_chunk_kernels_agree():
    """The tensor-core and warp-MMA per-chunk kernels take the same bf16 operands and
    accumulate in fp32: their gradients agree far inside the oracle tolerance (the
    bf16 outputs differ by the rounding of sums taken in another order)."""
    w = I.PREFILL.with_(B=2, H=8, T=1000)
    x = I.prefill_inputs(w, device="cuda")
    ct = I.cotangents(w, device="cuda")
    outs = []
    for variant in (1, 2):
        with gdr.option(bwd_variant=variant):
            outs.append(gdr.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min,
                                      x["init_state"], ct["d_out"], ct["d_final"]))
    torch.cuda.synchronize()
    for n, a, b in zip(NAMES, *outs):
        e = oracle.rel_l2(a, b)
        assert e <= 2e-3, (n, e)


def test_bwd_bf16_prefill_shape_log_decay():
    """The tensor-core kernels with the pages' log-domain decay (g_min = -1.25 on 64-token
    chunks, the range rule's limit)."""
    w = I.PREFILL.with_(B=1, H=2, T=200)
    check(*run(w, bound=-1.25, decay="log"), TOL["bf16"])


@pytest.mark.parametrize("dk,dv,chunk", [(64, 64, 64), (128, 64, 32)])
def test_bwd_bf16_other_shapes(dk, dv, chunk):
    """bf16 shapes outside the tensor-core kernels' (d = 128, chunk 64): the CUDA-core path."""
    w = I.PREFILL.with_(B=1, H=2, T=150, dk=dk, dv=dv, chunk=chunk)
    check(*run(w), TOL["bf16"])


@pytest.mark.parametrize("chunk,bound", [(16, -5.0), (64, -1.25)])
def test_bwd_log_decay(chunk, bound):
    """The pages' log-domain decay: g_min = -5 on 16-token chunks, -1.25 on 64."""
    w = I.CORRECTNESS.with_(T=130, chunk=chunk, init_std=0.3)
    check(*run(w, bound=bound, decay="log"), TOL["f32"])


@pytest.mark.parametrize("dk,dv,chunk", [(128, 128, 32), (32, 16, 16), (64, 128, 64)])
def test_bwd_other_shapes(dk, dv, chunk):
    w = I.CORRECTNESS.with_(T=97, dk=dk, dv=dv, chunk=chunk, init_std=0.3)
    check(*run(w), TOL["f32"])


def test_bwd_empty_sequence():
    """T = 0: the initial state's gradient is d_final; nothing else exists."""
    w = I.CORRECTNESS.with_(B=2, T=0, init_std=0.3)
    x = I.prefill_inputs(w, device="cuda")
    ct = I.cotangents(w, device="cuda")
    got = gdr.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, x["init_state"],
                        ct["d_out"], ct["d_final"])
    torch.cuda.synchronize()
    assert torch.equal(got[5], ct["d_final"])


@pytest.mark.slow
def test_bwd_bf16_prefill_full_heads():
    """Every head of the prefill workload's batch element 0 at full length (B = 1,
    H = 16, T = 4096): the whole sequence through the reverse chain."""
    w = I.PREFILL.with_(B=1)
    check(*run(w), TOL["bf16"])
