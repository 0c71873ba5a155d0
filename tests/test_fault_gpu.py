"""Failure detection without a GPU fault: the wait_limit_ns option set to 0 makes
every bounded wait of the prefill kernels give up at once.  The kernel must unwind (let
its own copies land, free TMEM, return), gdr_last_device_error must report
GDR_ERR_TIMEOUT, and the context must stay usable for the next call."""
from __future__ import annotations

import pytest
import torch

import oracle
import gated_delta_rule_gdr_gb300 as gdr
from gated_delta_rule_gdr_gb300 import inputs as I

pytestmark = pytest.mark.gpu


# (library options, workspace): the fused kernels on the single-launch path, the
# preparation and chain kernels on the two-kernel path
VARIANTS = {"single": ({"fused_variant": 1}, None),
            "pair": ({"fused_variant": 2}, None),
            "chain2": ({"chain_split": 2}, "auto"),
            "chain1": ({"chain_split": 1}, "auto"),
            "segments": ({"segments": 3}, "auto")}


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_injected_timeout_is_reported_and_recovers(variant):
    opts, ws = VARIANTS[variant]
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdr.load(build_if_missing=True)
    w = I.PREFILL.with_(B=1, H=2, T=300)
    x = I.prefill_inputs(w, device="cuda")
    with gdr.option(**opts):
        assert gdr.last_device_error() == 0
        with gdr.option(wait_limit_ns=0):
            gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, x["init_state"],
                          workspace=ws)
            assert gdr.last_device_error() == 5          # GDR_ERR_TIMEOUT
        assert gdr.last_device_error() == 0              # the word was cleared
        out, fin = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min,
                                 x["init_state"], workspace=ws)
        torch.cuda.synchronize()
    cpu = {n: t.cpu() for n, t in x.items()}
    ro, rf = oracle.fwd(cpu["q"], cpu["k"], cpu["v"], cpu["g"], cpu["beta"], w.a_min,
                        cpu["init_state"])
    assert oracle.rel_l2(out, ro) <= 5e-3 and oracle.rel_l2(fin, rf) <= 5e-3
    assert gdr.last_device_error() == 0


def test_backward_injected_timeout_is_reported_and_recovers():
    """The tensor-core per-chunk gradient kernel of the backward under the same injection:
    its loads land, its products drain, and the next call is correct."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdr.load(build_if_missing=True)
    w = I.PREFILL.with_(B=1, H=2, T=300)
    x = I.prefill_inputs(w, device="cuda")
    ct = I.cotangents(w, device="cuda")
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, x["init_state"], ct["d_out"],
            ct["d_final"])
    assert gdr.last_device_error() == 0
    with gdr.option(wait_limit_ns=0):
        gdr.chunk_bwd(*args)
        assert gdr.last_device_error() == 5          # GDR_ERR_TIMEOUT
    assert gdr.last_device_error() == 0
    got = gdr.chunk_bwd(*args)
    torch.cuda.synchronize()
    cpu = lambda t: None if t is None else t.cpu()
    ref = oracle.bwd(*(cpu(x[n]) for n in ("q", "k", "v", "g", "beta")), w.a_min,
                     cpu(x["init_state"]), cpu(ct["d_out"]), cpu(ct["d_final"]))
    for a, b in zip(got, ref):
        assert oracle.rel_l2(a, b) <= 5e-3
    assert gdr.last_device_error() == 0
