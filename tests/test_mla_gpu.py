"""GPU parity of one decode step of gated multi-head latent attention (gdr_mla_decode,
through the C ABI) against the fp64 oracle (oracle.mla_decode) on the same seeded
inputs: relative L2 over the whole output at most 5e-3 (bf16 operands, bf16 output).
Cases: one and several splits of the cache, ragged and empty sequences, two head
groups, cache rows past the length holding NaN, scores that grow along the cache (the
running-maximum rescale), the decode workload itself on sampled sequences, and an
injected timeout."""
from __future__ import annotations

import pytest
import torch

import oracle
import gated_delta_rule_gdr_gb300 as gdr
from gated_delta_rule_gdr_gb300 import inputs as I

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdr.load(build_if_missing=True)
    yield
    assert gdr.last_device_error() == 0


def run(x, w):
    out = gdr.mla_decode(x["q_abs"], x["ckv"], x["seqlens"], x["w_uv"], x["gate"], w.scale)
    torch.cuda.synchronize()
    return out


def ref(x, w):
    cpu = {n: t.cpu() for n, t in x.items()}
    return oracle.mla_decode(cpu["q_abs"], cpu["ckv"], cpu["seqlens"], cpu["w_uv"], cpu["gate"],
                             w.scale)


@pytest.mark.parametrize("N,H,L,lens", [(3, 64, 200, [200, 1, 65]), (2, 64, 4096, [4096, 3001]),
                                        (2, 128, 1000, [999, 64]), (4, 64, 700, [0, 700, 63, 129]),
                                        (1, 64, 64, [64]), (5, 64, 2500, [2500, 1, 1299, 2048, 77])])
def test_mla_matches_oracle(N, H, L, lens):
    w = I.MLA_DECODE.with_(N=N, H=H, L=L)
    x = {n: t.cuda() for n, t in I.mla_inputs(w).items()}
    x["seqlens"] = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = run(x, w)
    r = ref(x, w)
    e = oracle.rel_l2(out, r)
    assert e <= TOL, e
    for n, ln in enumerate(lens):
        if ln == 0:
            assert not out[n].any()            # an empty cache contributes zero
        else:
            assert oracle.rel_l2(out[n], r[n]) <= TOL


def test_mla_ignores_rows_past_the_length():
    w = I.MLA_DECODE.with_(N=2, L=300)
    x = {n: t.cuda() for n, t in I.mla_inputs(w).items()}
    x["seqlens"] = torch.tensor([130, 257], dtype=torch.int32, device="cuda")
    a = run(x, w)
    x["ckv"][0, 130:] = float("nan")
    x["ckv"][1, 257:] = float("inf")
    b = run(x, w)
    assert torch.isfinite(b.float()).all()
    assert torch.equal(a, b)


def test_mla_running_maximum_rescale():
    """Latents whose scale grows along the cache: every later tile raises the scores'
    maximum far beyond the first tile's, so the accumulated sums must be rescaled."""
    w = I.MLA_DECODE.with_(N=2, L=1024)
    x = {n: t.cuda() for n, t in I.mla_inputs(w).items()}
    grow = torch.linspace(0.2, 3.0, w.L, device="cuda").view(1, -1, 1)
    x["ckv"] = (x["ckv"].float() * grow).to(torch.bfloat16)
    out = run(x, w)
    e = oracle.rel_l2(out, ref(x, w))
    assert e <= TOL, e


@pytest.mark.slow
def test_mla_decode_workload_sampled():
    """The decode workload (N32 H64, 32768 cached tokens each): the oracle on sequences
    0, 13 and 31 (every head); every output finite."""
    w = I.MLA_DECODE
    x = {n: t for n, t in I.mla_inputs(w, device="cuda").items()}
    out = run(x, w)
    assert torch.isfinite(out.float()).all()
    pick = [0, 13, 31]
    sub = {n: t[pick] for n, t in x.items() if n != "w_uv"}
    sub["w_uv"] = x["w_uv"]
    r = ref(sub, w)
    e = oracle.rel_l2(out[pick], r)
    print(f"mla decode workload rel-L2 (sequences {pick}) {e:.3e}")
    assert e <= TOL, e


def test_mla_injected_timeout_is_reported_and_recovers():
    w = I.MLA_DECODE.with_(N=2, L=600)
    x = {n: t.cuda() for n, t in I.mla_inputs(w).items()}
    assert gdr.last_device_error() == 0
    with gdr.option(wait_limit_ns=0):
        gdr.mla_decode(x["q_abs"], x["ckv"], x["seqlens"], x["w_uv"], x["gate"], w.scale)
        assert gdr.last_device_error() == 5          # GDR_ERR_TIMEOUT
    assert gdr.last_device_error() == 0
    out = run(x, w)
    assert oracle.rel_l2(out, ref(x, w)) <= TOL
