"""GPU parity of the training pair gdr_chunk_fwd_train / gdr_chunk_bwd_saved (through
the C ABI) against the oracles on the same seeded inputs.

* The training forward's out and final state are bit-identical to gdr_chunk_fwd_ws
  (the same kernels; saving only adds stores).
* The saved buffer: every chunk's state M_n and tile W_n against the chunked oracle's
  intermediates (oracle.chunkwise.head, itself checked against the token loop), to
  5e-3 relative L2 (bf16 tiles of fp32 values, 2^-9 per element, plus the forward's
  own bf16 operand rounding); rows of W past the end of the sequence are zero.
* The saved-state backward against the fp64 oracle's gradients, 5e-3 relative L2
  per gradient (the tolerance of the recomputing bf16 backward, which it tracks:
  both read bf16 states), with ragged tails, sequence segments on and off, no
  initial state or final cotangent, and the log decay.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import chunkwise
import gated_delta_rule_gdr_gb300 as gdr
from gated_delta_rule_gdr_gb300 import inputs as I

pytestmark = pytest.mark.gpu
TOL = 5e-3
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dinit")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdr.load(build_if_missing=True)
    yield
    assert gdr.last_device_error() == 0


def saved_views(saved, B, H, T):
    """(states [B*H, NC, dk, dv] as M, W [B*H, NC, 64, dv]) from the saved buffer."""
    NC = (T + 63) // 64
    BH = B * H
    flat = saved[: gdr.chunk_saved_size(B, H, T, 128, 128)].view(torch.bfloat16)
    st = flat[: BH * NC * 128 * 128].view(BH, NC, 128, 128)        # [j][i] = M[i][j]
    wt = flat[BH * NC * 128 * 128:].view(BH, NC, 128, 64)          # [j][s] = W[s][j]
    return st.transpose(-1, -2).float(), wt.transpose(-1, -2).float()


def train_fwd(x, w, bound=None, decay="affine", init=True):
    bound = w.a_min if bound is None else bound
    return gdr.chunk_fwd_train(x["q"], x["k"], x["v"], x["g"], x["beta"], bound,
                               x["init_state"] if init else None, decay=decay)


@pytest.mark.parametrize("T,segments", [(64, 1), (200, 1), (1000, 1), (4096, 4), (3000, 3)])
def test_train_forward_matches_the_prefill(T, segments):
    w = I.PREFILL.with_(B=1, H=2, T=T)
    x = I.prefill_inputs(w, device="cuda")
    with gdr.option(segments=segments):
        out, fin, saved = train_fwd(x, w)
        ref_out, ref_fin = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min,
                                         x["init_state"])
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    assert torch.equal(fin, ref_fin)


@pytest.mark.parametrize("T,segments,split", [(64, 1, 0), (130, 1, 0), (777, 1, 0), (1600, 3, 0),
                                              (200, 1, 1), (1300, 3, 1)])
def test_saved_states_and_w_tiles(T, segments, split):
    """split 1 forces one chain CTA per head (all 128 value columns: the chain's other
    shape, taken when two CTAs per head would not all fit on the GPU)."""
    w = I.PREFILL.with_(B=1, H=2, T=T)
    x = I.prefill_inputs(w, device="cuda")
    with gdr.option(segments=segments, chain_split=split):
        _, _, saved = train_fwd(x, w)
    torch.cuda.synchronize()
    st, wt = saved_views(saved, w.B, w.H, T)
    cpu = {n: t.float().cpu().numpy() for n, t in x.items()}
    for h in range(w.H):
        _, _, inter = chunkwise.head(cpu["q"][0, h], cpu["k"][0, h], cpu["v"][0, h],
                                     cpu["g"][0, h], cpu["beta"][0, h], w.a_min,
                                     cpu["init_state"][0, h], keep=True)
        for n, (M, W) in enumerate(zip(inter["M"], inter["W"])):
            assert oracle.rel_l2(st[h, n], M) <= TOL, (h, n)
            c = W.shape[0]
            assert oracle.rel_l2(wt[h, n, :c], W) <= TOL, (h, n)
            assert not wt[h, n, c:].any()                     # past the end: zero


def bwd_pair(w, *, segments=1, init=True, final=True, bound=None, decay="affine", split=0):
    x = I.prefill_inputs(w, device="cuda")
    ct = I.cotangents(w, device="cuda")
    bound = w.a_min if bound is None else bound
    init_state = x["init_state"] if init else None
    d_final = ct["d_final"] if final else None
    with gdr.option(segments=segments, chain_split=split):
        _, _, saved = train_fwd(x, w, bound, decay, init)
    got = gdr.chunk_bwd_saved(x["q"], x["k"], x["v"], x["g"], x["beta"], bound, init_state,
                              ct["d_out"], saved, d_final, decay=decay)
    torch.cuda.synchronize()
    assert gdr.last_device_error() == 0
    return x, ct, init_state, d_final, got


def check(got, ref):
    errs = {}
    for n, a, b in zip(NAMES, got, ref):
        if b is None:
            continue
        assert np.isfinite(a.float().cpu().numpy()).all(), n
        errs[n] = oracle.rel_l2(a, b)
    print(" ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    assert all(e <= TOL for e in errs.values()), errs


@pytest.mark.parametrize("T,segments,split", [(1, 1, 0), (64, 1, 0), (65, 1, 0), (300, 1, 0),
                                              (2048, 4, 0), (300, 1, 1)])
def test_bwd_saved_matches_oracle(T, segments, split):
    w = I.PREFILL.with_(B=1, H=2, T=T)
    x, ct, init_state, d_final, got = bwd_pair(w, segments=segments, split=split)
    cpu = lambda t: None if t is None else t.cpu()
    ref = oracle.bwd(*(cpu(x[n]) for n in ("q", "k", "v", "g", "beta")), w.a_min,
                     cpu(init_state), cpu(ct["d_out"]), cpu(d_final))
    check(got, ref)


@pytest.mark.parametrize("init,final", [(False, False), (True, False), (False, True)])
def test_bwd_saved_optional_state_terms(init, final):
    w = I.PREFILL.with_(B=1, H=2, T=190)
    x, ct, init_state, d_final, got = bwd_pair(w, init=init, final=final)
    cpu = lambda t: None if t is None else t.cpu()
    ref = oracle.bwd(*(cpu(x[n]) for n in ("q", "k", "v", "g", "beta")), w.a_min,
                     cpu(init_state), cpu(ct["d_out"]), cpu(d_final))
    check(got, ref)


def test_bwd_saved_log_decay():
    w = I.PREFILL.with_(B=1, H=2, T=257)
    x, ct, init_state, d_final, got = bwd_pair(w, bound=-1.25, decay="log")
    cpu = lambda t: None if t is None else t.cpu()
    ref = oracle.bwd(*(cpu(x[n]) for n in ("q", "k", "v", "g", "beta")), -1.25,
                     cpu(init_state), cpu(ct["d_out"]), cpu(d_final), decay="log")
    check(got, ref)


def test_bwd_saved_tracks_the_recomputing_backward():
    """Both read bf16 states (the forward's operands, or recomputed in near-fp32 and
    rounded), so the two backward paths agree within the oracle tolerance: each is
    ~3e-3 from the fp64 gradients, partly through the same bf16 roundings, and the
    bf16 gradient outputs alone differ by up to an ulp (2^-9 relative) where their
    fp32 values straddle a rounding boundary."""
    w = I.PREFILL.with_(B=2, H=4, T=1000)
    x, ct, init_state, d_final, got = bwd_pair(w)
    rec = gdr.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, init_state,
                        ct["d_out"], d_final)
    torch.cuda.synchronize()
    errs = {n: oracle.rel_l2(a, b) for n, a, b in zip(NAMES, got, rec)}
    print(" ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    assert all(e <= TOL for e in errs.values()), errs


def test_train_pair_empty_sequence():
    w = I.PREFILL.with_(B=1, H=2, T=0)
    x = I.prefill_inputs(w, device="cuda")
    out, fin, saved = train_fwd(x, w)
    torch.cuda.synchronize()
    assert out.numel() == 0 and torch.equal(fin, x["init_state"])
    ct = I.cotangents(w, device="cuda")
    got = gdr.chunk_bwd_saved(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min,
                              x["init_state"], ct["d_out"], saved, ct["d_final"])
    torch.cuda.synchronize()
    assert torch.equal(got[5], ct["d_final"])                 # d_init = d_final


@pytest.mark.slow
def test_bwd_saved_prefill_workload_sampled():
    """The prefill workload (B4 H16 T4096): the training pair end to end, the oracle
    gradients of heads (0, 0) and (3, 15)."""
    w = I.PREFILL
    x, ct, init_state, d_final, got = bwd_pair(w)
    for b, h in ((0, 0), (3, 15)):
        sl = lambda t: None if t is None else t[b:b + 1, h:h + 1].cpu()
        ref = oracle.bwd(*(sl(x[n]) for n in ("q", "k", "v", "g", "beta")), w.a_min,
                         sl(init_state), sl(ct["d_out"]), sl(d_final))
        check([t[b:b + 1, h:h + 1] for t in got], ref)
