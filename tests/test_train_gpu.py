"""GPU parity of the training pair gdr_chunk_fwd_train / gdr_chunk_bwd_saved (through
the C ABI) against the oracles on the same seeded inputs.

* The training forward's out and final state are bit-identical to gdr_chunk_fwd_ws
  (the same kernels; saving only adds stores).
* The saved buffer: every chunk's state M_n, tile W_n, triangular inverse T_n and
  masked decayed scores P_n against the chunked oracle's intermediates
  (oracle.chunkwise.head, itself checked against the token loop), to 5e-3 relative
  L2 (bf16 tiles of fp32 values, 2^-9 per element, plus the forward's own bf16
  operand rounding), with the padding past the end of the sequence exact; the row
  scalars against the oracle's decay and a difference quotient of its log alpha.
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
    """The saved buffer's four regions: states [B*H, NC, dk, dv] as M, W [B*H, NC, 64, dv],
    T and P [B*H, NC, 64, 64], row scalars [B*H, NC, 4, 64] (gamma, 1 / gamma, beta,
    d log(alpha) / dg)."""
    NC = (T + 63) // 64
    BH = B * H
    raw = saved[: gdr.chunk_saved_size(B, H, T, 128, 128)]
    n_st, n_w, n_tp = BH * NC * 128 * 128, BH * NC * 128 * 64, BH * NC * 2 * 64 * 64
    flat = raw[: 2 * (n_st + n_w + n_tp)].view(torch.bfloat16)
    st = flat[:n_st].view(BH, NC, 128, 128)                        # [j][i] = M[i][j]
    wt = flat[n_st:n_st + n_w].view(BH, NC, 128, 64)               # [j][s] = W[s][j]
    tp = flat[n_st + n_w:].view(BH, NC, 2, 64, 8, 8).float()
    # T and P have their 16-byte chunks swizzled by row: plain chunk c of row r is stored
    # chunk c ^ (r % 8)
    r = torch.arange(64, device=saved.device)[:, None]
    c = torch.arange(8, device=saved.device)[None, :]
    tp = tp[:, :, :, r, c ^ (r % 8), :].reshape(BH, NC, 2, 64, 64)
    sc = raw[2 * (n_st + n_w + n_tp):].view(torch.float32).view(BH, NC, 4, 64)
    return st.transpose(-1, -2).float(), wt.transpose(-1, -2).float(), tp[:, :, 0], tp[:, :, 1], sc


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
    st, wt, tt, pt, sc = saved_views(saved, w.B, w.H, T)
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
            # T, P: bf16 tiles; past the end, the identity's rows and zero rows
            assert oracle.rel_l2(tt[h, n, :c, :c], inter["T"][n]) <= TOL, (h, n)
            assert oracle.rel_l2(pt[h, n, :c, :c], inter["P"][n]) <= TOL, (h, n)
            assert not tt[h, n, :c, c:].any() and not pt[h, n, :, c:].any()
            assert torch.equal(tt[h, n, c:, c:], torch.eye(64 - c, device=tt.device)) and not tt[h, n, c:, :c].any()
            assert not pt[h, n, c:].any()


@pytest.mark.parametrize("T,segments,decay", [(64, 1, "affine"), (333, 1, "affine"),
                                              (1600, 3, "affine"), (257, 1, "log")])
def test_saved_row_scalars(T, segments, decay):
    """The forward's per-chunk row scalars: gamma and 1 / gamma against the oracle's
    cumulative decay (fp32 exponent of an fp32 sum: 1e-5 relative), beta exactly, and
    d log(alpha) / dg against a central difference of the oracle's log alpha in fp64
    (step 1e-4: error ~1e-9; 1e-4 relative for the fp32 1 - sigmoid); past the end
    1, 1, 0, 0."""
    w = I.PREFILL.with_(B=1, H=2, T=T)
    x = I.prefill_inputs(w, device="cuda")
    bound = w.a_min if decay == "affine" else -1.25
    with gdr.option(segments=segments):
        _, _, saved = train_fwd(x, w, bound, decay)
    torch.cuda.synchronize()
    sc = saved_views(saved, w.B, w.H, T)[4].cpu().double().numpy()
    g = x["g"].cpu().double().numpy()
    beta = x["beta"].cpu().numpy()
    eps = 1e-4
    for h in range(w.H):
        _, gam, _ = chunkwise.chunk_decay(g[0, h], bound, 64, decay)
        dla = (chunkwise.log_alpha(g[0, h] + eps, bound, decay)
               - chunkwise.log_alpha(g[0, h] - eps, bound, decay)) / (2 * eps)
        for n in range((T + 63) // 64):
            sl = slice(64 * n, min(64 * n + 64, T))
            c = sl.stop - sl.start
            blk = sc[h, n]
            np.testing.assert_allclose(blk[0, :c], gam[sl], rtol=1e-5)
            np.testing.assert_allclose(blk[1, :c], 1.0 / gam[sl], rtol=1e-5)
            assert np.array_equal(blk[2, :c], beta[0, h, sl].astype(np.float64))
            np.testing.assert_allclose(blk[3, :c], dla[sl], rtol=1e-4, atol=1e-7)
            assert (blk[0, c:] == 1).all() and (blk[1, c:] == 1).all()
            assert not blk[2:, c:].any()


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
    with gdr.option(bwd_variant=2):   # the backward's own recomputation
        rec = gdr.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, init_state,
                            ct["d_out"], d_final)
    torch.cuda.synchronize()
    errs = {n: oracle.rel_l2(a, b) for n, a, b in zip(NAMES, got, rec)}
    print(" ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    assert all(e <= TOL for e in errs.values()), errs


def test_default_backward_is_the_saved_state_pair():
    """gdr_chunk_bwd's default for this shape runs the training forward's kernels into
    its workspace and then the saved-state backward: bit-identical to the pair called
    by hand (the same kernels on the same inputs, deterministic reductions)."""
    w = I.PREFILL.with_(B=2, H=4, T=1000)
    x, ct, init_state, d_final, got = bwd_pair(w)
    with gdr.option(segments=1):   # as bwd_pair's forward
        dflt = gdr.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, init_state,
                             ct["d_out"], d_final)
    torch.cuda.synchronize()
    for n, a, b in zip(NAMES, got, dflt):
        assert torch.equal(a, b), n


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
