"""Pins of the gated multi-head latent attention oracle (oracle/mla_oracle.c), CPU only.

Each check ties the oracle to something other than itself:
* attention written out over explicitly up-projected keys and values (k = W_uk c,
  v = W_uv c, no absorption of W_uk into the query), with scipy's softmax and
  sigmoid, on inputs whose absorbed query is exact in fp32 -- pins the absorption
  algebra, the scale, the softmax axis, the up-projection's orientation and the gate;
* one cached token: the softmax weight is exactly 1;
* identical latents: the output does not depend on the query;
* a zero query: every weight is 1 / len, the plain average;
* a score 1000 above the rest: the result is that token's, finite (the maximum
  subtraction of the softmax identity is what keeps exp in range);
* rows past a sequence's length do not matter, and length 0 gives zero;
* the gate's limits sigmoid(+inf) = 1, sigmoid(0) = 1/2, sigmoid(-inf) = 0.
test_mla_pins_catch_planted_mistakes shows each pin set catches plausible slips.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle


def _dyadic(rng, shape, scale, levels=4):
    """Small dyadic values: products and short sums of them are exact in fp32."""
    return (rng.integers(-levels, levels + 1, size=shape) * scale).astype(np.float32)


def _case(rng, N=2, H=3, L=7, dc=16, dh=8):
    ckv = _dyadic(rng, (N, L, dc), 0.25)
    w_uv = _dyadic(rng, (H, dh, dc), 0.125)
    gate = _dyadic(rng, (N, H, dh), 0.5)
    return ckv, w_uv, gate


def check_mla_matches_unabsorbed_attention():
    rng = np.random.default_rng(1)
    N, H, L, dc, dh = 2, 3, 7, 16, 8
    ckv, w_uv, gate = _case(rng, N, H, L, dc, dh)
    w_uk = _dyadic(rng, (H, dh, dc), 0.5, levels=2)
    q = _dyadic(rng, (N, H, dh), 0.25, levels=2)
    q_abs = np.einsum("hdc,nhd->nhc", w_uk.astype(np.float64), q.astype(np.float64))
    assert np.array_equal(q_abs.astype(np.float32).astype(np.float64), q_abs)   # exact in fp32
    lens = np.array([7, 4])
    scale = 0.125
    got = oracle.mla_decode(q_abs.astype(np.float32), ckv, lens, w_uv, gate, scale)
    for n in range(N):
        c = ckv[n, :lens[n]].astype(np.float64)
        for h in range(H):
            k = c @ w_uk[h].astype(np.float64).T          # [len, dh]: keys, up-projected
            v = c @ w_uv[h].astype(np.float64).T          # [len, dh]: values, up-projected
            p = softmax(scale * (k @ q[n, h].astype(np.float64)))
            ref = expit(gate[n, h].astype(np.float64)) * (p @ v)
            np.testing.assert_allclose(got[n, h], ref, rtol=1e-12, atol=1e-13)


def check_mla_one_token():
    rng = np.random.default_rng(2)
    ckv, w_uv, gate = _case(rng)
    q_abs = rng.standard_normal((2, 3, 16)).astype(np.float32)
    got = oracle.mla_decode(q_abs, ckv, np.array([1, 1]), w_uv, gate, 0.7)
    for n in range(2):
        for h in range(3):
            ref = expit(gate[n, h].astype(np.float64)) * (w_uv[h].astype(np.float64) @ ckv[n, 0])
            np.testing.assert_allclose(got[n, h], ref, rtol=1e-13, atol=1e-14)


def check_mla_identical_latents():
    rng = np.random.default_rng(3)
    ckv, w_uv, gate = _case(rng)
    ckv[:] = ckv[:, :1]                                   # every row the same latent
    q1 = rng.standard_normal((2, 3, 16)).astype(np.float32)
    q2 = 5 * rng.standard_normal((2, 3, 16)).astype(np.float32)
    a = oracle.mla_decode(q1, ckv, np.array([7, 5]), w_uv, gate, 0.3)
    b = oracle.mla_decode(q2, ckv, np.array([7, 5]), w_uv, gate, 0.3)
    ref = oracle.mla_decode(q1, ckv, np.array([1, 1]), w_uv, gate, 0.3)
    np.testing.assert_allclose(a, ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b, ref, rtol=1e-12, atol=1e-13)


def check_mla_zero_query_is_the_average():
    rng = np.random.default_rng(4)
    ckv, w_uv, gate = _case(rng)
    lens = np.array([7, 3])
    got = oracle.mla_decode(np.zeros((2, 3, 16), np.float32), ckv, lens, w_uv, gate, 0.9)
    for n in range(2):
        mean = ckv[n, :lens[n]].astype(np.float64).mean(0)
        for h in range(3):
            ref = expit(gate[n, h].astype(np.float64)) * (w_uv[h].astype(np.float64) @ mean)
            np.testing.assert_allclose(got[n, h], ref, rtol=1e-13, atol=1e-14)


def check_mla_dominant_score():
    """Scores far beyond exp's range (about 709): token 2 leads by 1000."""
    rng = np.random.default_rng(5)
    N, H, L, dc, dh = 1, 2, 6, 16, 8
    _, w_uv, gate = _case(rng, N, H, L, dc, dh)
    ckv = np.zeros((N, L, dc), np.float32)
    for t in range(L):
        ckv[0, t, t] = 1.0                                # latent t = e_t (plus a tail)
        ckv[0, t, 8:] = rng.standard_normal(8)
    q_abs = np.zeros((N, H, dc), np.float32)
    q_abs[0, :, :L] = 2000.0
    q_abs[0, :, 2] = 3000.0                               # score of token 2: 3000, others 2000
    got = oracle.mla_decode(q_abs, ckv, np.array([L]), w_uv, gate, 1.0)
    assert np.all(np.isfinite(got))
    for h in range(H):
        ref = expit(gate[0, h].astype(np.float64)) * (w_uv[h].astype(np.float64) @ ckv[0, 2])
        np.testing.assert_allclose(got[0, h], ref, rtol=1e-13, atol=1e-14)


def check_mla_length_masks_the_tail():
    rng = np.random.default_rng(6)
    ckv, w_uv, gate = _case(rng)
    q_abs = rng.standard_normal((2, 3, 16)).astype(np.float32)
    lens = np.array([4, 0])
    a = oracle.mla_decode(q_abs, ckv, lens, w_uv, gate, 0.5)
    ckv2 = ckv.copy()
    ckv2[0, 4:] = 99.0                                    # rows past the length
    ckv2[1] = -7.0
    b = oracle.mla_decode(q_abs, ckv2, lens, w_uv, gate, 0.5)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a[1], 0.0)              # an empty cache contributes nothing
    c = oracle.mla_decode(q_abs[:1], ckv[:1, :4], np.array([4]), w_uv, gate[:1], 0.5)
    np.testing.assert_array_equal(a[:1], c)


def check_mla_gate_limits():
    rng = np.random.default_rng(7)
    ckv, w_uv, _ = _case(rng)
    q_abs = rng.standard_normal((2, 3, 16)).astype(np.float32)
    lens = np.array([7, 6])
    full = oracle.mla_decode(q_abs, ckv, lens, w_uv, np.full((2, 3, 8), 60.0, np.float32), 0.4)
    half = oracle.mla_decode(q_abs, ckv, lens, w_uv, np.zeros((2, 3, 8), np.float32), 0.4)
    off = oracle.mla_decode(q_abs, ckv, lens, w_uv, np.full((2, 3, 8), -60.0, np.float32), 0.4)
    np.testing.assert_allclose(half, 0.5 * full, rtol=1e-12, atol=1e-14)
    assert np.abs(off).max() <= 1e-20 * max(1.0, np.abs(full).max())


ALL_MLA_CHECKS = [check_mla_matches_unabsorbed_attention, check_mla_one_token,
                  check_mla_identical_latents, check_mla_zero_query_is_the_average,
                  check_mla_dominant_score, check_mla_length_masks_the_tail,
                  check_mla_gate_limits]


@pytest.mark.parametrize("check", ALL_MLA_CHECKS, ids=lambda f: f.__name__)
def test_mla_oracle_pin(check):
    check()


# (name, text in mla_oracle.c, replacement): slips a restatement of the layer could make
MLA_MUTANTS = [
    ("scale dropped", "s[t] = scale * acc;", "s[t] = acc;"),
    ("maximum not subtracted", "const double p = exp(s[t] - m);", "const double p = exp(s[t]);"),
    ("weights not normalised", "for (c = 0; c < dc; ++c) ol[c] /= l;", "(void)l;"),
    ("first token skipped", "for (t = 0; t < len; ++t) {\n            const double p",
     "for (t = 1; t < len; ++t) {\n            const double p"),
    ("latents weighted by the score", "ol[c] += p * (double)ckv[t * dc + c];",
     "ol[c] += s[t] * (double)ckv[t * dc + c];"),
    ("gate applied to -z", "out[j] = sigmoid((double)z[j]) * o;",
     "out[j] = sigmoid(-(double)z[j]) * o;"),
    ("gate missing", "out[j] = sigmoid((double)z[j]) * o;", "out[j] = o;"),
    ("query read from the next head", "J->q_abs + (n * J->H + h) * J->dc",
     "J->q_abs + (n * J->H + (h + 1) % J->H) * J->dc"),
    ("length ignored", "mla_one(J->q_abs", "len = J->Lmax;\n            mla_one(J->q_abs"),
]


@contextlib.contextmanager
def _mla_lib(path):
    lib = ctypes.CDLL(path)
    oracle.set_mla_signature(lib)
    saved = oracle._load_mla()
    oracle._mla_lib = lib
    try:
        yield
    finally:
        oracle._mla_lib = saved


@pytest.mark.parametrize("mutant", MLA_MUTANTS, ids=[m[0] for m in MLA_MUTANTS])
def test_mla_pins_catch_planted_mistakes(mutant, tmp_path):
    name, old, new = mutant
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")).read()
    assert old in src, name
    src = src.replace(old, new, 1)
    c_path, so_path = tmp_path / "mutant.c", tmp_path / "mutant.so"
    c_path.write_text(src)
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-std=c11", "-o", str(so_path), str(c_path),
                    "-lm", "-lpthread"], check=True)
    caught = []
    with _mla_lib(str(so_path)):
        for check in ALL_MLA_CHECKS:
            try:
                with np.errstate(all="ignore"):
                    check()
            except AssertionError:
                caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake: {name}"
