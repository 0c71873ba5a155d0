"""Pins for the fp64 oracle: facts fixed by the mathematics, not by the oracle.

Each check below is chosen so that a plausible slip in the oracle (a dropped
decay factor, a wrong sign, k and q swapped, a transposed state, a flipped
sigmoid) breaks at least one of them; ``test_pins_catch_planted_mistakes``
plants such slips in a copy of the oracle's C source and proves it.

* unrolled products  -- for T <= 8 the recurrence is the closed form
  S_T = S_0 prod_t E_t + sum_t beta_t v_t k_t^T prod_{s>t} E_s with explicit
  dk x dk matrices E_t = alpha_t (I - beta_t k_t k_t^T); no u = S k shortcut.
* write/read         -- alpha = beta = 1 with orthonormal keys: after writing,
  S k_i returns v_i exactly (the correct-on-write semantics of the incremental
  rule, 'How to Think About Trillion-Parameter Sparse Multimodal LLMs', 2.2).
* closed forms       -- beta = 0 is pure decay; a_min = 1 removes g entirely.
* hand-worked case   -- tests/golden/hand_worked_t2_d2.json.
* chunked algebra    -- the independent chunkwise reformulation agrees with the
  token loop to ~1e-12 for C in {1, 8, 64} and ragged T.
* decay bounds       -- a_min^r <= gamma_r <= 1 and 1/gamma_r <= a_min^-C, the
  bounded reciprocal the pages' method relies on ('Trillion-Parameter MoE
  Multimodal LLMs: How to Evaluate the New Generation', 3.1), and the range
  figures the pages print (tests/golden/range_facts.json).
* the log-domain decay -- the pages' own log alpha = g_min sigmoid(g): limits and
  symmetry, both limits of g reproduced by the linear-domain form, the chunked
  algebra on 16-token chunks at g_min = -5, and its range bound.
"""
from __future__ import annotations

import contextlib
import ctypes
import json
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import chunkwise

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng_master = np.random.default_rng(12345)


def _rand_inputs(rng, B, H, T, dk, dv, unit=True, init=True):
    q = rng.standard_normal((B, H, T, dk)).astype(np.float32)
    k = rng.standard_normal((B, H, T, dk)).astype(np.float32)
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, dv)).astype(np.float32)
    g = rng.standard_normal((B, H, T)).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-rng.standard_normal((B, H, T))))).astype(np.float32)
    M0 = (0.3 * rng.standard_normal((B, H, dk, dv))).astype(np.float32) if init else None
    return q, k, v, g, beta, M0


# ----------------------------------------------------------------- checks
# Each returns normally when the pin holds and raises AssertionError otherwise.

def check_alpha_limits():
    for a_min in (0.0, 0.3, 0.9, 0.99, 1.0):
        a = oracle.alpha(np.array([0.0, 40.0, -40.0, 1.0, -1.0]), a_min)
        assert abs(a[0] - (1.0 + a_min) / 2.0) < 1e-15          # sigmoid(0) = 1/2
        assert abs(a[1] - 1.0) < 1e-15                           # g -> +inf: no decay
        assert abs(a[2] - a_min) < 1e-15                         # g -> -inf: the floor
        assert a[3] > a[0] > a[4] or a_min == 1.0                # increasing in g
        assert abs((a[3] - a_min) + (a[4] - a_min) - (1.0 - a_min)) < 1e-15  # s(x)+s(-x)=1


def check_hand_worked():
    fx = json.load(open(os.path.join(GOLDEN, "hand_worked_t2_d2.json")))
    q = np.array(fx["q"], np.float32)[None, None]
    k = np.array(fx["k"], np.float32)[None, None]
    v = np.array(fx["v"], np.float32)[None, None]
    g = np.array(fx["g"], np.float32)[None, None]
    beta = np.array(fx["beta"], np.float32)[None, None]
    M0 = np.array(fx["init_state_M"], np.float32)[None, None]
    out, fin = oracle.fwd(q, k, v, g, beta, fx["a_min"], M0)
    assert np.array_equal(out[0, 0], np.array(fx["out"])), out
    assert np.array_equal(fin[0, 0], np.array(fx["final_state_M"])), fin


def _unrolled(q, k, v, g, beta, a_min, M0):
    """Closed form of the recurrence for one head with explicit matrices."""
    T, dk = k.shape
    dv = v.shape[1]
    k64, v64, q64 = (x.astype(np.float64) for x in (k, v, q))
    al = a_min + (1.0 - a_min) / (1.0 + np.exp(-g.astype(np.float64)))
    E = [al[t] * (np.eye(dk) - beta[t] * np.outer(k64[t], k64[t])) for t in range(T)]
    S0 = M0.astype(np.float64).T
    outs = []
    for tt in range(1, T + 1):             # S after tt tokens, from scratch
        P = np.eye(dk)
        for t in range(tt):
            P = P @ E[t]
        S = S0 @ P
        for t in range(tt):
            tail = np.eye(dk)
            for s in range(t + 1, tt):
                tail = tail @ E[s]
            S = S + beta[t] * np.outer(v64[t], k64[t]) @ tail
        outs.append(S @ q64[tt - 1])
    return np.array(outs), S.T


def check_unrolled_products():
    rng = np.random.default_rng(7)
    for T, dk, dv in ((1, 3, 2), (5, 5, 3), (8, 4, 6)):
        q, k, v, g, beta, M0 = _rand_inputs(rng, 1, 1, T, dk, dv, unit=False)
        out, fin = oracle.fwd(q, k, v, g, beta, 0.7, M0)
        ref_o, ref_M = _unrolled(q[0, 0], k[0, 0], v[0, 0], g[0, 0], beta[0, 0], 0.7, M0[0, 0])
        assert np.allclose(out[0, 0], ref_o, rtol=1e-12, atol=1e-12)
        assert np.allclose(fin[0, 0], ref_M, rtol=1e-12, atol=1e-12)


def _hadamard(n):
    Hm = np.array([[1.0]])
    while Hm.shape[0] < n:
        Hm = np.block([[Hm, Hm], [Hm, -Hm]])
    return Hm / math.sqrt(n)      # n = 4**m gives exact binary entries


def check_orthonormal_write_read():
    rng = np.random.default_rng(3)
    dk, dv = 16, 5
    basis = _hadamard(dk)                           # entries +-1/4: exactly orthonormal
    perm = rng.permutation(dk)
    for T in (3, 16):
        k = basis[perm[:T]].astype(np.float32)[None, None]
        v = rng.standard_normal((1, 1, T, dv)).astype(np.float32)
        q = k.copy()                                # read back each key as it is written
        g = rng.standard_normal((1, 1, T)).astype(np.float32)
        beta = np.ones((1, 1, T), np.float32)
        M0 = rng.standard_normal((1, 1, dk, dv)).astype(np.float32)
        out, fin = oracle.fwd(q, k, v, g, beta, 1.0, M0)   # a_min = 1: alpha == 1
        S = fin[0, 0].T
        for i in range(T):
            assert np.allclose(S @ k[0, 0, i], v[0, 0, i], atol=1e-13), (T, i)
            assert np.allclose(out[0, 0, i], v[0, 0, i], atol=1e-13), (T, i)
        # directions never written keep what the initial state returned
        for i in perm[T:]:
            x = basis[i]
            assert np.allclose(S @ x, M0[0, 0].astype(np.float64).T @ x, atol=1e-12)


def check_beta_zero_is_pure_decay():
    rng = np.random.default_rng(11)
    q, k, v, g, beta, M0 = _rand_inputs(rng, 1, 2, 37, 6, 4)
    beta[:] = 0.0
    a_min = 0.8
    out, fin = oracle.fwd(q, k, v, g, beta, a_min, M0)
    al = oracle.alpha(g.astype(np.float64), a_min)
    gam = np.cumprod(al, axis=-1)                  # gamma_t = prod_{s<=t} alpha_s
    for h in range(2):
        M = M0[0, h].astype(np.float64)
        assert np.allclose(fin[0, h], gam[0, h, -1] * M, rtol=1e-12, atol=1e-14)
        ref = gam[0, h][:, None] * (q[0, h].astype(np.float64) @ M)
        assert np.allclose(out[0, h], ref, rtol=1e-12, atol=1e-14)
    out0, fin0 = oracle.fwd(q, k, v, g, beta, a_min, None)
    assert not out0.any() and not fin0.any()


def check_a_min_one_ignores_g():
    rng = np.random.default_rng(5)
    q, k, v, g, beta, M0 = _rand_inputs(rng, 1, 1, 20, 8, 8)
    out1, fin1 = oracle.fwd(q, k, v, g, beta, 1.0, M0)
    out2, fin2 = oracle.fwd(q, k, v, -3.0 * g + 1.0, beta, 1.0, M0)
    assert np.array_equal(out1, out2) and np.array_equal(fin1, fin2)
    ref_o, ref_M = _unrolled(q[0, 0, :6], k[0, 0, :6], v[0, 0, :6], g[0, 0, :6],
                             beta[0, 0, :6], 1.0, M0[0, 0])
    o6, f6 = oracle.fwd(q[..., :6, :], k[..., :6, :], v[..., :6, :], g[..., :6],
                        beta[..., :6], 1.0, M0)
    assert np.allclose(o6[0, 0], ref_o, rtol=1e-12, atol=1e-12)
    assert np.allclose(f6[0, 0], ref_M, rtol=1e-12, atol=1e-12)


def check_chunkwise_agrees():
    rng = np.random.default_rng(21)
    for (T, C, dk, dv, init) in ((100, 8, 16, 8, True), (256, 64, 32, 32, False),
                                 (65, 64, 16, 16, True), (9, 1, 4, 4, True)):
        q, k, v, g, beta, M0 = _rand_inputs(rng, 1, 2, T, dk, dv, init=init)
        out, fin = oracle.fwd(q, k, v, g, beta, 0.9, M0)
        oc, fc = chunkwise.fwd(q, k, v, g, beta, 0.9, M0, C=C)
        assert np.max(np.abs(out - oc)) < 1e-11, (T, C, np.max(np.abs(out - oc)))
        assert np.max(np.abs(fin - fc)) < 1e-11, (T, C)


def check_split_resume_and_decode():
    rng = np.random.default_rng(8)
    T, T1 = 50, 21
    q, k, v, g, beta, M0 = _rand_inputs(rng, 2, 2, T, 8, 6)
    out, fin = oracle.fwd(q, k, v, g, beta, 0.85, M0)
    o1, f1 = oracle.fwd(q[:, :, :T1], k[:, :, :T1], v[:, :, :T1], g[:, :, :T1],
                        beta[:, :, :T1], 0.85, M0)
    o2, f2 = oracle.fwd(q[:, :, T1:], k[:, :, T1:], v[:, :, T1:], g[:, :, T1:],
                        beta[:, :, T1:], 0.85, f1.astype(np.float32))
    # the hand-off state is rounded to fp32 (the library's state dtype)
    assert np.allclose(out[:, :, :T1], o1, rtol=0, atol=0)
    assert np.allclose(out[:, :, T1:], o2, rtol=1e-6, atol=1e-6)
    # decode: one token per call, in place, equals the forward over the same tokens
    st = M0.astype(np.float64).copy()
    for t in range(T):
        o = oracle.decode(q[:, :, t], k[:, :, t], v[:, :, t], g[:, :, t], beta[:, :, t],
                          0.85, st)
        assert np.allclose(o, out[:, :, t], rtol=1e-13, atol=1e-13)
    assert np.allclose(st, fin, rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------- the log-domain decay
# The pages' own form of the bound: log alpha = g_min sigmoid(g), g_min = -5 on 16-token
# tiles ('Trillion-Parameter MoE Multimodal LLMs: How to Evaluate the New Generation',
# 3.1; 'What a Trillion-Parameter MoE Model Reveals About the Next Stage of LLM Scaling',
# 3.2).  Its pins: the limits and the symmetry of the sigmoid, the two limits of g
# reproduced by the (separately pinned) linear-domain oracle, and the chunked algebra
# on 16-token chunks at the pages' floor.

def check_log_alpha_limits():
    for g_min in (-5.0, -1.0, -0.25):
        a = oracle.alpha(np.array([0.0, 40.0, -40.0, 1.0, -1.0]), g_min, "log")
        assert abs(a[0] - math.exp(g_min / 2.0)) < 1e-15          # sigmoid(0) = 1/2
        assert abs(a[1] - math.exp(g_min)) < 1e-15                # g -> +inf: the floor e^g_min
        assert abs(a[2] - 1.0) < 1e-15                            # g -> -inf: no decay
        assert a[4] > a[0] > a[3]                                  # decreasing in g
        assert abs(math.log(a[3]) + math.log(a[4]) - g_min) < 1e-14   # s(x) + s(-x) = 1


def check_log_decay_limits_match_linear_form():
    # g -> +inf: alpha = e^g_min, which the linear form gives at its floor (g -> -inf,
    # a_min = e^g_min); g -> -inf: alpha = 1, the linear form with a_min = 1
    rng = np.random.default_rng(33)
    q, k, v, _, beta, M0 = _rand_inputs(rng, 1, 2, 40, 8, 6)
    up, down = np.full((1, 2, 40), 40.0, np.float32), np.full((1, 2, 40), -40.0, np.float32)
    for g_min in (-5.0, -0.5):
        o_log, f_log = oracle.fwd(q, k, v, up, beta, g_min, M0, decay="log")
        o_lin, f_lin = oracle.fwd(q, k, v, down, beta, math.exp(g_min), M0)
        assert np.max(np.abs(o_log - o_lin)) < 1e-12 and np.max(np.abs(f_log - f_lin)) < 1e-12
    o_log, f_log = oracle.fwd(q, k, v, down, beta, -5.0, M0, decay="log")
    o_lin, f_lin = oracle.fwd(q, k, v, up, beta, 1.0, M0)
    assert np.max(np.abs(o_log - o_lin)) < 1e-12 and np.max(np.abs(f_log - f_lin)) < 1e-12
    # and the decode step takes the same decay
    st = M0.astype(np.float64).copy()
    o = oracle.decode(q[:, :, 0], k[:, :, 0], v[:, :, 0], up[:, :, 0], beta[:, :, 0], -5.0,
                      st, decay="log")
    o1, f1 = oracle.fwd(q[:, :, :1], k[:, :, :1], v[:, :, :1], up[:, :, :1], beta[:, :, :1],
                        -5.0, M0, decay="log")
    assert np.max(np.abs(o - o1[:, :, 0])) < 1e-13 and np.max(np.abs(st - f1)) < 1e-13


def check_log_chunkwise_agrees():
    # 16-token chunks at the pages' floor g_min = -5: in-chunk decay down to e^-80
    rng = np.random.default_rng(44)
    for (T, C, g_min) in ((70, 16, -5.0), (64, 16, -2.0), (33, 64, -1.25)):
        q, k, v, g, beta, M0 = _rand_inputs(rng, 1, 2, T, 16, 8)
        out, fin = oracle.fwd(q, k, v, g, beta, g_min, M0, decay="log")
        oc, fc = chunkwise.fwd(q, k, v, g, beta, g_min, M0, C=C, decay="log")
        scale = max(1.0, float(np.max(np.abs(out))))
        assert np.max(np.abs(out - oc)) < 1e-9 * scale, (T, C, np.max(np.abs(out - oc)))
        assert np.max(np.abs(fin - fc)) < 1e-9 * scale, (T, C)


# ---- the backward: gradients of L = <d_out, out> + <d_final, final_state>

def _loss(args, dout, dfin, bound, decay):
    out, fin = oracle.fwd(*args[:5], bound, args[5], decay=decay)
    return float((out * dout).sum() + (fin * dfin).sum())


def _bwd_case(rng, T, dk, dv, bound, decay):
    q, k, v, g, beta, M0 = _rand_inputs(rng, 1, 1, T, dk, dv)
    dout = rng.standard_normal((1, 1, T, dv)).astype(np.float32)
    dfin = rng.standard_normal((1, 1, dk, dv)).astype(np.float32)
    return [q, k, v, g, beta, M0], dout, dfin


def check_bwd_finite_differences():
    # every gradient element against a central difference of the forward loss (fp32
    # inputs perturbed by 2^-10, the exact perturbation as denominator); one case
    # crosses the 64-token replay boundary, both decay forms
    rng = np.random.default_rng(61)
    for (T, dk, dv, bound, decay) in ((5, 3, 4, 0.9, "affine"), (6, 2, 3, -2.0, "log"),
                                      (70, 2, 2, 0.8, "affine")):
        args, dout, dfin = _bwd_case(rng, T, dk, dv, bound, decay)
        grads = oracle.bwd(*args[:5], bound, args[5], dout, dfin, decay=decay)
        for n, (a, gr) in enumerate(zip(args, grads)):
            flat = a.reshape(-1)
            fd = np.empty(flat.size)
            for idx in range(flat.size):
                x0 = flat[idx]
                flat[idx] = x0 + np.float32(2.0 ** -10)
                lp = _loss(args, dout, dfin, bound, decay)
                xp = float(flat[idx])
                flat[idx] = x0 - np.float32(2.0 ** -10)
                lm = _loss(args, dout, dfin, bound, decay)
                xm = float(flat[idx])
                flat[idx] = x0
                fd[idx] = (lp - lm) / (xp - xm)
            err = np.max(np.abs(fd - gr.reshape(-1))) / max(1e-30, np.max(np.abs(fd)))
            assert err < 1e-5, (T, decay, n, err)


def check_bwd_exact_in_linear_inputs():
    # L is exactly linear in q, in v and in the initial state (each alone): a finite
    # step of any size changes L by exactly <grad, step>
    rng = np.random.default_rng(62)
    args, dout, dfin = _bwd_case(rng, 40, 8, 6, 0.85, "affine")
    grads = oracle.bwd(*args[:5], 0.85, args[5], dout, dfin)
    l0 = _loss(args, dout, dfin, 0.85, "affine")
    for n in (0, 2, 5):
        step = rng.standard_normal(args[n].shape).astype(np.float32)
        moved = list(args)
        moved[n] = (args[n] + step).astype(np.float32)
        actual = moved[n].astype(np.float64) - args[n].astype(np.float64)
        dl = _loss(moved, dout, dfin, 0.85, "affine") - l0
        pred = float((grads[n] * actual).sum())
        assert abs(dl - pred) < 1e-10 * max(1.0, abs(dl)), (n, dl, pred)


def check_bwd_zero_cotangent_and_pure_decay():
    # no cotangent gives zero gradients; with beta = 0 and only d_final, the state is
    # pure decay M_T = prod(alpha) M_0: dinit = prod(alpha) d_final exactly, and
    # dv = 0 (beta scales every write)
    rng = np.random.default_rng(63)
    args, dout, dfin = _bwd_case(rng, 9, 4, 5, 0.7, "affine")
    for gr in oracle.bwd(*args[:5], 0.7, args[5], None, None):
        assert not np.any(gr)
    args[4] = np.zeros_like(args[4])
    gq, gk, gv, gg, gb, gi = oracle.bwd(*args[:5], 0.7, args[5], None, dfin)
    pa = float(np.prod(oracle.alpha(args[3].reshape(-1), 0.7)))
    assert np.allclose(gi, pa * dfin.astype(np.float64), rtol=1e-13, atol=0)
    assert not np.any(gv) and not np.any(gq)


ALL_CHECKS = [check_alpha_limits, check_hand_worked, check_unrolled_products,
              check_orthonormal_write_read, check_beta_zero_is_pure_decay,
              check_a_min_one_ignores_g, check_chunkwise_agrees,
              check_split_resume_and_decode, check_log_alpha_limits,
              check_log_decay_limits_match_linear_form, check_log_chunkwise_agrees,
              check_bwd_finite_differences, check_bwd_exact_in_linear_inputs,
              check_bwd_zero_cotangent_and_pure_decay]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check()


# ----------------------------------------------------------------- decay / range facts

def test_pages_range_facts():
    fx = json.load(open(os.path.join(GOLDEN, "range_facts.json")))
    values = {"exp(-80)": math.exp(-80.0), "exp(80)": math.exp(80.0), "exp(-5)": math.exp(-5.0),
              "float32_tiny": float(np.finfo(np.float32).tiny),
              "float32_max": float(np.finfo(np.float32).max)}
    for f in fx["facts"]:
        got = values[f["expr"]]
        assert abs(got - f["printed"]) <= f["rel_tol"] * f["printed"], (f["name"], got)
    # the argument itself: 16 steps at the floor stay inside the fp32 normal range
    worst = fx["tile_tokens"] * fx["log_decay_floor"]
    assert math.exp(worst) > np.finfo(np.float32).tiny
    assert math.exp(-worst) < np.finfo(np.float32).max


@pytest.mark.parametrize("g_min,C", [(-5.0, 16), (-1.25, 64)])
def test_log_chunk_decay_bounds(g_min, C):
    # the pages' range argument: with log alpha >= g_min, a C-row chunk keeps gamma >=
    # e^(C g_min) >= e^-80 and 1/gamma <= e^80, both normal fp32 numbers
    g = np.concatenate([np.full(70, 60.0), np.random.default_rng(1).normal(0, 3, 300)])
    b, gam, inv = chunkwise.chunk_decay(g, g_min, C, decay="log")
    r = (np.arange(len(g)) % C) + 1
    assert np.all(gam <= 1.0) and np.all(gam >= np.exp(g_min * r) * (1 - 1e-12))
    assert np.all(inv <= math.exp(-g_min * C) * (1 + 1e-12)) and C * -g_min <= 80.0
    assert np.all(np.isfinite(np.float32(inv))) and np.all(np.float32(gam) > 0)


@pytest.mark.parametrize("a_min,C", [(0.9, 64), (0.95, 64), (0.98, 64), (0.99, 64), (0.3, 64)])
def test_chunk_decay_bounds(a_min, C):
    g = np.concatenate([np.full(70, -60.0), np.random.default_rng(0).normal(0, 3, 300)])
    b, gam, inv = chunkwise.chunk_decay(g, a_min, C)
    r = (np.arange(len(g)) % C) + 1
    assert np.all(gam <= 1.0) and np.all(gam >= a_min ** r * (1 - 1e-12))
    assert np.all(inv <= a_min ** (-C) * (1 + 1e-12))
    assert np.all(np.isfinite(np.float32(inv)))          # finite in fp32
    assert np.all(np.float32(gam) > 0)                   # no underflow to zero in fp32


def test_rel_l2():
    x = np.array([3.0, 4.0])
    assert oracle.rel_l2(x, x) == 0.0
    assert abs(oracle.rel_l2(x + np.array([0.3, 0.4]), x) - 0.1) < 1e-15


# ----------------------------------------------------------------- planted mistakes

MUTANTS = [
    ("alpha dropped on the kept state", "*s = a * (*s - b * uj * ki) + b * vj * ki;",
     "*s = (*s - b * uj * ki) + b * vj * ki;"),
    ("alpha also on the write", "*s = a * (*s - b * uj * ki) + b * vj * ki;",
     "*s = a * (*s - b * uj * ki + b * vj * ki);"),
    ("wrong sign of the correction", "*s = a * (*s - b * uj * ki) + b * vj * ki;",
     "*s = a * (*s + b * uj * ki) + b * vj * ki;"),
    ("beta dropped on the write", "*s = a * (*s - b * uj * ki) + b * vj * ki;",
     "*s = a * (*s - b * uj * ki) + vj * ki;"),
    ("u read with q instead of k", "acc += S[(int64_t)j * dk + i] * (double)kt[i];",
     "acc += S[(int64_t)j * dk + i] * (double)qt[i];"),
    ("output read with k instead of q", "acc += S[(int64_t)j * dk + i] * (double)qt[i];",
     "acc += S[(int64_t)j * dk + i] * (double)kt[i];"),
    ("initial state not transposed",
     "S[(int64_t)j * dk + i] = init ? (double)init[(int64_t)i * dv + j] : 0.0;",
     "S[(int64_t)j * dk + i] = init ? (double)init[(int64_t)j * dk + i] : 0.0;"),
    ("final state not transposed", "final_state[(int64_t)i * dv + j] = S[(int64_t)j * dk + i];",
     "final_state[(int64_t)i * dv + j] = S[(int64_t)i * dk + j];"),
    ("sigmoid sign flipped", "(1.0 + exp(-g))", "(1.0 + exp(g))"),
    ("floor and range swapped", "return a_min + (1.0 - a_min) / (1.0 + exp(-g));",
     "return (1.0 - a_min) + a_min / (1.0 + exp(-g));"),
    ("decode: alpha dropped", "*s = a * (*s - b * uj * ki) + b * vj * ki;",
     "*s = (*s - b * uj * ki) + b * vj * ki;"),
    ("log form: sign of the floor flipped", "return exp(g_min / (1.0 + exp(-g)));",
     "return exp(-g_min / (1.0 + exp(-g)));"),
    ("log form: sigmoid flipped", "return exp(g_min / (1.0 + exp(-g)));",
     "return exp(g_min / (1.0 + exp(g)));"),
    ("log form: exponential dropped", "return exp(g_min / (1.0 + exp(-g)));",
     "return 1.0 + g_min / (1.0 + exp(-g));"),
    ("log form ignored by the forward", "return decay == 1 ? gdr_oracle_alpha_log(g, bound)",
     "return decay == 2 ? gdr_oracle_alpha_log(g, bound)"),
    ("bwd: query gradient read from S_{t-1}", "acc += St[(int64_t)j * dk + i] * (double)dot[j];",
     "acc += Sp[(int64_t)j * dk + i] * (double)dot[j];"),
    ("bwd: state gradient not decayed",
     "G[(int64_t)j * dk + i] = a * G[(int64_t)j * dk + i] + du[j] * (double)kt[i];",
     "G[(int64_t)j * dk + i] = G[(int64_t)j * dk + i] + du[j] * (double)kt[i];"),
    ("bwd: correction path dropped from the key gradient",
     "acc += G[(int64_t)j * dk + i] * w[j] + Sp[(int64_t)j * dk + i] * du[j];",
     "acc += G[(int64_t)j * dk + i] * w[j];"),
    ("bwd: sign of the decay's correction term", "dalpha -= b * dw[j] * u[j];",
     "dalpha += b * dw[j] * u[j];"),
    ("bwd: output cotangent not fed into the state",
     "G[(int64_t)j * dk + i] += (double)dot[j] * (double)qt[i];",
     "G[(int64_t)j * dk + i] += 0.0 * (double)qt[i];"),
    ("bwd: log-form derivative without alpha",
     "return gdr_oracle_alpha_log(g, bound) * bound * s * (1.0 - s);",
     "return bound * s * (1.0 - s);"),
    ("bwd: replay from the previous checkpoint", "memcpy(st, ck + sg * SZ,",
     "memcpy(st, ck + (sg > 0 ? sg - 1 : 0) * SZ,"),
]


@contextlib.contextmanager
def _oracle_lib(path):
    lib = ctypes.CDLL(path)
    saved = oracle._load()
    for name in ("gdr_oracle_alpha", "gdr_oracle_alpha_log", "gdr_oracle_fwd", "gdr_oracle_decode",
                 "gdr_oracle_bwd"):
        getattr(lib, name).restype = getattr(saved, name).restype
        getattr(lib, name).argtypes = getattr(saved, name).argtypes
    oracle._lib = lib
    try:
        yield
    finally:
        oracle._lib = saved


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistakes(mutant, tmp_path):
    name, old, new = mutant
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gdr_oracle.c")).read()
    bwd_at = src.index("/* ------------------------------------------------------------------ backward")
    if "decode" in name:
        # only the copy inside the decode step
        idx = src.index("static void oracle_decode_one")
        assert old in src[idx:bwd_at], name
        src = src[:idx] + src[idx:].replace(old, new, 1)
    elif name.startswith("bwd:"):
        assert old in src[bwd_at:], name
        src = src[:bwd_at] + src[bwd_at:].replace(old, new)
    else:
        # the forward loop (the backward replays its own copy of the step)
        assert old in src[:bwd_at], name
        src = src[:bwd_at].replace(old, new) + src[bwd_at:]
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "mutant.so"
    c_path.write_text(src)
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-std=c11", "-o", str(so_path),
                    str(c_path), "-lm", "-lpthread"], check=True)
    caught = []
    with _oracle_lib(str(so_path)):
        for check in ALL_CHECKS:
            try:
                check()
            except AssertionError:
                caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake: {name}"
