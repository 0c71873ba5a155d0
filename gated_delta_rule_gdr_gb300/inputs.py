"""Seeded synthetic inputs for the gated delta rule workloads.

This module is shared by the tests, the benchmark and the oracle checks.  It
holds the input *recipe* only -- distributions, shapes and seeds -- and none
of the method's arithmetic (no decay, no recurrence).

Recipe (one per workload, all drawn with torch's generator on the requested
device, one generator per tensor seeded from (seed, tensor id)):

* q, k ~ N(0, 1) in fp32, L2-normalised per token and head in fp32, then cast
  to the compute dtype (bf16 values are what both the kernels and the oracle
  receive; their norms are ~1, not exactly 1).
* v ~ N(0, 1), cast to the compute dtype.
* beta = sigmoid(N(0, 1)) in fp32 -- the write strength in (0, 1).
* g ~ N(g_mean, 1) in fp32 -- the raw decay logit (g_mean = 2 for the long
  prefill so that alpha stays close to 1).
* init_state ~ N(0, init_std) fp32 [B,H,dk,dv] (standard deviation 0.02) where
  the workload says so, else None (zero state).

Decode draws fresh q, k, v, g, beta every step from a seed derived from
(seed, step); its starting state is N(0, 0.02).

The backward takes cotangents: d_out ~ N(0, 1) in the compute dtype [B,H,T,dv] and
d_final ~ N(0, 1) fp32 [B,H,dk,dv] (``cotangents``).

Gated multi-head latent attention, one decode step (``mla_inputs``): the absorbed
query q_abs ~ N(0, 1) bf16 [N,H,dc], the latent cache ckv ~ N(0, 1) bf16 [N,L,dc]
(unit-variance latents, as after a normalisation), the value up-projection
w_uv ~ N(0, 1/dc) bf16 [H,dh,dc] (fan-in scaled), the gate's pre-activation
z ~ N(0, 1) fp32 [N,H,dh], cache lengths L for every sequence or (ragged) uniform in
[1, L], and the score scale 1/sqrt(dh).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import math

import torch

_TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "g": 4, "beta": 5, "init": 6, "lengths": 7,
               "d_out": 8, "d_final": 9, "q_abs": 10, "ckv": 11, "w_uv": 12, "gate": 13,
               "seqlens": 14}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    chunk: int
    dtype: str            # "f32" or "bf16": dtype of q, k, v and out
    a_min: float
    g_mean: float = 0.0
    init_std: float | None = None   # None -> zero initial state
    final_state: bool = True
    seed: int = 0
    steps: int = 0        # decode workloads only: number of single-token steps

    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the gated-delta-rule hot path (prefill shapes are
# [B, H, T, d]; decode is N sequences x H heads, one token per step).
CORRECTNESS = Workload("correctness_b1h2t256_d64_f32", 1, 2, 256, 64, 64, 64, "f32", 0.9)
PREFILL = Workload("prefill_b4h16t4096_d128_bf16", 4, 16, 4096, 128, 128, 64, "bf16", 0.95,
                   init_std=0.02)
LONG_PREFILL = Workload("long_prefill_b1h32t65536_d128_bf16", 1, 32, 65536, 128, 128, 64,
                        "bf16", 0.98, g_mean=2.0)
MILLION_PREFILL = Workload("million_prefill_b1h16t1048576_d128_bf16", 1, 16, 1048576, 128,
                           128, 64, "bf16", 0.99)
DECODE = Workload("decode_n256h32_d128_bf16_64steps", 256, 32, 1, 128, 128, 64, "bf16", 0.95,
                  init_std=0.02, steps=64)

# Packed variable-length prefill (the serving shape): B = 32 sequences, H = 16, lengths
# log-uniform in [16, T] (``varlen_lengths``), everything else as the prefill workload.
VARLEN = Workload("varlen_s32h16_len16to4096_d128_bf16", 32, 16, 4096, 128, 128, 64, "bf16", 0.95,
                  init_std=0.02)

WORKLOADS = {w.name: w for w in (CORRECTNESS, PREFILL, LONG_PREFILL, MILLION_PREFILL, DECODE,
                                 VARLEN)}


def _gen(device, seed: int, tensor: str, extra: int = 0) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed((seed * 1_000_003 + _TENSOR_IDS[tensor] * 7919 + extra * 104729)
                    & 0x7FFF_FFFF_FFFF_FFFF)
    return gen


def _unit_rows(shape, device, gen, dtype):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    return x.to(dtype)


def prefill_inputs(w: Workload, device="cpu"):
    """Returns dict(q, k, v, g, beta, init_state) for a prefill workload."""
    dt = w.torch_dtype()
    B, H, T = w.B, w.H, w.T
    q = _unit_rows((B, H, T, w.dk), device, _gen(device, w.seed, "q"), dt)
    k = _unit_rows((B, H, T, w.dk), device, _gen(device, w.seed, "k"), dt)
    v = torch.randn((B, H, T, w.dv), generator=_gen(device, w.seed, "v"), device=device,
                    dtype=torch.float32).to(dt)
    g = torch.randn((B, H, T), generator=_gen(device, w.seed, "g"), device=device,
                    dtype=torch.float32) + w.g_mean
    beta = torch.sigmoid(torch.randn((B, H, T), generator=_gen(device, w.seed, "beta"),
                                     device=device, dtype=torch.float32))
    init = None
    if w.init_std is not None:
        init = torch.randn((B, H, w.dk, w.dv), generator=_gen(device, w.seed, "init"),
                           device=device, dtype=torch.float32) * w.init_std
    return dict(q=q, k=k, v=v, g=g, beta=beta, init_state=init)


def decode_state(w: Workload, device="cpu"):
    """Starting fp32 state [N,H,dk,dv] of a decode workload."""
    std = 0.02 if w.init_std is None else w.init_std
    return torch.randn((w.B, w.H, w.dk, w.dv), generator=_gen(device, w.seed, "init"),
                       device=device, dtype=torch.float32) * std


def decode_step_inputs(w: Workload, step: int, device="cpu"):
    """Fresh q, k, v [N,H,d], g, beta [N,H] for decode step ``step``."""
    dt = w.torch_dtype()
    N, H = w.B, w.H
    q = _unit_rows((N, H, w.dk), device, _gen(device, w.seed, "q", step + 1), dt)
    k = _unit_rows((N, H, w.dk), device, _gen(device, w.seed, "k", step + 1), dt)
    v = torch.randn((N, H, w.dv), generator=_gen(device, w.seed, "v", step + 1),
                    device=device, dtype=torch.float32).to(dt)
    g = torch.randn((N, H), generator=_gen(device, w.seed, "g", step + 1), device=device,
                    dtype=torch.float32) + w.g_mean
    beta = torch.sigmoid(torch.randn((N, H), generator=_gen(device, w.seed, "beta", step + 1),
                                     device=device, dtype=torch.float32))
    return dict(q=q, k=k, v=v, g=g, beta=beta)


def varlen_inputs(w: Workload, lengths, device="cpu"):
    """Packed variable-length prefill inputs: sequence s has ``lengths[s]`` tokens,
    drawn as ``prefill_inputs`` of ``w`` with B = 1, T = lengths[s] and its own seed.
    Returns dict(q, k, v [total_T,H,d], g, beta [total_T,H], init_state [S,H,dk,dv] or
    None, cu_seqlens int32 [S+1], seqs = the per-sequence dense dicts [1,H,T,...])."""
    seqs = [prefill_inputs(w.with_(B=1, T=int(n), seed=w.seed * 1000 + s + 1), device)
            for s, n in enumerate(lengths)]
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))

    def pack(name):   # [1,H,T,...] per sequence -> [total_T,H,...]
        return torch.cat([x[name][0].transpose(0, 1) for x in seqs], 0).contiguous()

    init = None
    if w.init_std is not None:
        init = torch.cat([x["init_state"] for x in seqs], 0).contiguous()
    return dict(q=pack("q"), k=pack("k"), v=pack("v"), g=pack("g"), beta=pack("beta"),
                init_state=init, cu_seqlens=torch.tensor(cu, dtype=torch.int32, device=device),
                seqs=seqs)


def varlen_lengths(w: Workload):
    """Seeded sequence lengths of a packed workload: w.B values, log-uniform in [16, w.T]."""
    u = torch.rand(w.B, generator=_gen("cpu", w.seed, "lengths"), dtype=torch.float64)
    lo, hi = math.log(16.0), math.log(float(w.T))
    return [int(round(math.exp(lo + (hi - lo) * float(x)))) for x in u]


def cotangents(w: Workload, device="cpu"):
    """Returns dict(d_out, d_final): the gradients of a loss with respect to the
    prefill's output and final state, for the backward."""
    d_out = torch.randn((w.B, w.H, w.T, w.dv), generator=_gen(device, w.seed, "d_out"),
                        device=device, dtype=torch.float32).to(w.torch_dtype())
    d_final = torch.randn((w.B, w.H, w.dk, w.dv), generator=_gen(device, w.seed, "d_final"),
                          device=device, dtype=torch.float32)
    return dict(d_out=d_out, d_final=d_final)


@dataclass(frozen=True)
class MlaWorkload:
    """One decode step of gated multi-head latent attention: N sequences, H heads, a
    latent cache of up to L tokens of dc values per sequence, dh values per head after
    the value up-projection."""
    name: str
    N: int
    H: int
    L: int
    dc: int
    dh: int
    ragged: bool = False      # cache lengths uniform in [1, L] instead of all L
    seed: int = 0

    def with_(self, **kw) -> "MlaWorkload":
        return replace(self, **kw)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dh)


MLA_DECODE = MlaWorkload("mla_decode_n32h64_l32768_dc512_dh128_bf16", 32, 64, 32768, 512, 128)


def mla_inputs(w: MlaWorkload, device="cpu"):
    """Returns dict(q_abs, ckv, w_uv, gate, seqlens) for a latent-attention decode step."""
    q_abs = torch.randn((w.N, w.H, w.dc), generator=_gen(device, w.seed, "q_abs"), device=device,
                        dtype=torch.float32).to(torch.bfloat16)
    ckv = torch.randn((w.N, w.L, w.dc), generator=_gen(device, w.seed, "ckv"), device=device,
                      dtype=torch.float32).to(torch.bfloat16)
    w_uv = (torch.randn((w.H, w.dh, w.dc), generator=_gen(device, w.seed, "w_uv"), device=device,
                        dtype=torch.float32) / math.sqrt(w.dc)).to(torch.bfloat16)
    gate = torch.randn((w.N, w.H, w.dh), generator=_gen(device, w.seed, "gate"), device=device,
                       dtype=torch.float32)
    if w.ragged:
        lens = torch.randint(1, w.L + 1, (w.N,), generator=_gen("cpu", w.seed, "seqlens"),
                             dtype=torch.int32)
    else:
        lens = torch.full((w.N,), w.L, dtype=torch.int32)
    return dict(q_abs=q_abs, ckv=ckv, w_uv=w_uv, gate=gate, seqlens=lens.to(device))
