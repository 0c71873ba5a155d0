"""GPU parity: libgdr.so (through its C ABI) against the fp64 oracle on the same
seeded inputs.  Tolerances are relative L2 over the whole tensor: 1e-5 for the
fp32 path, 5e-3 for the bf16 paths, for outputs and final states alike."""
from __future__ import annotations

import contextlib

import numpy as np
import pytest
import torch

import oracle
from oracle import chunkwise
import gated_delta_rule_gdr_gb300 as gdr
from gated_delta_rule_gdr_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 5e-3}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdr.load(build_if_missing=True)
    yield
    assert gdr.last_device_error() == 0


def rel(x, ref):
    return oracle.rel_l2(x, ref)


def run_gpu(x, w, init=None, chunk=None, workspace="auto"):
    out, fin = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min,
                             x["init_state"] if init is None else init,
                             chunk=chunk or w.chunk, workspace=workspace)
    torch.cuda.synchronize()
    return out, fin


def to(x, device):
    return {k_: (None if t is None else t.to(device)) for k_, t in x.items()}


# The kernels of the bf16, d = 128, chunk 64 prefill: the single-launch fused kernel
# with one CTA per head ("single") or a two-CTA cluster per head ("pair"), and the
# two-kernel path (preparation, then the chain kernel) with two CTAs per head
# ("chain2") or one ("chain1").  Value: (library options, workspace argument).
VARIANTS = {"single": ({"fused_variant": 1}, None),
            "pair": ({"fused_variant": 2}, None),
            "chain2": ({"chain_split": 2}, "auto"),
            "chain1": ({"chain_split": 1}, "auto")}


@contextlib.contextmanager
def path_variant(name):
    """Force one of VARIANTS (by default the launchers pick by the number of
    heads); yields the workspace argument that selects its path."""
    opts, ws = VARIANTS[name]
    with gdr.option(**opts):
        yield ws


# ------------------------------------------------------------------ the correctness workload
# workspace "auto": the staged kernels on a caller-owned workspace (gdr_chunk_fwd_ws);
# None: the one-pass kernel of gdr_chunk_fwd, which allocates nothing
@pytest.mark.parametrize("workspace", ["auto", None])
def test_correctness_workload_fp32(workspace):
    w = I.CORRECTNESS
    x = to(I.prefill_inputs(w), "cuda")
    expect = 1 if workspace else 6
    assert gdr.chunk_fwd_path(w.B, w.H, w.T, w.dk, w.dv, w.chunk, w.a_min, torch.float32,
                              workspace=bool(workspace)) == expect
    out, fin = run_gpu(x, w, workspace=workspace)
    ro, rf = oracle.fwd(*(x[n].cpu() for n in ("q", "k", "v", "g", "beta")), w.a_min, None)
    assert rel(out, ro) <= TOL["f32"], rel(out, ro)
    assert rel(fin, rf) <= TOL["f32"], rel(fin, rf)


# ------------------------------------------------------------------ per-step parity
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,C,d", [(256, 64, 64), (100, 32, 32), (65, 16, 128)])
def test_staged_steps_match_chunked_algebra(dtype, T, C, d):
    w = I.CORRECTNESS.with_(B=1, H=2, T=T, dk=d, dv=d, chunk=C, dtype=dtype, init_std=0.5)
    x = to(I.prefill_inputs(w), "cuda")
    BH = w.B * w.H
    gamma = gdr.chunk_decay(x["g"], w.a_min, C)
    U, Wk = gdr.chunk_wy(x["k"], x["v"], x["beta"], gamma, C)
    W, Mn, fin = gdr.chunk_state(x["k"], gamma, U, Wk, x["init_state"], C)
    out = gdr.chunk_output(x["q"], x["k"], gamma, Mn, W, C)
    torch.cuda.synchronize()
    tol = 2e-6 if dtype == "f32" else 2e-6   # steps compute in fp32 on exact inputs
    for h in range(BH):
        b_, h_ = divmod(h, w.H)
        args = [x[n][b_, h_].float().cpu().numpy() for n in ("q", "k", "v")]
        ref_o, ref_M, inter = chunkwise.head(*args, x["g"][b_, h_].cpu().numpy(),
                                             x["beta"][b_, h_].cpu().numpy(), w.a_min,
                                             x["init_state"][b_, h_].cpu().numpy(), C, keep=True)
        assert rel(gamma[b_, h_], np.concatenate(inter["gamma"])) <= tol
        assert rel(U[b_, h_], np.concatenate(inter["U"])) <= 1e-5
        assert rel(Wk[b_, h_], np.concatenate(inter["Wk"])) <= 1e-5
        assert rel(W[b_, h_], np.concatenate(inter["W"])) <= 1e-5
        assert rel(Mn[b_, h_], np.stack(inter["M"])) <= 1e-5
        assert rel(fin[b_, h_], ref_M) <= 1e-5
        assert rel(out[b_, h_], ref_o) <= (1e-5 if dtype == "f32" else TOL["bf16"])


def test_decay_bounds_on_device():
    g = torch.cat([torch.full((1, 1, 70), -80.0), torch.full((1, 1, 58), 60.0),
                   torch.randn(1, 1, 128) * 4], dim=-1).cuda()
    for a_min in (0.3, 0.9, 0.99):
        gam = gdr.chunk_decay(g, a_min, 64).cpu().double().numpy().ravel()
        r = (np.arange(gam.size) % 64) + 1
        assert np.all(gam <= 1.0 + 1e-7)
        assert np.all(gam >= a_min ** r * (1 - 1e-5))
        assert np.all(np.isfinite(1.0 / gam.astype(np.float32)))


# ------------------------------------------------------------------ edge cases
@pytest.mark.parametrize("workspace", ["auto", None])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 100, 200])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_and_tiny(dtype, T, d, workspace):
    w = I.CORRECTNESS.with_(B=1, H=1, T=T, dk=d, dv=d, dtype=dtype, init_std=0.02)
    x = to(I.prefill_inputs(w), "cuda")
    out, fin = run_gpu(x, w, workspace=workspace)
    ro, rf = oracle.fwd(*(x[n].cpu() for n in ("q", "k", "v", "g", "beta")), w.a_min,
                        x["init_state"].cpu())
    assert rel(out, ro) <= TOL[dtype]
    assert rel(fin, rf) <= TOL[dtype]
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("B,H,T", [(1, 1, 1), (1, 2, 63), (2, 1, 64), (1, 3, 65), (2, 2, 200),
                                   (1, 2, 700)])
def test_fused_variants(variant, B, H, T):
    """Every kernel of the bf16, dk = dv = 128, chunk 64 prefill against the oracle:
    ragged tails, one to several input-stage rounds, several heads."""
    w = I.PREFILL.with_(B=B, H=H, T=T)
    x = to(I.prefill_inputs(w), "cuda")
    with path_variant(variant) as ws:
        out, fin = run_gpu(x, w, workspace=ws)
    ro, rf = oracle.fwd(*(x[n].cpu() for n in ("q", "k", "v", "g", "beta")), w.a_min,
                        x["init_state"].cpu())
    assert rel(out, ro) <= TOL["bf16"], rel(out, ro)
    assert rel(fin, rf) <= TOL["bf16"], rel(fin, rf)


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_varlen_packed_sequences(variant):
    """Packed variable-length sequences (empty, 1-token, ragged and multi-chunk ones in
    one launch) against the oracle run on each sequence on its own; the final states
    then feed one decode step, which must equal the oracle's next token."""
    w = I.PREFILL.with_(H=2)
    lengths = [1, 63, 64, 0, 65, 200, 700, 130]
    x = I.varlen_inputs(w, lengths, device="cuda")
    with path_variant(variant) as ws:
        out, fin = gdr.chunk_fwd_varlen(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min,
                                        x["cu_seqlens"], x["init_state"], workspace=ws)
    torch.cuda.synchronize()
    cu = x["cu_seqlens"].tolist()
    ref_out, ref_fin = [], []
    for s, xs in enumerate(x["seqs"]):
        cpu = {n: (None if t is None else t.cpu()) for n, t in xs.items()}
        if lengths[s] == 0:
            ref_fin.append(cpu["init_state"][0].double())
            continue
        ro, rf = oracle.fwd(cpu["q"], cpu["k"], cpu["v"], cpu["g"], cpu["beta"], w.a_min,
                            cpu["init_state"])
        ref_out.append(torch.as_tensor(ro)[0].transpose(0, 1))
        ref_fin.append(torch.as_tensor(rf)[0])
    e_o = rel(out.cpu(), torch.cat(ref_out, 0))
    e_f = rel(fin.cpu(), torch.stack(ref_fin, 0))
    assert e_o <= TOL["bf16"] and e_f <= TOL["bf16"], (e_o, e_f)
    for s in range(len(lengths)):   # every sequence on its own, and the empty one exactly
        if lengths[s]:
            assert rel(out[cu[s]:cu[s + 1]].cpu(), ref_out[sum(1 for t in lengths[:s] if t)]) \
                <= TOL["bf16"]
    assert torch.equal(fin[3], x["init_state"][3])
    # prefill -> decode handoff: one more token per sequence from the varlen final states
    nxt = I.decode_step_inputs(w.with_(B=len(lengths)), 0, device="cuda")
    st = fin.clone()
    o1 = gdr.decode_step(nxt["q"], nxt["k"], nxt["v"], nxt["g"], nxt["beta"], w.a_min, st)
    torch.cuda.synchronize()
    ref_st = torch.stack(ref_fin, 0).numpy().copy()
    r1 = oracle.decode(nxt["q"].cpu(), nxt["k"].cpu(), nxt["v"].cpu(), nxt["g"].cpu(),
                       nxt["beta"].cpu(), w.a_min, ref_st)
    assert rel(o1.cpu(), r1) <= TOL["bf16"]
    assert gdr.last_device_error() == 0   # no bounded wait ran out (e.g. on the empty sequence)


@pytest.mark.parametrize("dtype,d,C", [("f32", 64, 32), ("bf16", 64, 64), ("f32", 128, 16),
                                       ("bf16", 32, 16)])
def test_varlen_one_pass_kernel(dtype, d, C):
    """Packed sequences of fp32 and of the shapes the tensor-core kernels do not take run
    on the one-pass kernel: each sequence against the oracle on its own (fp32 at 1e-5),
    an empty sequence keeps its initial state, and the final states feed a decode step."""
    w = I.CORRECTNESS.with_(H=2, dk=d, dv=d, chunk=C, dtype=dtype, init_std=0.1)
    lengths = [1, C - 1, C, 0, C + 1, 3 * C + 7, 130]
    x = I.varlen_inputs(w, lengths, device="cuda")
    out, fin = gdr.chunk_fwd_varlen(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min,
                                    x["cu_seqlens"], x["init_state"], chunk=C)
    torch.cuda.synchronize()
    cu = x["cu_seqlens"].tolist()
    ref_fin = []
    for s, xs in enumerate(x["seqs"]):
        cpu = {n: (None if t is None else t.cpu()) for n, t in xs.items()}
        if lengths[s] == 0:
            ref_fin.append(cpu["init_state"][0].double())
            assert torch.equal(fin[s], x["init_state"][s])
            continue
        ro, rf = oracle.fwd(cpu["q"], cpu["k"], cpu["v"], cpu["g"], cpu["beta"], w.a_min,
                            cpu["init_state"])
        got = out[cu[s]:cu[s + 1]].transpose(0, 1).unsqueeze(0).cpu()
        assert rel(got, ro) <= TOL[dtype], (s, rel(got, ro))
        assert rel(fin[s:s + 1].cpu(), rf) <= TOL[dtype]
        ref_fin.append(torch.as_tensor(rf)[0])
    nxt = I.decode_step_inputs(w.with_(B=len(lengths)), 0, device="cuda")
    st = fin.clone()
    o1 = gdr.decode_step(nxt["q"], nxt["k"], nxt["v"], nxt["g"], nxt["beta"], w.a_min, st)
    torch.cuda.synchronize()
    ref_st = torch.stack(ref_fin, 0).numpy().copy()
    r1 = oracle.decode(*(nxt[n].cpu() for n in ("q", "k", "v", "g", "beta")), w.a_min, ref_st)
    assert rel(o1.cpu(), r1) <= TOL[dtype]


# ------------------------------------------------------------------ the log-domain decay
# The pages' own bound, log alpha = g_min sigmoid(g) (g_min = -5 on 16-token chunks), on
# the staged kernels; a floor that chunk 64 allows (g_min = -1.25) on the four kernels of
# the bf16, d = 128 prefill; and the decode step.

@pytest.mark.parametrize("dtype,d,T,C,g_min", [("f32", 64, 100, 16, -5.0), ("bf16", 128, 100, 16, -5.0),
                                               ("f32", 128, 70, 32, -2.5), ("bf16", 64, 33, 64, -1.0)])
def test_log_decay_staged(dtype, d, T, C, g_min):
    w = I.CORRECTNESS.with_(B=1, H=2, T=T, dk=d, dv=d, chunk=C, dtype=dtype, init_std=0.02)
    x = to(I.prefill_inputs(w), "cuda")
    out, fin = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], g_min, x["init_state"],
                             chunk=C, decay="log", workspace=None)
    torch.cuda.synchronize()
    ro, rf = oracle.fwd(*(x[n].cpu() for n in ("q", "k", "v", "g", "beta")), g_min,
                        x["init_state"].cpu(), decay="log")
    assert rel(out, ro) <= TOL[dtype], rel(out, ro)
    assert rel(fin, rf) <= TOL[dtype], rel(fin, rf)


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_log_decay_fused_paths(variant):
    g_min = -1.25
    w = I.PREFILL.with_(B=1, H=2, T=300)
    x = to(I.prefill_inputs(w), "cuda")
    with path_variant(variant) as ws:
        out, fin = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], g_min,
                                 x["init_state"], decay="log", workspace=ws)
    torch.cuda.synchronize()
    ro, rf = oracle.fwd(*(x[n].cpu() for n in ("q", "k", "v", "g", "beta")), g_min,
                        x["init_state"].cpu(), decay="log")
    assert rel(out, ro) <= TOL["bf16"], rel(out, ro)
    assert rel(fin, rf) <= TOL["bf16"], rel(fin, rf)


@pytest.mark.parametrize("variant", ["chain2", "chain1"])
@pytest.mark.parametrize("decay,bound", [("log", -5.0), ("affine", 0.05)])
@pytest.mark.parametrize("T", [209, 700])
def test_wide_range_two_kernel(variant, decay, bound, T):
    """The pages' own setting, log alpha = -5 sigmoid(g), and a linear-domain floor of
    0.05 on the two-kernel path, whose range rule spans a 16-token tile: over a 64-token
    chunk the decay here falls to about e^-160, so gamma and gamma_C underflow fp32 and
    1/gamma would overflow -- the preparation's 16-row reference points and the chain's
    factors of at most 1 must still give the oracle's result.  Ragged last chunk, several
    chunks, both chain splits."""
    w = I.PREFILL.with_(B=1, H=2, T=T)
    x = to(I.prefill_inputs(w), "cuda")
    with path_variant(variant) as ws:
        out, fin = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], bound,
                                 x["init_state"], decay=decay, workspace=ws)
    torch.cuda.synchronize()
    assert gdr.last_device_error() == 0
    ro, rf = oracle.fwd(*(x[n].cpu() for n in ("q", "k", "v", "g", "beta")), bound,
                        x["init_state"].cpu(), decay=decay)
    assert np.isfinite(out.float().cpu().numpy()).all()
    assert rel(out, ro) <= TOL["bf16"], rel(out, ro)
    assert rel(fin, rf) <= TOL["bf16"], rel(fin, rf)


def test_wide_range_needs_the_workspace_path():
    """Without a workspace the single-launch kernels keep the chunk-wide range rule."""
    w = I.PREFILL.with_(B=1, H=1, T=64)
    x = to(I.prefill_inputs(w), "cuda")
    with pytest.raises(gdr.GdrError):
        gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], -5.0, None, decay="log",
                      workspace=None)


@pytest.mark.parametrize("variant", ["chain2", "chain1"])
def test_wide_range_varlen(variant):
    """Packed sequences on the two-kernel path with a floor of 0.05 (chunk-wide decay
    far below fp32's range), each sequence against the oracle on its own."""
    w = I.PREFILL.with_(H=2)
    lengths = [1, 65, 0, 200, 130]
    x = I.varlen_inputs(w, lengths, device="cuda")
    with path_variant(variant) as ws:
        out, fin = gdr.chunk_fwd_varlen(x["q"], x["k"], x["v"], x["g"], x["beta"], 0.05,
                                        x["cu_seqlens"], x["init_state"], workspace=ws)
    torch.cuda.synchronize()
    cu = x["cu_seqlens"].tolist()
    for s, xs in enumerate(x["seqs"]):
        if lengths[s] == 0:
            assert torch.equal(fin[s], x["init_state"][s])
            continue
        cpu = {n: (None if t is None else t.cpu()) for n, t in xs.items()}
        ro, rf = oracle.fwd(cpu["q"], cpu["k"], cpu["v"], cpu["g"], cpu["beta"], 0.05,
                            cpu["init_state"])
        e_o = rel(out[cu[s]:cu[s + 1]].cpu(), torch.as_tensor(ro)[0].transpose(0, 1))
        e_f = rel(fin[s].cpu(), torch.as_tensor(rf)[0])
        assert e_o <= TOL["bf16"] and e_f <= TOL["bf16"], (s, e_o, e_f)


@pytest.mark.parametrize("dtype,pinned", [("bf16", True), ("bf16", False), ("f32", True)])
def test_host_buffers_match_device_call(dtype, pinned):
    """gdr_chunk_fwd_host (host buffers in and out, copies on the stream) gives exactly
    the device call's output and final state, and the oracle's within tolerance."""
    w = (I.PREFILL.with_(B=2, H=2, T=300) if dtype == "bf16"
         else I.CORRECTNESS.with_(T=200, dk=128, dv=128, init_std=0.3))
    x = I.prefill_inputs(w)
    host = {n: (None if t is None else (t.pin_memory() if pinned else t.contiguous()))
            for n, t in x.items()}
    buf = torch.empty(gdr.chunk_fwd_host_buffer_size(w.B, w.H, w.T, w.dk, w.dv, w.chunk,
                                                     w.torch_dtype()),
                      dtype=torch.uint8, device="cuda")
    out_h = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.torch_dtype(), pin_memory=pinned)
    fin_h = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, pin_memory=pinned)
    gdr.chunk_fwd_host(host["q"], host["k"], host["v"], host["g"], host["beta"], w.a_min,
                       host["init_state"], out_h, fin_h, buf, chunk=w.chunk)
    torch.cuda.synchronize()
    out_d, fin_d = run_gpu(to(x, "cuda"), w)
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(fin_h, fin_d.cpu())
    ro, rf = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, x["init_state"])
    assert rel(out_h, ro) <= TOL[dtype] and rel(fin_h, rf) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_log_decay_decode(dtype):
    w = I.DECODE.with_(B=8, H=4, dtype=dtype)
    state = I.decode_state(w, device="cuda")
    ref = state.cpu().double().numpy().copy()
    for s in range(3):
        x = I.decode_step_inputs(w, s, device="cuda")
        o = gdr.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], -5.0, state, decay="log")
        torch.cuda.synchronize()
        r = oracle.decode(*(x[n].cpu() for n in ("q", "k", "v", "g", "beta")), -5.0, ref,
                          decay="log")
        assert rel(o, r) <= TOL[dtype], rel(o, r)
    assert rel(state, ref) <= 1e-5


def test_zero_length_copies_state():
    w = I.PREFILL.with_(B=2, H=3, T=0)
    init = torch.randn(2, 3, 128, 128, device="cuda")
    e = torch.empty(2, 3, 0, 128, device="cuda", dtype=torch.bfloat16)
    z = torch.empty(2, 3, 0, device="cuda")
    out, fin = gdr.chunk_fwd(e, e, e, z, z, 0.95, init)
    torch.cuda.synchronize()
    assert torch.equal(fin, init)
    out, fin = gdr.chunk_fwd(e, e, e, z, z, 0.95, None)
    torch.cuda.synchronize()
    assert not fin.any()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_init_may_alias_final(dtype):
    w = I.CORRECTNESS.with_(B=2, H=2, T=130, dk=128, dv=128, dtype=dtype, init_std=0.02)
    x = to(I.prefill_inputs(w), "cuda")
    ref_out, ref_fin = run_gpu(x, w)
    st = x["init_state"].clone()
    gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, st, final_state=st)
    torch.cuda.synchronize()
    assert torch.equal(st, ref_fin)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T1", [64, 100, 1])
def test_split_resume_and_prefill_to_decode(dtype, T1):
    """One call over [0,T) equals two calls [0,T1), [T1,T) carrying the state;
    a decode step after a prefill equals a prefill one token longer."""
    T = 257
    w = I.CORRECTNESS.with_(B=1, H=2, T=T, dk=128, dv=128, dtype=dtype, init_std=0.02)
    x = to(I.prefill_inputs(w), "cuda")
    tol = TOL[dtype]
    full_o, full_f = run_gpu(x, w)
    a = {n: (x[n][:, :, :T1].contiguous() if n != "init_state" else x[n]) for n in x}
    b = {n: (x[n][:, :, T1:].contiguous() if n != "init_state" else None) for n in x}
    o1, f1 = run_gpu(a, w)
    o2, f2 = run_gpu(b, w, init=f1)
    assert rel(torch.cat([o1, o2], 2), full_o) <= tol
    assert rel(f2, full_f) <= tol
    # prefill T-1 tokens, then decode the last one
    p = {n: (x[n][:, :, :T - 1].contiguous() if n != "init_state" else x[n]) for n in x}
    po, pf = run_gpu(p, w)
    o_last = gdr.decode_step(x["q"][:, :, -1].contiguous(), x["k"][:, :, -1].contiguous(),
                             x["v"][:, :, -1].contiguous(), x["g"][:, :, -1].contiguous(),
                             x["beta"][:, :, -1].contiguous(), w.a_min, pf)
    torch.cuda.synchronize()
    assert rel(o_last, full_o[:, :, -1]) <= tol
    assert rel(pf, full_f) <= tol


# ------------------------------------------------------------------ the prefill workloads
def _prefill_full(w):
    x = I.prefill_inputs(w, device="cuda")
    out, fin = run_gpu(x, w)
    cpu = {n: (None if t is None else t.cpu()) for n, t in x.items()}
    return x, cpu, out, fin


def test_prefill_b4h16t4096():
    w = I.PREFILL
    x, cpu, out, fin = _prefill_full(w)
    ro, rf = oracle.fwd(cpu["q"], cpu["k"], cpu["v"], cpu["g"], cpu["beta"], w.a_min,
                        cpu["init_state"])
    e_o, e_f = rel(out, ro), rel(fin, rf)
    print(f"prefill rel-L2 out {e_o:.3e} final {e_f:.3e}")
    assert e_o <= TOL["bf16"] and e_f <= TOL["bf16"]
    # every other kernel on the same inputs
    for name in VARIANTS:
        with path_variant(name) as ws:
            out1, fin1 = run_gpu(x, w, workspace=ws)
        e_o, e_f = rel(out1, ro), rel(fin1, rf)
        print(f"prefill ({name}) rel-L2 out {e_o:.3e} final {e_f:.3e}")
        assert e_o <= TOL["bf16"] and e_f <= TOL["bf16"]


@pytest.mark.slow
def test_long_prefill_b1h32t65536():
    w = I.LONG_PREFILL
    x, cpu, out, fin = _prefill_full(w)
    ro, rf = oracle.fwd(cpu["q"], cpu["k"], cpu["v"], cpu["g"], cpu["beta"], w.a_min, None)
    e_o, e_f = rel(out, ro), rel(fin, rf)
    print(f"long prefill rel-L2 out {e_o:.3e} final {e_f:.3e}")
    assert e_o <= TOL["bf16"] and e_f <= TOL["bf16"]


@pytest.mark.slow
def test_million_prefill_b1h16t1048576():
    """The oracle checks heads 0-1 over the first 32768 tokens and head 0's final
    state over the full million tokens; every output is finite."""
    w = I.MILLION_PREFILL
    x = I.prefill_inputs(w, device="cuda")
    out, fin = run_gpu(x, w)
    assert torch.isfinite(out).all() and torch.isfinite(fin).all()
    P = 32768
    sub = {n: x[n][:, :2, :P].cpu() for n in ("q", "k", "v", "g", "beta")}
    ro, _ = oracle.fwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], w.a_min, None,
                       want_final=False)
    e_o = rel(out[:, :2, :P], ro)
    h0 = {n: x[n][:, :1].cpu() for n in ("q", "k", "v", "g", "beta")}
    _, rf = oracle.fwd(h0["q"], h0["k"], h0["v"], h0["g"], h0["beta"], w.a_min, None,
                       want_out=False)
    e_f = rel(fin[:, :1], rf)
    # head 0 over the first 2^18 tokens: the boundary between the first two segments
    # of the default segment split lies inside (at most 2^18 tokens per segment for
    # five segments and more)
    P2 = 1 << 18
    s2 = {n: x[n][:, :1, :P2].cpu() for n in ("q", "k", "v", "g", "beta")}
    r2, _ = oracle.fwd(s2["q"], s2["k"], s2["v"], s2["g"], s2["beta"], w.a_min, None,
                       want_final=False)
    e_2 = rel(out[:, :1, :P2], r2)
    print(f"million prefill rel-L2 out[h0-1,:32768] {e_o:.3e} out[h0,:2^18] {e_2:.3e} "
          f"final[h0] {e_f:.3e}")
    assert e_o <= TOL["bf16"] and e_f <= TOL["bf16"] and e_2 <= TOL["bf16"]


# ------------------------------------------------------------------ the decode workload
def test_decode_n256h32_64steps():
    w = I.DECODE
    state = I.decode_state(w, device="cuda")
    ref_state = state.cpu().double().numpy().copy()
    worst_o = 0.0
    for s in range(w.steps):
        x = I.decode_step_inputs(w, s, device="cuda")
        out = gdr.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, state)
        ro = oracle.decode(*(x[n].cpu() for n in ("q", "k", "v", "g", "beta")), w.a_min,
                           ref_state)
        e = rel(out, ro)
        worst_o = max(worst_o, e)
        assert e <= TOL["bf16"], (s, e)
    e_f = rel(state, ref_state)
    print(f"decode worst step rel-L2 out {worst_o:.3e}; final state {e_f:.3e}")
    assert e_f <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [(64, 64), (128, 64), (32, 128), (128, 128)])
def test_decode_shapes(dtype, d):
    dk, dv = d
    w = I.DECODE.with_(B=5, H=3, dk=dk, dv=dv, dtype=dtype)
    state = I.decode_state(w, device="cuda")
    ref_state = state.cpu().double().numpy().copy()
    for s in range(4):
        x = I.decode_step_inputs(w, s, device="cuda")
        out = gdr.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, state)
        ro = oracle.decode(*(x[n].cpu() for n in ("q", "k", "v", "g", "beta")), w.a_min,
                           ref_state)
        assert rel(out, ro) <= (1e-5 if dtype == "f32" else TOL["bf16"])
    assert rel(state, ref_state) <= 1e-5


# the one-pass kernel on every dimension and chunk it takes, ragged, with and without
# an initial state, against the oracle at the fp32 tolerance
@pytest.mark.parametrize("dk,dv,C,T", [(16, 16, 16, 37), (32, 128, 32, 130), (128, 16, 64, 129),
                                       (64, 32, 16, 300), (128, 128, 64, 200)])
@pytest.mark.parametrize("init", [None, 0.3])
def test_one_pass_kernel_shapes(dk, dv, C, T, init):
    w = I.CORRECTNESS.with_(B=2, H=2, T=T, dk=dk, dv=dv, chunk=C, dtype="f32", init_std=init)
    x = to(I.prefill_inputs(w), "cuda")
    out, fin = run_gpu(x, w, workspace=None)
    cpu = {n: (None if t is None else t.cpu()) for n, t in x.items()}
    ro, rf = oracle.fwd(cpu["q"], cpu["k"], cpu["v"], cpu["g"], cpu["beta"], w.a_min,
                        cpu["init_state"])
    assert rel(out, ro) <= TOL["f32"], rel(out, ro)
    assert rel(fin, rf) <= TOL["f32"], rel(fin, rf)


# ------------------------------------------------------------------ sequence segments
# The two-kernel path with S segments per head: every segment's offset map and
# transition at once, the scan over segments, then every segment's chain at once.
# Forced segment counts on small shapes: several chunks per segment, ragged last
# segments, with and without an initial state, both chain splits, both decay forms
# (the pages' g_min = -5 included, where the decay over a chunk underflows fp32).
@pytest.mark.parametrize("S", [2, 3, 5])
@pytest.mark.parametrize("split", [1, 2])
@pytest.mark.parametrize("decay,bound", [("affine", 0.95), ("log", -5.0)])
@pytest.mark.parametrize("T,init", [(64 * 12, 0.02), (64 * 10 + 17, None), (64 * 7 + 1, 0.3)])
def test_segmented_two_kernel(S, split, decay, bound, T, init):
    w = I.PREFILL.with_(B=2, H=2, T=T, init_std=init)
    x = to(I.prefill_inputs(w), "cuda")
    with gdr.option(segments=S, chain_split=split):
        # (the path query takes the linear-domain floor; the path is the same for both forms)
        assert gdr.chunk_fwd_path(w.B, w.H, w.T, w.dk, w.dv, w.chunk, w.a_min) == 7
        out, fin = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], bound,
                                 x["init_state"], decay=decay, workspace="auto")
    torch.cuda.synchronize()
    cpu = {n: (None if t is None else t.cpu()) for n, t in x.items()}
    ro, rf = oracle.fwd(cpu["q"], cpu["k"], cpu["v"], cpu["g"], cpu["beta"], bound,
                        cpu["init_state"], decay=decay)
    assert rel(out, ro) <= TOL["bf16"], rel(out, ro)
    assert rel(fin, rf) <= TOL["bf16"], rel(fin, rf)
    # every segment's rows on their own: a wrong segment state would show in its rows
    nc = (T + 63) // 64
    L = (nc + S - 1) // S
    for s0 in range(0, nc, L):
        a, b = s0 * 64, min(T, (s0 + L) * 64)
        assert rel(out[:, :, a:b], ro[:, :, a:b]) <= TOL["bf16"], (s0, rel(out[:, :, a:b], ro[:, :, a:b]))


def test_segmented_matches_unsegmented_and_may_alias():
    """The segmented path against the single-segment chain (same tiles, same chain
    arithmetic: they differ only by the scan's fp32 products and the segment maps'
    roundings), and the initial state aliasing the final state."""
    w = I.PREFILL.with_(B=1, H=3, T=64 * 20 + 5)
    x = to(I.prefill_inputs(w), "cuda")
    with gdr.option(segments=1):
        ref_out, ref_fin = run_gpu(x, w)
    with gdr.option(segments=4):
        out, fin = run_gpu(x, w)
        st = x["init_state"].clone()
        out2, _ = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, st,
                                final_state=st)
        torch.cuda.synchronize()
    assert rel(out, ref_out) <= 3e-3 and rel(fin, ref_fin) <= 3e-3
    assert torch.equal(out2, out) and torch.equal(st, fin)


def test_segment_count_is_automatic_for_few_heads():
    """Few heads and long sequences take the segmented path by default; many heads
    do not (every SM already has a chain)."""
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    assert gdr.chunk_fwd_path(1, 16, 1 << 20, 128, 128, 64, 0.99) == (7 if sms >= 48 else 4)
    assert gdr.chunk_fwd_path(4, 16, 4096, 128, 128, 64, 0.95) in (4, 5)
    assert gdr.chunk_fwd_path(1, 16, 256, 128, 128, 64, 0.99) in (4, 5)   # too short to split
