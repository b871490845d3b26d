"""Backward pass: the CUDA path against the CPU oracle (needs a GB300).

The GPU forward runs first; its out and lse feed the GPU backward, as in
training.  The oracle (oracle.lg_oracle.attn_bwd / etc_attn_bwd) takes the
same rounded inputs and the same dout in float64 and recomputes its own
forward.  Every element of dq, dk, dv is compared.
"""
import numpy as np
import pytest
import torch

from oracle import lg_oracle
from sparse_long_sequence_window_gb300 import workloads
from sparse_long_sequence_window_gb300.workloads import Workload
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


def W(name, dtype, B, H, N, D, wl, wr, dil=(), causal=False, g=None, nrand=0, seed=300, **kw):
    return Workload(name, dtype, B, H, N, D, wl, wr, tuple(dil), causal, g, nrand, seed=seed, **kw)


def grad_errors(name, got, ref, floor=1e-30):
    """max |err| / max |ref| and mean |err| / mean |ref| of one gradient.

    floor: the smallest reference scale used.  A gradient can be exactly zero
    (a row whose only key is itself has P = 1, dP = Delta, dS = 0), and then
    the kernel's fp32 rounding of dP - Delta is to be compared with the size of
    one term of that gradient, not with zero (see ``term_floors``)."""
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), f"{name}: non-finite gradient"
    err = np.abs(g - ref)
    return err.max() / max(np.abs(ref).max(), floor), err.mean() / max(np.abs(ref).mean(), floor)


def term_floors(q, k, v, dout, D, scale):
    """1e-4 of the largest single term of dQ (s dS_ij k_j, |dS| <= D |dO| |v|), dK and dV (P_ij dO_i)."""
    s = scale if scale else 1.0 / np.sqrt(D)
    mx = lambda x: float(np.abs(x).max())
    base = s * D * mx(dout) * mx(v)
    return {"dq": 1e-4 * base * mx(k), "dk": 1e-4 * base * mx(q), "dv": 1e-4 * mx(dout)}


def run_bwd(lg, w, scale=None):
    inp = workloads.make_inputs(w)
    gr = workloads.make_grad_out(w)
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    dout = gr["dout"].to(dev)
    g = inp["global_idx"]
    gd = torch.from_numpy(g).to(dev) if g.size else None
    out, lse = lg.attn_fwd(q, k, v, w.w_left, w.w_right, w.dilations(), w.causal, gd, scale=scale)
    assert lg.query_status(lg.attn_fwd.last_workspace) == 0
    dq, dk, dv = lg.attn_bwd(q, k, v, out, lse, dout, w.w_left, w.w_right, w.dilations(), w.causal, gd, scale=scale)
    torch.cuda.synchronize()
    assert lg.query_status(lg.attn_bwd.last_workspace) == 0
    qn, kn, vn, don = (pu.to_np32(x) for x in (inp["q"], inp["k"], inp["v"], gr["dout"]))
    rq, rk, rv = lg_oracle.attn_bwd(qn, kn, vn, don, w.w_left, w.w_right, w.dilations(), w.causal, g, scale=scale)
    fl = term_floors(qn, kn, vn, don, w.D, scale)
    return {n: grad_errors(f"{w.name} {n}", x, r, fl[n]) for n, x, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv))}


def run_etc_bwd(lg, w, scale=None):
    inp = workloads.make_inputs(w)
    gr = workloads.make_grad_out(w)
    dev = torch.device("cuda")
    t = [inp[n].to(dev) for n in ("q", "k", "v", "q_g", "k_g", "v_g")]
    out_l, out_g, lse_l, lse_g = lg.etc_attn_fwd(*t, w.radius, scale=scale)
    assert lg.query_status(lg.etc_attn_fwd.last_workspace) == 0
    grads = lg.etc_attn_bwd(*t, out_l, out_g, lse_l, lse_g, gr["dout"].to(dev), gr["dout_g"].to(dev), w.radius,
                            scale=scale)
    torch.cuda.synchronize()
    assert lg.query_status(lg.etc_attn_bwd.last_workspace) == 0
    npx = [pu.to_np32(inp[n]) for n in ("q", "k", "v", "q_g", "k_g", "v_g")]
    ref = lg_oracle.etc_attn_bwd(*npx, w.radius, pu.to_np32(gr["dout"]), pu.to_np32(gr["dout_g"]), scale=scale)
    names = ("dq_l", "dk_l", "dv_l", "dq_g", "dk_g", "dv_g")
    fl = term_floors(np.concatenate([npx[0], npx[3]], 2), np.concatenate([npx[1], npx[4]], 2),
                     np.concatenate([npx[2], npx[5]], 2), pu.to_np32(gr["dout"]), w.D, scale)
    return {n: grad_errors(f"{w.name} {n}", x, r, fl[n[:2]]) for n, x, r in zip(names, grads, ref)}


BWD_TOL = {"f32": (1e-5, 1e-5), "bf16": (2e-2, 1e-2)}   # (max rel. to max |ref|, mean rel. to mean |ref|)


def check(w, errs):
    tmax, tmean = BWD_TOL[w.dtype]
    for n, (emax, emean) in errs.items():
        print(f"{w.name} {n}: max {emax:.2e} mean {emean:.2e}")
        assert emax <= tmax and emean <= tmean, f"{w.name} {n}: max {emax:.2e} mean {emean:.2e}"


BWD_CASES = [
    W("bwd bf16 D64 two tiles + tail", "bf16", 1, 2, 300, 64, 16, 16),
    W("bwd bf16 D128 two tiles + tail", "bf16", 1, 2, 300, 128, 16, 16),
    W("bwd bf16 single token", "bf16", 1, 1, 1, 64, 4, 4),
    W("bwd bf16 asymmetric window", "bf16", 2, 2, 700, 64, 100, 37),
    W("bwd bf16 causal D128", "bf16", 1, 2, 777, 128, 200, 50, (), True),
    W("bwd bf16 dilation 1..4 + globals", "bf16", 1, 4, 1000, 64, 60, 20, (1, 2, 3, 4), False, (0, 5, 999)),
    W("bwd bf16 dilation 1..8", "bf16", 1, 8, 1500, 64, 40, 40, (1, 2, 3, 4, 5, 6, 7, 8)),
    W("bwd bf16 dilation 5..8 causal D128", "bf16", 1, 4, 1100, 128, 50, 9, (5, 6, 7, 8), True),
    W("bwd bf16 130 globals (two tiles)", "bf16", 1, 2, 2000, 64, 64, 64, (), False, None, 130),
    W("bwd bf16 globals at edges D128", "bf16", 1, 3, 1025, 128, 100, 100, (1, 1, 2), False, (0, 1, 511, 1023, 1024)),
    W("bwd bf16 causal with globals", "bf16", 1, 2, 600, 64, 64, 64, (1, 3), True, (10, 590)),
    W("bwd bf16 every token global", "bf16", 1, 1, 140, 64, 2, 2, (), False, tuple(range(140))),
    W("bwd bf16 dense globals in dilated bands", "bf16", 1, 4, 700, 64, 40, 40, (1, 2, 3, 5), False,
      tuple(range(100, 400, 3))),
    W("bwd bf16 full window", "bf16", 1, 2, 513, 64, 600, 600),
]


@pytest.mark.parametrize("w", BWD_CASES, ids=lambda w: w.name)
def test_bwd_bf16(cuda_lib, w):
    check(w, run_bwd(cuda_lib, w))


F32_BWD = [
    W("bwd f32 ragged D=36", "f32", 2, 3, 77, 36, 5, 2, (1, 2, 3), False, (0, 40, 76)),
    W("bwd f32 causal dilated", "f32", 1, 4, 190, 64, 9, 9, (1, 2, 5, 11), True, (3, 100)),
    W("bwd f32 every token global", "f32", 1, 1, 40, 8, 1, 1, (), False, tuple(range(40))),
]


@pytest.mark.parametrize("w", F32_BWD, ids=lambda w: w.name)
def test_bwd_f32(cuda_lib, w):
    check(w, run_bwd(cuda_lib, w))


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("bf16", 128), ("f32", 32)])
def test_bwd_etc(cuda_lib, dtype, D):
    w = W(f"bwd etc {dtype} D{D}", dtype, 2, 2, 700 if dtype == "bf16" else 130, D, 0, 0, etc_G=70 if dtype == "bf16" else 9,
          radius=20 if dtype == "bf16" else 6)
    check(w, run_etc_bwd(cuda_lib, w))


def test_bwd_etc_star(cuda_lib):
    w = W("bwd etc star", "bf16", 1, 2, 300, 64, 0, 0, etc_G=1, radius=1)
    check(w, run_etc_bwd(cuda_lib, w))


@pytest.mark.parametrize("w,scale", [
    (W("bwd bf16 scale D64", "bf16", 1, 3, 600, 64, 50, 30, (1, 2, 3), False, (0, 300)), 0.37),
    (W("bwd bf16 scale D128 causal", "bf16", 1, 2, 500, 128, 60, 0, (1, 2), True, None, 7), 0.05),
    (W("bwd f32 scale", "f32", 1, 2, 150, 32, 10, 10, (1, 3), False, (4,)), 0.37),
], ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_bwd_explicit_scale(cuda_lib, w, scale):
    check(w, run_bwd(cuda_lib, w, scale=scale))


def test_bwd_longformer_base_full(cuda_lib):
    """bf16 B1 H12 N4096 D64, window 256/256, globals 0..64: every element of dq, dk, dv."""
    w = workloads.PRESETS["longformer_base"]
    check(w, run_bwd(cuda_lib, w))


# ---------------------------------------------------------------- the reference workloads at full size

def _fwd_bwd(lg, w):
    inp = workloads.make_inputs(w)
    gr = workloads.make_grad_out(w)
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    dout = gr["dout"].to(dev)
    g = inp["global_idx"]
    gd = torch.from_numpy(g).to(dev) if g.size else None
    out, lse = lg.attn_fwd(q, k, v, w.w_left, w.w_right, w.dilations(), w.causal, gd)
    assert lg.query_status(lg.attn_fwd.last_workspace) == 0
    dq, dk, dv = lg.attn_bwd(q, k, v, out, lse, dout, w.w_left, w.w_right, w.dilations(), w.causal, gd)
    torch.cuda.synchronize()
    assert lg.query_status(lg.attn_bwd.last_workspace) == 0
    return inp, gr, (dq.cpu(), dk.cpu(), dv.cpu())


def _sum_identities(name, dk, dv, dout):
    """Exact at any size: shifting every key leaves O unchanged (sum_j dK_j = 0)
    and every row of P sums to 1 (sum_j dV_j = sum_i dO_i), per (b, h)."""
    dk = dk.double().numpy(); dv = dv.double().numpy(); do = dout.double().numpy()
    ek = np.abs(dk.sum(axis=2)).max() / np.abs(dk).sum(axis=2).max()
    ev = np.abs(dv.sum(axis=2) - do.sum(axis=2)).max() / np.abs(dv).sum(axis=2).max()
    print(f"{name}: sum identities: dK {ek:.2e}, dV {ev:.2e}")
    assert ek < 5e-3 and ev < 5e-3


def _check_sampled(w, got, ref, what):
    tmax, tmean = BWD_TOL[w.dtype]
    g = got.double().numpy()
    err = np.abs(g - ref)
    emax, emean = err.max() / np.abs(ref).max(), err.mean() / np.abs(ref).mean()
    print(f"{w.name} {what}: max {emax:.2e} mean {emean:.2e}")
    assert emax <= tmax and emean <= tmean


def test_bwd_charlm_full_sampled(cuda_lib):
    """bf16 B1 H8 N16384 D64 causal wl 512, dilation [1,1,2,2,3,3,4,4]: sampled dQ rows and dK, dV keys."""
    w = workloads.PRESETS["charlm_dilated"]
    inp, gr, (dq, dk, dv) = _fwd_bwd(cuda_lib, w)
    qn, kn, vn, don = (pu.to_np32(x) for x in (inp["q"], inp["k"], inp["v"], gr["dout"]))
    rows = pu.sample_rows(w.N, dilations=(1, 2, 3, 4), n_random=24, seed=41)
    _check_sampled(w, dq[:, :, rows], lg_oracle.attn_bwd_rows(qn, kn, vn, don, w.w_left, w.w_right, w.dilations(),
                                                               w.causal, [], rows), "dq rows")
    cols = pu.sample_rows(w.N, dilations=(1, 2, 3, 4), n_random=8, seed=42)[::3]
    rk, rv = lg_oracle.attn_bwd_cols(qn, kn, vn, don, w.w_left, w.w_right, w.dilations(), w.causal, [], cols)
    _check_sampled(w, dk[:, :, cols], rk, "dk keys")
    _check_sampled(w, dv[:, :, cols], rv, "dv keys")
    _sum_identities(w.name, dk, dv, gr["dout"])


def test_bwd_long_scale_full_sampled(cuda_lib):
    """bf16 B1 H16 N131072 D128, window 512/512, 128 random globals (the benchmarked launch):
    sampled dQ rows (band and global) on every head, sampled band keys' dK, dV on two heads,
    and the sum identities (which take in every global key) on every head."""
    w = workloads.PRESETS["long_128k"]
    inp, gr, (dq, dk, dv) = _fwd_bwd(cuda_lib, w)
    g = workloads.global_positions(w)
    qn, kn, vn, don = (pu.to_np32(x) for x in (inp["q"], inp["k"], inp["v"], gr["dout"]))
    rows = pu.sample_rows(w.N, globals_=g.tolist()[:4], n_random=12, seed=43)
    _check_sampled(w, dq[:, :, rows], lg_oracle.attn_bwd_rows(qn, kn, vn, don, w.w_left, w.w_right, w.dilations(),
                                                               w.causal, g, rows), "dq rows")
    gset = set(g.tolist())
    cols = [c for c in (0, 127, 128, 4095, 65536, w.N - 1) if c not in gset]
    heads = [0, w.H - 1]
    rk, rv = lg_oracle.attn_bwd_cols(qn, kn, vn, don, w.w_left, w.w_right, w.dilations(), w.causal, g, cols,
                                     heads=heads)
    _check_sampled(w, dk[:, heads][:, :, cols], rk[:, heads], "dk keys")
    _check_sampled(w, dv[:, heads][:, :, cols], rv[:, heads], "dv keys")
    _sum_identities(w.name, dk, dv, gr["dout"])


def test_bwd_etc_base_two_slices(cuda_lib):
    """bf16 ETC B2 H12 L4096 G256 D64 r84: every gradient element of two (b, h) slices against the dense oracle."""
    lg = cuda_lib
    w = workloads.PRESETS["etc_base"]
    inp = workloads.make_inputs(w)
    gr = workloads.make_grad_out(w)
    dev = torch.device("cuda")
    t = [inp[n].to(dev) for n in ("q", "k", "v", "q_g", "k_g", "v_g")]
    out_l, out_g, lse_l, lse_g = lg.etc_attn_fwd(*t, w.radius)
    assert lg.query_status(lg.etc_attn_fwd.last_workspace) == 0
    grads = lg.etc_attn_bwd(*t, out_l, out_g, lse_l, lse_g, gr["dout"].to(dev), gr["dout_g"].to(dev), w.radius)
    torch.cuda.synchronize()
    assert lg.query_status(lg.etc_attn_bwd.last_workspace) == 0
    names = ("dq_l", "dk_l", "dv_l", "dq_g", "dk_g", "dv_g")
    for b, h in ((0, 0), (1, 11)):
        sl = lambda x: pu.to_np32(x)[b:b + 1, h:h + 1]
        ref = lg_oracle.etc_attn_bwd(*(sl(inp[n]) for n in ("q", "k", "v", "q_g", "k_g", "v_g")), w.radius,
                                     sl(gr["dout"]), sl(gr["dout_g"]))
        for n, x, r in zip(names, grads, ref):
            _check_sampled(w, x.cpu()[b:b + 1, h:h + 1], r, f"{n} (b={b}, h={h})")
