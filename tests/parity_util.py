"""Helpers of the GPU parity tests: run the CUDA path and the CPU oracle on the
same seeded inputs and compare element by element."""
from __future__ import annotations

import numpy as np
import torch

from oracle import lg_oracle
from sparse_long_sequence_window_gb300 import workloads

# Tolerances (max abs on O; mean abs on O for bf16; abs on LSE).
TOL = {
    "f32": dict(o_max=1e-5, o_mean=None, lse=1e-3),
    "bf16": dict(o_max=2e-2, o_mean=2e-3, lse=1e-3),
}


def to_np32(t: torch.Tensor) -> np.ndarray:
    """Exact float32 copy of an input tensor (bf16 values are exact in f32)."""
    return t.float().numpy()


def compare(name, dtype, out_gpu, lse_gpu, out_ref, lse_ref):
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(o).all(), f"{name}: non-finite output"
    assert np.isfinite(l).all(), f"{name}: non-finite lse"
    err = np.abs(o - out_ref)
    lerr = np.abs(l - lse_ref)
    tol = TOL[dtype]
    assert err.max() <= tol["o_max"], f"{name}: max |dO| {err.max():.3e} > {tol['o_max']}"
    if tol["o_mean"] is not None:
        assert err.mean() <= tol["o_mean"], f"{name}: mean |dO| {err.mean():.3e} > {tol['o_mean']}"
    assert lerr.max() <= tol["lse"], f"{name}: max |dLSE| {lerr.max():.3e} > {tol['lse']}"
    return float(err.max()), float(err.mean()), float(lerr.max())


def run_longformer(lg, w: workloads.Workload, rows=None, scale=None, key_ramp=None, workspace_fill=None):
    """CUDA path vs oracle for a (non-ETC) workload; rows=None compares every row.

    scale: the logit scale passed to both sides (None: the default 1/sqrt(D)).
    key_ramp: if given, key n is multiplied by 1 + key_ramp * n / N (rounded back to the
    input dtype; both sides get the same keys), so the logits grow along the sequence.
    workspace_fill: if given, the call gets its own workspace with every byte set to this
    value first (0xFF makes every float in it a NaN), so that a value the library reads
    without having written it in this call shows in the output."""
    inp = workloads.make_inputs(w)
    if key_ramp is not None:
        ramp = 1.0 + key_ramp * torch.arange(w.N, dtype=torch.float32) / w.N
        inp["k"] = (inp["k"].float() * ramp[None, None, :, None]).to(inp["k"].dtype)
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    g = inp["global_idx"]
    gd = torch.from_numpy(g).to(dev) if g.size else None
    ws = None
    if workspace_fill is not None:
        nbytes = lg.attn_fwd_workspace_size(w.B, w.H, w.N, w.D, int(g.size), 1 if w.dtype == "bf16" else 0)
        ws = torch.full((max(nbytes, 256),), workspace_fill, dtype=torch.uint8, device=dev)
    out, lse = lg.attn_fwd(q, k, v, w.w_left, w.w_right, w.dilations(), w.causal, gd, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    st = lg.query_status(lg.attn_fwd.last_workspace)
    assert st == 0, lg.status_string(st)
    qn, kn, vn = (to_np32(inp[n]) for n in ("q", "k", "v"))
    if rows is None:
        ref_o, ref_l = lg_oracle.attn_fwd(qn, kn, vn, w.w_left, w.w_right, w.dilations(), w.causal, g, scale=scale)
        return compare(w.name, w.dtype, out.cpu(), lse.cpu(), ref_o, ref_l)
    rows = np.asarray(sorted(set(int(r) for r in rows if 0 <= r < w.N)), dtype=np.int64)
    ref_o, ref_l = lg_oracle.attn_fwd_rows(qn, kn, vn, w.w_left, w.w_right, w.dilations(), w.causal, g, rows,
                                           scale=scale)
    return compare(w.name, w.dtype, out.cpu()[:, :, rows], lse.cpu()[:, :, rows], ref_o, ref_l)


def run_etc(lg, w: workloads.Workload, long_rows=None, scale=None):
    inp = workloads.make_inputs(w)
    dev = torch.device("cuda")
    t = [inp[n].to(dev) for n in ("q", "k", "v", "q_g", "k_g", "v_g")]
    out_l, out_g, lse_l, lse_g = lg.etc_attn_fwd(*t, w.radius, scale=scale)
    torch.cuda.synchronize()
    st = lg.query_status(lg.etc_attn_fwd.last_workspace)
    assert st == 0, lg.status_string(st)
    npx = [to_np32(inp[n]) for n in ("q", "k", "v", "q_g", "k_g", "v_g")]
    if long_rows is None:
        rl, rg, rll, rlg = lg_oracle.etc_attn_fwd(*npx, w.radius, scale=scale)
        a = compare(w.name + " long", w.dtype, out_l.cpu(), lse_l.cpu(), rl, rll)
    else:
        long_rows = np.asarray(sorted(set(int(r) for r in long_rows if 0 <= r < w.N)), dtype=np.int64)
        rl, rg, rll, rlg = lg_oracle.etc_attn_fwd_rows(*npx, w.radius, long_rows, scale=scale)
        a = compare(w.name + " long", w.dtype, out_l.cpu()[:, :, long_rows], lse_l.cpu()[:, :, long_rows], rl, rll)
    b = compare(w.name + " global", w.dtype, out_g.cpu(), lse_g.cpu(), rg, rlg)
    return a, b


def sample_rows(N, globals_=(), dilations=(1,), n_random=48, seed=0):
    """Edge rows, rows around tile boundaries and residue-class starts, some globals, random rows."""
    rng = np.random.default_rng(seed)
    rows = set(range(0, min(N, 6))) | set(range(max(0, N - 6), N))
    for t in (127, 128, 129, 255, 256, 511, 512, 513):
        for d in dilations:
            rows.update({t * d, t * d + d - 1, N - 1 - t * d})
    g = list(globals_)
    rows.update(g[:8] + g[-8:])
    rows.update(rng.integers(0, N, size=n_random).tolist())
    return sorted(r for r in rows if 0 <= r < N)
