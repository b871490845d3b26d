"""LongNet mixture of dilated attentions: the CUDA path against the CPU oracle
(needs a GB300).

Small cases compare every element: the strided layout (r divides w, r <= 8)
and the packed one (any other r), causal and not, ragged N, D 64 and 128,
r > 8, r > w, rows that no pattern keeps, and the two launch plans (all
patterns in one launch up to 8 patterns and 32 heads, else one per pattern).  The LongNet language-model
workload at full size compares sampled rows, which the oracle computes one
at a time.  Tolerances as for the other bf16 outputs: max |dO| <= 2e-2,
mean |dO| <= 2e-3 over the kept rows, |dLSE| <= 1e-3; a row no pattern
keeps must come out as O = 0 and LSE = -inf exactly.
"""
import numpy as np
import pytest
import torch

from oracle import lg_oracle
from sparse_long_sequence_window_gb300 import workloads
from sparse_long_sequence_window_gb300.workloads import Workload
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


def L(name, B, H, N, D, ws, rs, causal=False, seed=300):
    return Workload(name, "bf16", B, H, N, D, causal=causal, seg_w=tuple(ws), seg_r=tuple(rs), seed=seed)


CASES = [
    L("one pattern covering the sequence", 1, 2, 300, 64, [512], [1]),
    L("strided two patterns ragged N", 1, 4, 1000, 64, [64, 256], [1, 4]),
    L("strided causal D128", 1, 3, 777, 128, [128, 512], [2, 8], True),
    L("packed r not dividing w", 2, 6, 1500, 64, [96, 500], [1, 6]),
    L("packed r above 8 causal", 1, 12, 2000, 64, [2048, 1000], [12, 16], True),
    L("r above w and uncovered rows", 1, 8, 300, 64, [4, 64], [8, 3]),
    L("packed D128 several segments", 1, 5, 1300, 128, [300, 650], [3, 5]),
    L("mixture of five patterns at 4K causal", 1, 12, 4096, 64, [256, 512, 1024, 2048, 4096],
      [1, 2, 4, 6, 12], True),
    L("single token", 1, 2, 1, 64, [16, 4], [1, 2]),
    L("one-row segments", 1, 3, 130, 64, [1, 3], [1, 5]),
    # Up to 8 patterns and 32 heads share one tensor-core launch; beyond that each
    # pattern has its own launch (and the packed patterns share one set of buffers).
    L("eight patterns in one launch", 1, 4, 900, 64, [32, 64, 96, 128, 256, 300, 512, 900],
      [1, 2, 3, 4, 6, 7, 8, 10], True),
    L("nine patterns, one launch each", 1, 4, 900, 64, [32, 64, 96, 128, 256, 300, 512, 900, 450],
      [1, 2, 3, 4, 6, 7, 8, 10, 9], True),
    L("33 heads, one launch per pattern", 1, 33, 400, 64, [64, 200], [2, 6]),
]


def compare_longnet(name, out, lse, ref_o, ref_l):
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.float().cpu().numpy().astype(np.float64)
    kept = np.isfinite(ref_l)
    assert np.array_equal(np.isneginf(l), ~kept), f"{name}: -inf LSE rows differ"
    assert np.isfinite(o).all(), f"{name}: non-finite output"
    assert (o[~kept] == 0).all(), f"{name}: a row no pattern keeps is not zero"
    if not kept.any():
        return
    tol = pu.TOL["bf16"]
    err = np.abs(o - ref_o)[kept]
    lerr = np.abs(l[kept] - ref_l[kept])
    assert err.max() <= tol["o_max"], f"{name}: max |dO| {err.max():.3e}"
    assert err.mean() <= tol["o_mean"], f"{name}: mean |dO| {err.mean():.3e}"
    assert lerr.max() <= tol["lse"], f"{name}: max |dLSE| {lerr.max():.3e}"


def run_case(lg, w, rows=None, scale=None):
    inp = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    out, lse = lg.longnet_attn_fwd(q, k, v, w.seg_w, w.seg_r, w.causal, scale=scale)
    torch.cuda.synchronize()
    st = lg.query_status(lg.longnet_attn_fwd.last_workspace)
    assert st == 0, lg.status_string(st)
    qn, kn, vn = (pu.to_np32(inp[n]) for n in ("q", "k", "v"))
    if rows is None:
        ref_o, ref_l = lg_oracle.longnet_attn_fwd(qn, kn, vn, w.seg_w, w.seg_r, w.causal, scale=scale)
        compare_longnet(w.name, out.cpu(), lse.cpu(), ref_o, ref_l)
    else:
        ref_o, ref_l = lg_oracle.longnet_attn_fwd_rows(qn, kn, vn, w.seg_w, w.seg_r, w.causal, rows, scale=scale)
        compare_longnet(w.name, out.cpu()[:, :, rows], lse.cpu()[:, :, rows], ref_o, ref_l)
    return out, lse


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_longnet_small(cuda_lib, w):
    run_case(cuda_lib, w)


def test_longnet_explicit_scale(cuda_lib):
    run_case(cuda_lib, L("explicit scale", 1, 4, 700, 64, [128, 350], [2, 7], True), scale=0.3)


def test_longnet_repeated_pattern_is_idempotent(cuda_lib):
    """A pattern mixed with itself gives its own output, and LSE + ln 2 (both patterns' denominators)."""
    w1 = L("single", 1, 4, 900, 64, [300], [3])
    w2 = L("twice", 1, 4, 900, 64, [300, 300], [3, 3])
    o1, l1 = run_case(cuda_lib, w1)
    o2, l2 = run_case(cuda_lib, w2)
    assert torch.equal(o1, o2) or (o1.float() - o2.float()).abs().max().item() <= 2 ** -8
    fin = torch.isfinite(l1)
    assert torch.equal(fin, torch.isfinite(l2))
    assert (l2[fin] - l1[fin] - np.log(2.0)).abs().max().item() < 1e-5


def test_longnet_lm_full_size_sampled_rows(cuda_lib):
    """The LongNet language-model mixture (B1 H12 N32768 D64, causal, w 2K..32K, r 1,2,4,6,12)
    in the benchmark's configuration; rows at segment edges plus random rows."""
    w = workloads.PRESETS["longnet_lm"]
    rng = np.random.default_rng(17)
    edges = [0, 1, 2047, 2048, 4095, 4096, 8191, 8192, 16383, 16384, 16385, 24575, 32766, 32767]
    rows = sorted(set(edges + rng.integers(0, w.N, size=40).tolist()))
    run_case(cuda_lib, w, rows=rows)


def test_longnet_reuses_caller_workspace(cuda_lib):
    """Two calls through one caller-owned workspace (the second with other patterns) give the
    same results as fresh workspaces."""
    lg = cuda_lib
    w = L("ws reuse", 1, 6, 1200, 64, [200, 600], [1, 6], True)
    inp = workloads.make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o_ref, l_ref = lg.longnet_attn_fwd(q, k, v, [64, 1200], [3, 12], False)
    o_ref2, l_ref2 = lg.longnet_attn_fwd(q, k, v, w.seg_w, w.seg_r, True)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    o_a, l_a = lg.longnet_attn_fwd(q, k, v, [64, 1200], [3, 12], False, workspace=ws)
    o_b, l_b = lg.longnet_attn_fwd(q, k, v, w.seg_w, w.seg_r, True, workspace=ws)
    torch.cuda.synchronize()
    assert lg.query_status(ws) == 0
    assert torch.equal(o_a, o_ref) and torch.equal(o_b, o_ref2)
    assert torch.equal(l_a, l_ref) and torch.equal(l_b, l_ref2)
