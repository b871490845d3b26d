"""CUDA path against the CPU oracle on the same seeded inputs (needs a GB300).

Small cases compare every output element (several tiles plus a ragged tail,
every edge case the method has); the full-size workloads compare sampled rows
that the oracle computes one by one, in the same launch configuration the
benchmark times.  Tolerances: fp32 max |dO| <= 1e-5; bf16 max |dO| <= 2e-2 and
mean |dO| <= 2e-3; |dLSE| <= 1e-3.
"""
import numpy as np
import pytest
import torch

from oracle import lg_oracle
from sparse_long_sequence_window_gb300 import workloads
from sparse_long_sequence_window_gb300.workloads import Workload
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


def W(name, dtype, B, H, N, D, wl, wr, dil=(), causal=False, g=None, nrand=0, seed=100, **kw):
    return Workload(name, dtype, B, H, N, D, wl, wr, tuple(dil), causal, g, nrand, seed=seed, **kw)


# ---------------------------------------------------------------- fp32 path (CUDA cores)

F32_CASES = [
    W("f32 single token", "f32", 1, 1, 1, 64, 3, 3),
    W("f32 ragged D=36 window", "f32", 2, 3, 77, 36, 5, 2, (1, 2, 3), False, (0, 40, 76)),
    W("f32 causal dilated", "f32", 1, 4, 190, 64, 9, 9, (1, 2, 5, 11), True, (3, 100)),
    W("f32 full window", "f32", 1, 2, 150, 128, 200, 200),
    W("f32 identity window", "f32", 1, 2, 64, 16, 0, 0, (1, 3)),
    W("f32 every token global", "f32", 1, 1, 40, 8, 1, 1, (), False, tuple(range(40))),
]


@pytest.mark.parametrize("w", F32_CASES, ids=lambda w: w.name)
def test_f32_small(cuda_lib, w):
    pu.run_longformer(cuda_lib, w)


def test_f32_tiny_preset(cuda_lib):
    """fp32 B1 H2 N512 D64, window 64/64, one global token at 0: every element."""
    pu.run_longformer(cuda_lib, workloads.PRESETS["tiny_f32"])


def test_f32_etc_small(cuda_lib):
    pu.run_etc(cuda_lib, W("f32 etc", "f32", 2, 2, 130, 32, 0, 0, etc_G=9, radius=6))


# ---------------------------------------------------------------- bf16 path (tensor cores)

BF16_CASES = [
    W("bf16 D64 two tiles + tail", "bf16", 1, 2, 300, 64, 16, 16),
    W("bf16 D128 two tiles + tail", "bf16", 1, 2, 300, 128, 16, 16),
    W("bf16 single token", "bf16", 1, 1, 1, 64, 4, 4),
    W("bf16 identity window", "bf16", 1, 2, 200, 64, 0, 0),
    W("bf16 asymmetric window", "bf16", 2, 2, 700, 64, 100, 37),
    W("bf16 full window", "bf16", 1, 2, 513, 64, 600, 600),
    W("bf16 causal D128", "bf16", 1, 2, 777, 128, 200, 50, (), True),
    W("bf16 dilation 1..4 + globals", "bf16", 1, 4, 1000, 64, 60, 20, (1, 2, 3, 4), False, (0, 5, 999)),
    W("bf16 dilation 1..8", "bf16", 1, 8, 1500, 64, 40, 40, (1, 2, 3, 4, 5, 6, 7, 8)),
    W("bf16 dilation 5..8 causal D128", "bf16", 1, 4, 1100, 128, 50, 9, (5, 6, 7, 8), True),
    W("bf16 130 globals (two tiles)", "bf16", 1, 2, 2000, 64, 64, 64, (), False, None, 130),
    W("bf16 globals at edges D128", "bf16", 1, 3, 1025, 128, 100, 100, (1, 1, 2), False, (0, 1, 511, 1023, 1024)),
    W("bf16 causal with globals", "bf16", 1, 2, 600, 64, 64, 64, (1, 3), True, (10, 590)),
    W("bf16 dilation beyond N", "bf16", 1, 2, 5, 64, 2, 2, (7, 8)),
    W("bf16 every token global", "bf16", 1, 1, 140, 64, 2, 2, (), False, tuple(range(140))),
    W("bf16 many heads", "bf16", 3, 16, 257, 64, 30, 30, tuple([1, 2] * 8)),
    W("bf16 dense globals in dilated bands", "bf16", 1, 4, 700, 64, 40, 40, (1, 2, 3, 5), False,
      tuple(range(100, 400, 3))),
    W("bf16 globals in causal dilated bands D128", "bf16", 1, 3, 900, 128, 70, 0, (2, 4, 7), True,
      tuple(range(0, 900, 7))),
    # one head, short window: the global-query rows are split into 8-tile pieces (16 partials)
    W("bf16 fine global-row splits D128", "bf16", 1, 1, 8192, 128, 64, 64, (), False, None, 128),
]


# Keys whose magnitude grows 30-fold along the sequence: every new key tile raises the row
# maximum past the lazy-rescale threshold (2^8), so O is rescaled on nearly every tile, a
# path that N(0, 1) inputs rarely take; band rows, global-query rows and causal rows.
RESCALE_CASES = [
    W("bf16 rising keys D64 dilated + globals", "bf16", 1, 2, 1100, 64, 300, 300, (1, 2), False, (0, 700)),
    W("bf16 rising keys D128 causal", "bf16", 1, 2, 900, 128, 400, 0, (), True),
    W("bf16 rising keys D128 + 130 globals", "bf16", 1, 1, 1500, 128, 128, 128, (), False, None, 130),
]


@pytest.mark.parametrize("w", RESCALE_CASES, ids=lambda w: w.name)
def test_bf16_running_max_rescales(cuda_lib, w):
    pu.run_longformer(cuda_lib, w, key_ramp=30.0)


@pytest.mark.parametrize("w", BF16_CASES, ids=lambda w: w.name)
def test_bf16_small(cuda_lib, w):
    pu.run_longformer(cuda_lib, w)


# Global rows over a sequence of one key tile: of the two warpgroups that share a global
# row's key tiles (alternate tiles), the second gets none and leaves an empty partial
# (maximum -inf, accumulator never written), which the merge must leave out.  The
# workspace is filled with 0xFF bytes (NaN as floats) before the call, so an accumulator
# read anyway would show; any bytes are a valid workspace (the call clears its status area).
@pytest.mark.parametrize("D", [64, 128])
def test_bf16_empty_global_partials_nan_workspace(cuda_lib, D):
    w = W(f"bf16 one key tile + globals D{D}", "bf16", 1, 2, 100, D, 10, 10, (), False, (0, 37, 99))
    pu.run_longformer(cuda_lib, w, workspace_fill=0xFF)


@pytest.mark.parametrize("name", ["bf16 globals at edges D128", "bf16 fine global-row splits D128"])
def test_bf16_nan_workspace(cuda_lib, name):
    """Global rows with several key splits (few partials per row, and many), on a
    NaN-filled workspace."""
    w = next(c for c in BF16_CASES if c.name == name)
    pu.run_longformer(cuda_lib, w, workspace_fill=0xFF)


@pytest.mark.parametrize("D", [64, 128])
def test_bf16_etc_small(cuda_lib, D):
    pu.run_etc(cuda_lib, W(f"bf16 etc D{D}", "bf16", 2, 2, 700, D, 0, 0, etc_G=70, radius=20))


def test_bf16_etc_star(cuda_lib):
    """ETC with r = 1 and one global token (the star pattern)."""
    pu.run_etc(cuda_lib, W("bf16 etc star", "bf16", 1, 2, 300, 64, 0, 0, etc_G=1, radius=1))


# ---------------------------------------------------------------- a logit scale other than 1/sqrt(D)

SCALE_CASES = [
    (W("f32 scale dilated globals", "f32", 1, 3, 300, 64, 20, 12, (1, 2, 3), False, (0, 150, 299)), 0.37),
    (W("f32 scale causal", "f32", 1, 2, 200, 32, 30, 30, (1, 4), True, (7,)), 0.05),
    (W("bf16 scale D64 dilated globals", "bf16", 1, 4, 900, 64, 50, 30, (1, 2, 3, 5), False, (0, 5, 450, 899)), 0.37),
    (W("bf16 scale D64 causal", "bf16", 1, 2, 700, 64, 100, 0, (1, 2), True, None, 9), 0.05),
    (W("bf16 scale D128 dilated globals", "bf16", 1, 3, 1100, 128, 64, 64, (1, 2, 4), False, None, 40), 0.37),
    (W("bf16 scale D128 causal", "bf16", 1, 2, 800, 128, 90, 0, (3, 1), True, (0, 799)), 0.05),
]


@pytest.mark.parametrize("w,scale", SCALE_CASES, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_explicit_scale(cuda_lib, w, scale):
    """The ABI's scale argument, taken by both the kernels and the oracle."""
    pu.run_longformer(cuda_lib, w, scale=scale)


@pytest.mark.parametrize("dtype,D,scale", [("f32", 32, 0.37), ("bf16", 64, 0.05), ("bf16", 128, 0.37)])
def test_explicit_scale_etc(cuda_lib, dtype, D, scale):
    pu.run_etc(cuda_lib, W(f"{dtype} etc scale D{D}", dtype, 1, 2, 500, D, 0, 0, etc_G=40, radius=15), scale=scale)


# ---------------------------------------------------------------- separate global projections

def run_gproj(lg, w):
    inp = workloads.make_inputs(w)
    gp = workloads.make_global_projections(w)
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    qg, kg, vg = (gp[n].to(dev) for n in ("q_glob", "k_glob", "v_glob"))
    g = inp["global_idx"]
    gd = torch.from_numpy(g).to(dev)
    out, lse = lg.attn_fwd(q, k, v, w.w_left, w.w_right, w.dilations(), w.causal, gd,
                           q_global=qg, k_global=kg, v_global=vg)
    torch.cuda.synchronize()
    assert lg.query_status(lg.attn_fwd.last_workspace) == 0
    npx = [pu.to_np32(x) for x in (inp["q"], inp["k"], inp["v"], gp["q_glob"], gp["k_glob"], gp["v_glob"])]
    ref_o, ref_l = lg_oracle.attn_fwd_gproj(*npx, w.w_left, w.w_right, w.dilations(), w.causal, g)
    return pu.compare(w.name, w.dtype, out.cpu(), lse.cpu(), ref_o, ref_l)


GPROJ_CASES = [
    W("gproj bf16 D64 dilated globals", "bf16", 1, 4, 900, 64, 50, 30, (1, 2, 3, 5), False, (0, 5, 450, 899)),
    W("gproj bf16 D128 causal random globals", "bf16", 1, 2, 1300, 128, 90, 0, (1, 2), True, None, 150),
    W("gproj f32 globals", "f32", 1, 3, 300, 64, 20, 12, (1, 2, 3), False, (0, 150, 299)),
    W("gproj bf16 every token global", "bf16", 1, 1, 140, 64, 2, 2, (), False, tuple(range(140))),
]


@pytest.mark.parametrize("w", GPROJ_CASES, ids=lambda w: w.name)
def test_separate_global_projections(cuda_lib, w):
    run_gproj(cuda_lib, w)


def test_separate_global_projections_longformer_base_full(cuda_lib):
    """bf16 B1 H12 N4096 D64, window 256/256, globals 0..64, separate global projections: every element."""
    run_gproj(cuda_lib, workloads.PRESETS["longformer_base"])


def test_equal_global_projections_match_shared(cuda_lib):
    """Passing q, k, v as the global projections gives lg_attn_fwd's bits."""
    lg = cuda_lib
    w = W("gproj equal", "bf16", 1, 3, 700, 128, 40, 40, (1, 2, 1), False, (0, 300, 699))
    inp = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    gd = torch.from_numpy(inp["global_idx"]).to(dev)
    o1, l1 = lg.attn_fwd(q, k, v, w.w_left, w.w_right, w.dilations(), False, gd)
    o1, l1 = o1.clone(), l1.clone()
    o2, l2 = lg.attn_fwd(q, k, v, w.w_left, w.w_right, w.dilations(), False, gd, q_global=q, k_global=k, v_global=v)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ---------------------------------------------------------------- the reference workloads at full size

def test_longformer_base_full(cuda_lib):
    """bf16 B1 H12 N4096 D64, window 256/256, globals 0..64: every element."""
    pu.run_longformer(cuda_lib, workloads.PRESETS["longformer_base"])


def test_etc_base_sampled(cuda_lib):
    """bf16 ETC B2 H12 L4096 G256 D64 r84: every global row and sampled long rows."""
    w = workloads.PRESETS["etc_base"]
    pu.run_etc(cuda_lib, w, pu.sample_rows(w.N, n_random=64, seed=3))


def test_charlm_dilated_sampled(cuda_lib):
    """bf16 B1 H8 N16384 D64 causal wl 512, dilation [1,1,2,2,3,3,4,4]: sampled rows."""
    w = workloads.PRESETS["charlm_dilated"]
    pu.run_longformer(cuda_lib, w, pu.sample_rows(w.N, dilations=(1, 2, 3, 4), n_random=64, seed=4))


@pytest.mark.parametrize("preset", ["long_8k", "long_32k", "long_128k"])
def test_long_scale_sampled(cuda_lib, preset):
    """bf16 B1 H16 D128, window 512/512, 128 random globals: sampled rows incl. global rows."""
    w = workloads.PRESETS[preset]
    g = workloads.global_positions(w)
    pu.run_longformer(cuda_lib, w, pu.sample_rows(w.N, globals_=g.tolist(), n_random=40, seed=5))


# ---------------------------------------------------------------- device-side status

def test_bad_global_list_reports_status(cuda_lib):
    lg = cuda_lib
    dev = torch.device("cuda")
    q = torch.randn(1, 2, 300, 64, device=dev).to(torch.bfloat16)
    for bad in ([5, 3], [0, 300], [-1, 4], [7, 7]):
        gidx = torch.tensor(bad, dtype=torch.int32, device=dev)
        lg.attn_fwd(q, q, q, 8, 8, None, False, gidx)
        assert lg.query_status(lg.attn_fwd.last_workspace) == lg.LG_ERR_GLOBAL_IDX
    # a good call on the same workspace reports OK again
    gidx = torch.tensor([3, 5], dtype=torch.int32, device=dev)
    ws = lg.attn_fwd.last_workspace
    lg.attn_fwd(q, q, q, 8, 8, None, False, gidx, workspace=ws)
    assert lg.query_status(ws) == 0


def test_repeat_calls_are_deterministic(cuda_lib):
    lg = cuda_lib
    w = W("repeat", "bf16", 1, 4, 1200, 128, 128, 128, (1, 2, 1, 3), False, (0, 600))
    inp = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    g = torch.from_numpy(inp["global_idx"]).to(dev)
    o1, l1 = lg.attn_fwd(q, k, v, w.w_left, w.w_right, w.dilations(), False, g)
    o1, l1 = o1.clone(), l1.clone()
    o2, l2 = lg.attn_fwd(q, k, v, w.w_left, w.w_right, w.dilations(), False, g)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("groups", [1, 4])
def test_host_entry_matches_device_entry(cuda_lib, groups):
    """lg_attn_fwd_host (host tensors, groups of heads overlapped with the copies)
    gives the same bits as lg_attn_fwd on the same inputs, and both match the oracle."""
    lg = cuda_lib
    w = W("host entry", "bf16", 2, 3, 900, 128, 70, 40, (1, 2, 3), False, (0, 11, 500, 899))
    inp = workloads.make_inputs(w)
    dev = torch.device("cuda")
    g = torch.from_numpy(inp["global_idx"]).to(dev)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    o_ref, l_ref = lg.attn_fwd(q, k, v, w.w_left, w.w_right, w.dilations(), False, g)
    qh, kh, vh = (inp[n].pin_memory() for n in ("q", "k", "v"))
    o_h, l_h = lg.attn_fwd_host(qh, kh, vh, w.w_left, w.w_right, w.dilations(), False, g, n_groups=groups)
    torch.cuda.synchronize()
    assert lg.query_status(lg.attn_fwd_host.last_workspace) == 0
    assert torch.equal(o_h, o_ref.cpu()) and torch.equal(l_h, l_ref.cpu())
    pu.run_longformer(cuda_lib, w)
