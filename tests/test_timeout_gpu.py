"""The device-side timeout path (needs a GB300).

Every wait of the tensor-core kernel is bounded.  Here a test switch makes the
kernel issue no TMA load and no MMA, so its first wait for a tile runs out
with nothing in flight (no fault, no hang: a flag that nothing sets).  The
call must report LG_ERR_TIMEOUT through lg_query_status, and the next normal
call on the same workspace must report LG_OK and match the CPU oracle, i.e.
the context and the workspace stay usable.
"""
import pytest
import torch

from sparse_long_sequence_window_gb300.workloads import Workload, make_inputs
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

CAP_CYCLES = 2_000_000      # about 1 ms at the SM clock


@pytest.mark.parametrize("w", [
    Workload("timeout D64", "bf16", 1, 2, 600, 64, 40, 40, (1, 3), False, (0, 300), seed=61),
    Workload("timeout D128", "bf16", 1, 2, 500, 128, 30, 30, (), True, None, 20, seed=62),
], ids=lambda w: w.name)
def test_wait_runs_out_then_next_call_is_clean(cuda_lib, w):
    lg = cuda_lib
    dev = torch.device("cuda")
    inp = make_inputs(w)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    g = torch.from_numpy(inp["global_idx"]).to(dev) if inp["global_idx"].size else None
    lg.debug_timeout_test(True, CAP_CYCLES)
    try:
        lg.attn_fwd(q, k, v, w.w_left, w.w_right, w.dilations(), w.causal, g)
        ws = lg.attn_fwd.last_workspace
        st = lg.query_status(ws)
    finally:
        lg.debug_timeout_test(False, 0)
    assert st == lg.LG_ERR_TIMEOUT, lg.status_string(st)
    # the same workspace, normal operation: LG_OK and oracle parity
    out, lse = lg.attn_fwd(q, k, v, w.w_left, w.w_right, w.dilations(), w.causal, g, workspace=ws)
    assert lg.query_status(ws) == lg.LG_OK
    from oracle import lg_oracle
    qn, kn, vn = (pu.to_np32(inp[n]) for n in ("q", "k", "v"))
    ref_o, ref_l = lg_oracle.attn_fwd(qn, kn, vn, w.w_left, w.w_right, w.dilations(), w.causal, inp["global_idx"])
    pu.compare(w.name, w.dtype, out.cpu(), lse.cpu(), ref_o, ref_l)


def test_etc_wait_runs_out_then_next_call_is_clean(cuda_lib):
    lg = cuda_lib
    w = Workload("timeout etc", "bf16", 1, 2, 400, 64, etc_G=30, radius=10, seed=63)
    dev = torch.device("cuda")
    inp = make_inputs(w)
    t = [inp[n].to(dev) for n in ("q", "k", "v", "q_g", "k_g", "v_g")]
    lg.debug_timeout_test(True, CAP_CYCLES)
    try:
        lg.etc_attn_fwd(*t, w.radius)
        ws = lg.etc_attn_fwd.last_workspace
        st = lg.query_status(ws)
    finally:
        lg.debug_timeout_test(False, 0)
    assert st == lg.LG_ERR_TIMEOUT, lg.status_string(st)
    pu.run_etc(lg, w)
