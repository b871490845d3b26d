"""The no-allocation entry point, lg_attn_fwd_noalloc (needs a GB300).

Some callers cannot allocate device memory while they run: code inside a host
framework that plans all device memory in advance, or a process whose GPU
memory is already taken by another allocator.  For them the library offers a
variant of lg_attn_fwd whose scratch space is a fixed array inside the
library.  These tests call it through the C ABI twice in a row, on two
different problems, and compare each result with the regular entry point's
(which uses a caller-allocated workspace) within the bf16 parity tolerances.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_long_sequence_window_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


def noalloc_fn(lib):
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f = lib.lg_attn_fwd_noalloc
    f.restype = i32
    f.argtypes = [vp] * 5 + [i32] * 7 + [vp, i32, vp, i32, f32, vp]
    return f


def call_noalloc(lg, w, q, k, v, g):
    f = noalloc_fn(lg.load())
    B, H, N, D = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    dil = np.ascontiguousarray(np.asarray(w.dilations(), dtype=np.int32))
    st = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), 1, B, H, N, D,
           w.w_left, w.w_right, dil.ctypes.data, int(w.causal),
           g.data_ptr() if g is not None else None, 0 if g is None else g.numel(), 0.0,
           torch.cuda.current_stream().cuda_stream)
    return st, out, lse


PROBLEMS = [
    Workload("noalloc a", "bf16", 1, 4, 1000, 64, 60, 20, (1, 2, 3, 4), False, (0, 5, 999), seed=41),
    Workload("noalloc b", "bf16", 2, 3, 777, 128, 100, 100, (1, 1, 2), True, None, 70, seed=42),
]


def test_noalloc_matches_workspace_entry_point_twice(cuda_lib):
    lg = cuda_lib
    dev = torch.device("cuda")
    for w in PROBLEMS:                           # two calls in a row, sharing the fixed scratch
        inp = make_inputs(w)
        q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
        g = torch.from_numpy(inp["global_idx"]).to(dev) if inp["global_idx"].size else None
        ref_out, ref_lse = lg.attn_fwd(q, k, v, w.w_left, w.w_right, w.dilations(), w.causal, g)
        st, out, lse = call_noalloc(lg, w, q, k, v, g)
        assert st == 0, lg.status_string(st)
        torch.cuda.synchronize()
        err = (out.float() - ref_out.float()).abs()
        assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
        assert (lse - ref_lse).abs().max().item() <= 1e-3


def test_noalloc_refuses_problems_beyond_the_scratch(cuda_lib):
    lg = cuda_lib
    need = lg.attn_fwd_workspace_size(1, 16, 131072, 128, 128, 1)
    assert need > SCRATCH_BYTES
    f = noalloc_fn(lg.load())
    dil = (ctypes.c_int32 * 16)(*([1] * 16))
    fake = 1 << 20   # never dereferenced: the size check returns first
    st = f(fake, fake, fake, fake, fake, 1, 1, 16, 131072, 128, 512, 512, ctypes.cast(dil, ctypes.c_void_p),
           0, fake, 128, 0.0, None)
    assert st == lg.LG_ERR_WORKSPACE
