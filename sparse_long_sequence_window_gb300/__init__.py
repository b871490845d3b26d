"""Window + dilation + global sparse self-attention (forward and backward) for one GB300 GPU.

Python binding of the C ABI in ``include/lg_attn.h``.  This module only
marshals arguments (device pointers, sizes, the current CUDA stream) into the
shared library ``liblg_attn.so``; every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.

There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "LgError", "load", "attn_fwd", "attn_fwd_host", "etc_attn_fwd", "attn_fwd_workspace_size",
    "attn_bwd", "etc_attn_bwd", "attn_bwd_workspace_size", "etc_attn_bwd_workspace_size",
    "longnet_attn_fwd", "longnet_count_pairs", "longnet_attn_fwd_workspace_size",
    "etc_struct_attn_fwd", "etc_struct_attn_fwd_workspace_size",
    "etc_attn_fwd_workspace_size", "query_status", "count_pairs", "etc_count_pairs",
    "profile_begin", "profile_end", "status_string", "debug_timeout_test", "LIB_PATH",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblg_attn.so")

LG_OK, LG_ERR_INVALID_ARG, LG_ERR_UNSUPPORTED, LG_ERR_CUDA, LG_ERR_TIMEOUT, LG_ERR_WORKSPACE, LG_ERR_GLOBAL_IDX = range(7)
LG_F32, LG_BF16 = 0, 1

_lib = None


class LgError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def load() -> ctypes.CDLL:
    """Loads liblg_attn.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m sparse_long_sequence_window_gb300._build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    lib.lg_status_string.restype = ctypes.c_char_p
    lib.lg_status_string.argtypes = [i32]
    lib.lg_version.restype = ctypes.c_char_p
    lib.lg_attn_fwd_workspace_size.restype = sz
    lib.lg_attn_fwd_workspace_size.argtypes = [i32] * 5 + [i32]
    lib.lg_etc_attn_fwd_workspace_size.restype = sz
    lib.lg_etc_attn_fwd_workspace_size.argtypes = [i32] * 5 + [i32]
    lib.lg_attn_fwd.restype = i32
    lib.lg_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, i32, vp, i32, f32,
                                vp, sz, vp]
    lib.lg_attn_fwd_gproj.restype = i32
    lib.lg_attn_fwd_gproj.argtypes = [vp] * 8 + [i32] * 7 + [vp, i32, vp, i32, f32, vp, sz, vp]
    lib.lg_attn_fwd_host.restype = i32
    lib.lg_attn_fwd_host.argtypes = [vp] * 10 + [i32] * 7 + [vp, i32, vp, i32, f32, vp, sz, i32, vp]
    lib.lg_etc_attn_fwd.restype = i32
    lib.lg_etc_attn_fwd.argtypes = [vp] * 10 + [i32] * 7 + [f32, vp, sz, vp]
    lib.lg_query_status.restype = i32
    lib.lg_query_status.argtypes = [vp, vp]
    lib.lg_count_pairs.restype = ctypes.c_int64
    lib.lg_count_pairs.argtypes = [i32, i32, i32, i32, i32, vp, i32]
    lib.lg_etc_count_pairs.restype = ctypes.c_int64
    lib.lg_etc_count_pairs.argtypes = [i32, i32, i32]
    lib.lg_attn_bwd_workspace_size.restype = sz
    lib.lg_attn_bwd_workspace_size.argtypes = [i32] * 6
    lib.lg_etc_attn_bwd_workspace_size.restype = sz
    lib.lg_etc_attn_bwd_workspace_size.argtypes = [i32] * 6
    lib.lg_attn_bwd.restype = i32
    lib.lg_attn_bwd.argtypes = [vp] * 9 + [i32] * 7 + [vp, i32, vp, i32, f32, vp, sz, vp]
    lib.lg_etc_attn_bwd.restype = i32
    lib.lg_etc_attn_bwd.argtypes = [vp] * 18 + [i32] * 7 + [f32, vp, sz, vp]
    lib.lg_longnet_attn_fwd_workspace_size.restype = sz
    lib.lg_longnet_attn_fwd_workspace_size.argtypes = [i32] * 5 + [vp, vp, i32]
    lib.lg_longnet_attn_fwd.restype = i32
    lib.lg_longnet_attn_fwd.argtypes = [vp] * 5 + [i32] * 6 + [vp, vp, i32, f32, vp, sz, vp]
    lib.lg_longnet_count_pairs.restype = ctypes.c_int64
    lib.lg_longnet_count_pairs.argtypes = [i32, i32, vp, vp, i32, i32]
    lib.lg_etc_struct_attn_fwd_workspace_size.restype = sz
    lib.lg_etc_struct_attn_fwd_workspace_size.argtypes = [i32] * 8
    lib.lg_etc_struct_attn_fwd.restype = i32
    lib.lg_etc_struct_attn_fwd.argtypes = [vp] * 11 + [i32] + [vp] * 4 + [i32] * 7 + [f32, vp, sz, vp]
    lib.lg_debug_timeout_test.restype = i32
    lib.lg_debug_timeout_test.argtypes = [i32, ctypes.c_longlong]
    lib.lg_profile_begin.restype = i32
    lib.lg_profile_begin.argtypes = []
    lib.lg_profile_end.restype = i32
    lib.lg_profile_end.argtypes = [ctypes.POINTER(f32), ctypes.POINTER(i32)]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().lg_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != LG_OK:
        raise LgError(status, what)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return LG_F32
    if t.dtype == torch.bfloat16:
        return LG_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")


def _ptr(t) -> int:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _same(ref, what, *ts):
    """Every tensor in ts has ref's shape, dtype and device (the library trusts the sizes it is given)."""
    for t in ts:
        if t.shape != ref.shape or t.dtype != ref.dtype or t.device != ref.device:
            raise ValueError(f"{what}: expected {tuple(ref.shape)} {ref.dtype} on {ref.device}, "
                             f"got {tuple(t.shape)} {t.dtype} on {t.device}")


def _check_out(t, shape, dtype, device, what):
    if t.shape != tuple(shape) or t.dtype != dtype or t.device != device:
        raise ValueError(f"{what}: expected {tuple(shape)} {dtype} on {device}, "
                         f"got {tuple(t.shape)} {t.dtype} on {t.device}")


def _stream(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _keep_for(stream, *tensors):
    """Tensors allocated here but used by work queued on another stream than the
    current one: tell the caching allocator, so that their memory is not handed
    out again before that work has completed."""
    import torch
    if stream is None or stream == torch.cuda.current_stream(stream.device):
        return
    for t in tensors:
        if t is not None and t.is_cuda:
            t.record_stream(stream)


def attn_fwd_workspace_size(B, H, N, D, n_global, dtype_code) -> int:
    return int(load().lg_attn_fwd_workspace_size(B, H, N, D, n_global, dtype_code))


def etc_attn_fwd_workspace_size(B, H, L, G, D, dtype_code) -> int:
    return int(load().lg_etc_attn_fwd_workspace_size(B, H, L, G, D, dtype_code))


def _workspace(nbytes: int, device, workspace):
    import torch
    if workspace is not None:
        if workspace.device != device or not workspace.is_contiguous():
            raise ValueError(f"workspace must be a contiguous tensor on {device}")
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def attn_fwd(q, k, v, w_left: int, w_right: int, dilation: Optional[Sequence[int]] = None,
             causal: bool = False, global_idx=None, scale: Optional[float] = None,
             out=None, lse=None, workspace=None, stream=None, q_global=None, k_global=None, v_global=None):
    """Longformer-style window + dilation + global attention forward.

    q, k, v: CUDA tensors [B, H, N, D] (float32 or bfloat16, contiguous).
    dilation: H ints (default all 1).  global_idx: sorted unique int32 CUDA
    tensor of positions (or None).  q_global, k_global, v_global: optional
    separate projections for global attention (all three or none, shaped like
    q; lg_attn_fwd_gproj).  Returns (out [B, H, N, D], lse [B, H, N]
    float32).  Asynchronous on the current stream.
    """
    import torch
    lib = load()
    if q.dim() != 4 or not q.is_cuda:
        raise ValueError("q must be a CUDA tensor [B, H, N, D]")
    _same(q, "k", k)
    _same(q, "v", v)
    B, H, N, D = q.shape
    dil = np.ascontiguousarray(np.asarray(dilation if dilation is not None else [1] * H, dtype=np.int32))
    if dil.size != H:
        raise ValueError("dilation needs H entries")
    n_global = 0 if global_idx is None else int(global_idx.numel())
    if global_idx is not None and (global_idx.dtype != torch.int32 or global_idx.device != q.device):
        raise TypeError("global_idx must be an int32 tensor on q's device")
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    _check_out(out, q.shape, q.dtype, q.device, "out")
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_out(lse, (B, H, N), torch.float32, q.device, "lse")
    need = attn_fwd_workspace_size(B, H, N, D, n_global, dt)
    ws = _workspace(need, q.device, workspace)
    gp = (q_global, k_global, v_global)
    if any(x is not None for x in gp):
        if any(x is None for x in gp):
            raise ValueError("q_global, k_global and v_global go together")
        _same(q, "global projections", *gp)
        st = lib.lg_attn_fwd_gproj(_ptr(q), _ptr(k), _ptr(v), *(_ptr(x) for x in gp), _ptr(out), _ptr(lse), dt,
                                   B, H, N, D, int(w_left), int(w_right), dil.ctypes.data, int(bool(causal)),
                                   _ptr(global_idx) if n_global else None, n_global,
                                   float(scale) if scale else 0.0, ws.data_ptr(), _nbytes(ws), _stream(stream))
        _check(st, "lg_attn_fwd_gproj")
    else:
        st = lib.lg_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), dt, B, H, N, D,
                             int(w_left), int(w_right), dil.ctypes.data, int(bool(causal)),
                             _ptr(global_idx) if n_global else None, n_global,
                             float(scale) if scale else 0.0, ws.data_ptr(), _nbytes(ws), _stream(stream))
        _check(st, "lg_attn_fwd")
    if workspace is None:
        _keep_for(stream, ws)
    attn_fwd.last_workspace = ws
    return out, lse


def attn_fwd_host(q_h, k_h, v_h, w_left: int, w_right: int, dilation: Optional[Sequence[int]] = None,
                  causal: bool = False, global_idx=None, scale: Optional[float] = None,
                  out_h=None, lse_h=None, staging=None, workspace=None, n_groups: int = 4, stream=None):
    """attn_fwd on host tensors: q_h, k_h, v_h [B, H, N, D] in (preferably pinned)
    host memory; the library copies them in and out/lse back, overlapping the
    copies of one group of heads with the kernels of another.  staging: the
    device buffers (q, k, v, out, lse) it may use (allocated here if None).
    global_idx: int32 CUDA tensor (or None).  Asynchronous on the current
    stream; returns (out_h, lse_h).
    """
    import torch
    lib = load()
    if q_h.dim() != 4 or q_h.is_cuda:
        raise ValueError("q_h must be a host tensor [B, H, N, D]")
    _same(q_h, "k_h", k_h)
    _same(q_h, "v_h", v_h)
    B, H, N, D = q_h.shape
    dil = np.ascontiguousarray(np.asarray(dilation if dilation is not None else [1] * H, dtype=np.int32))
    if dil.size != H:
        raise ValueError("dilation needs H entries")
    n_global = 0 if global_idx is None else int(global_idx.numel())
    if global_idx is not None and (global_idx.dtype != torch.int32 or not global_idx.is_cuda):
        raise TypeError("global_idx must be an int32 CUDA tensor")
    dt = _dtype_code(q_h)
    dev = torch.device("cuda", torch.cuda.current_device())
    if out_h is None:
        out_h = torch.empty(q_h.shape, dtype=q_h.dtype, pin_memory=True)
    if lse_h is None:
        lse_h = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
    _check_out(out_h, q_h.shape, q_h.dtype, q_h.device, "out_h")
    _check_out(lse_h, (B, H, N), torch.float32, q_h.device, "lse_h")
    own_staging = staging is None
    if own_staging:
        staging = tuple(torch.empty(q_h.shape, dtype=q_h.dtype, device=dev) for _ in range(4)) + (
            torch.empty((B, H, N), dtype=torch.float32, device=dev),)
    if len(staging) != 5:
        raise ValueError("staging holds five device tensors: q, k, v, out, lse")
    for t, name in zip(staging[:4], ("q", "k", "v", "out")):
        _check_out(t, q_h.shape, q_h.dtype, dev, f"staging {name}")
    _check_out(staging[4], (B, H, N), torch.float32, dev, "staging lse")
    need = attn_fwd_workspace_size(B, H, N, D, n_global, dt)
    ws = _workspace(need, dev, workspace)
    st = lib.lg_attn_fwd_host(_ptr(q_h), _ptr(k_h), _ptr(v_h), _ptr(out_h), _ptr(lse_h),
                              *(_ptr(x) for x in staging), dt, B, H, N, D, int(w_left), int(w_right),
                              dil.ctypes.data, int(bool(causal)), _ptr(global_idx) if n_global else None, n_global,
                              float(scale) if scale else 0.0, ws.data_ptr(), _nbytes(ws), int(n_groups),
                              _stream(stream))
    _check(st, "lg_attn_fwd_host")
    # The library queues work on its own copy streams too, all joined into
    # `stream`; buffers allocated here must outlive that stream's work.
    s = stream if stream is not None else torch.cuda.current_stream()
    if own_staging:
        for t in staging:
            t.record_stream(s)
    if workspace is None:
        ws.record_stream(s)
    attn_fwd_host.last_workspace = ws
    return out_h, lse_h


def etc_attn_fwd(q_l, k_l, v_l, q_g, k_g, v_g, radius: int, scale: Optional[float] = None,
                 out_l=None, out_g=None, lse_l=None, lse_g=None, workspace=None, stream=None):
    """ETC-style global-local attention forward.  Returns (out_l, out_g, lse_l, lse_g)."""
    import torch
    lib = load()
    if q_l.dim() != 4 or q_g.dim() != 4 or not q_l.is_cuda:
        raise ValueError("q_l, q_g must be CUDA tensors [B, H, L, D] and [B, H, G, D]")
    _same(q_l, "k_l", k_l)
    _same(q_l, "v_l", v_l)
    _same(q_g, "k_g", k_g)
    _same(q_g, "v_g", v_g)
    B, H, L, D = q_l.shape
    G = q_g.shape[2]
    if q_g.shape[:2] != q_l.shape[:2] or q_g.shape[3] != D or q_g.dtype != q_l.dtype or q_g.device != q_l.device:
        raise ValueError("q_g must match q_l in B, H, D, dtype and device")
    dt = _dtype_code(q_l)
    out_l = torch.empty_like(q_l) if out_l is None else out_l
    out_g = torch.empty_like(q_g) if out_g is None else out_g
    lse_l = torch.empty((B, H, L), dtype=torch.float32, device=q_l.device) if lse_l is None else lse_l
    lse_g = torch.empty((B, H, G), dtype=torch.float32, device=q_l.device) if lse_g is None else lse_g
    _check_out(out_l, q_l.shape, q_l.dtype, q_l.device, "out_l")
    _check_out(out_g, q_g.shape, q_g.dtype, q_l.device, "out_g")
    _check_out(lse_l, (B, H, L), torch.float32, q_l.device, "lse_l")
    _check_out(lse_g, (B, H, G), torch.float32, q_l.device, "lse_g")
    need = etc_attn_fwd_workspace_size(B, H, L, G, D, dt)
    ws = _workspace(need, q_l.device, workspace)
    st = lib.lg_etc_attn_fwd(_ptr(q_l), _ptr(k_l), _ptr(v_l), _ptr(q_g), _ptr(k_g), _ptr(v_g),
                             _ptr(out_l), _ptr(out_g), _ptr(lse_l), _ptr(lse_g), dt, B, H, L, G, D,
                             int(radius), float(scale) if scale else 0.0, ws.data_ptr(), _nbytes(ws),
                             _stream(stream))
    _check(st, "lg_etc_attn_fwd")
    if workspace is None:
        _keep_for(stream, ws)
    etc_attn_fwd.last_workspace = ws
    return out_l, out_g, lse_l, lse_g


def attn_bwd_workspace_size(B, H, N, D, n_global, dtype_code) -> int:
    return int(load().lg_attn_bwd_workspace_size(B, H, N, D, n_global, dtype_code))


def etc_attn_bwd_workspace_size(B, H, L, G, D, dtype_code) -> int:
    return int(load().lg_etc_attn_bwd_workspace_size(B, H, L, G, D, dtype_code))


def attn_bwd(q, k, v, out, lse, dout, w_left: int, w_right: int, dilation: Optional[Sequence[int]] = None,
             causal: bool = False, global_idx=None, scale: Optional[float] = None,
             dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward of attn_fwd: (dq, dk, dv) given the forward's out and lse and dout.

    Same arguments as attn_fwd plus out [B, H, N, D], lse [B, H, N] float32 and
    dout [B, H, N, D].  Asynchronous on the current stream.
    """
    import torch
    lib = load()
    if q.dim() != 4 or not q.is_cuda:
        raise ValueError("q must be a CUDA tensor [B, H, N, D]")
    _same(q, "k", k, v, out, dout)
    B, H, N, D = q.shape
    _check_out(lse, (B, H, N), torch.float32, q.device, "lse")
    dil = np.ascontiguousarray(np.asarray(dilation if dilation is not None else [1] * H, dtype=np.int32))
    if dil.size != H:
        raise ValueError("dilation needs H entries")
    n_global = 0 if global_idx is None else int(global_idx.numel())
    if global_idx is not None and (global_idx.dtype != torch.int32 or global_idx.device != q.device):
        raise TypeError("global_idx must be an int32 tensor on q's device")
    dt = _dtype_code(q)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for t, name in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check_out(t, q.shape, q.dtype, q.device, name)
    need = attn_bwd_workspace_size(B, H, N, D, n_global, dt)
    ws = _workspace(need, q.device, workspace)
    st = lib.lg_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                         dt, B, H, N, D, int(w_left), int(w_right), dil.ctypes.data, int(bool(causal)),
                         _ptr(global_idx) if n_global else None, n_global, float(scale) if scale else 0.0,
                         ws.data_ptr(), _nbytes(ws), _stream(stream))
    _check(st, "lg_attn_bwd")
    if workspace is None:
        _keep_for(stream, ws)
    attn_bwd.last_workspace = ws
    return dq, dk, dv


def etc_attn_bwd(q_l, k_l, v_l, q_g, k_g, v_g, out_l, out_g, lse_l, lse_g, dout_l, dout_g, radius: int,
                 scale: Optional[float] = None, workspace=None, stream=None):
    """Backward of etc_attn_fwd.  Returns (dq_l, dk_l, dv_l, dq_g, dk_g, dv_g)."""
    import torch
    lib = load()
    if q_l.dim() != 4 or q_g.dim() != 4 or not q_l.is_cuda:
        raise ValueError("q_l, q_g must be CUDA tensors [B, H, L, D] and [B, H, G, D]")
    _same(q_l, "long input", k_l, v_l, out_l, dout_l)
    _same(q_g, "global input", k_g, v_g, out_g, dout_g)
    B, H, L, D = q_l.shape
    G = q_g.shape[2]
    if q_g.shape[:2] != q_l.shape[:2] or q_g.shape[3] != D or q_g.dtype != q_l.dtype or q_g.device != q_l.device:
        raise ValueError("q_g must match q_l in B, H, D, dtype and device")
    _check_out(lse_l, (B, H, L), torch.float32, q_l.device, "lse_l")
    _check_out(lse_g, (B, H, G), torch.float32, q_l.device, "lse_g")
    dt = _dtype_code(q_l)
    grads = [torch.empty_like(x) for x in (q_l, q_l, q_l, q_g, q_g, q_g)]
    need = etc_attn_bwd_workspace_size(B, H, L, G, D, dt)
    ws = _workspace(need, q_l.device, workspace)
    st = lib.lg_etc_attn_bwd(_ptr(q_l), _ptr(k_l), _ptr(v_l), _ptr(q_g), _ptr(k_g), _ptr(v_g),
                             _ptr(out_l), _ptr(out_g), _ptr(lse_l), _ptr(lse_g), _ptr(dout_l), _ptr(dout_g),
                             *(_ptr(x) for x in grads), dt, B, H, L, G, D, int(radius),
                             float(scale) if scale else 0.0, ws.data_ptr(), _nbytes(ws), _stream(stream))
    _check(st, "lg_etc_attn_bwd")
    if workspace is None:
        _keep_for(stream, ws)
    etc_attn_bwd.last_workspace = ws
    return tuple(grads)


def etc_struct_attn_fwd(q_l, k_l, v_l, q_g, k_g, v_g, radius, rel_k=None, code_l2l=None, code_l2g=None,
                        code_g2l=None, code_g2g=None, scale: Optional[float] = None, out_l=None, out_g=None,
                        lse_l=None, lse_g=None, workspace=None, stream=None):
    """ETC attention with relative-position labels and per-instance masks (lg_etc_struct_attn_fwd).

    Long tensors [B, H, L, D], global [B, H, G, D] (bf16 CUDA); rel_k [H, V, D] or None; codes uint8
    CUDA tensors code_l2l [B, L, 2r+1], code_l2g [B, L, G], code_g2l [B, G, L], code_g2g [B, G, G]
    (label in bits 0..6, 128 = blocked) or None.  Returns (out_l, out_g, lse_l, lse_g)."""
    import torch
    lib = load()
    if q_l.dim() != 4 or not q_l.is_cuda:
        raise ValueError("q_l must be a CUDA tensor [B, H, L, D]")
    _same(q_l, "k_l", k_l, v_l)
    _same(q_g, "k_g", k_g, v_g)
    B, H, L, D = q_l.shape
    G = q_g.shape[2]
    if tuple(q_g.shape) != (B, H, G, D) or q_g.dtype != q_l.dtype or q_g.device != q_l.device:
        raise ValueError("q_g must be [B, H, G, D] with q_l's dtype and device")
    dt = _dtype_code(q_l)
    n_labels = 0
    if rel_k is not None:
        if rel_k.dim() != 3 or rel_k.shape[0] != H or rel_k.shape[2] != D or rel_k.dtype != q_l.dtype \
                or rel_k.device != q_l.device or not rel_k.is_contiguous():
            raise ValueError("rel_k must be a contiguous [H, V, D] tensor of q_l's dtype and device")
        n_labels = int(rel_k.shape[1])
    shapes = {"code_l2l": (B, L, 2 * int(radius) + 1), "code_l2g": (B, L, G), "code_g2l": (B, G, L),
              "code_g2g": (B, G, G)}
    codes = {"code_l2l": code_l2l, "code_l2g": code_l2g, "code_g2l": code_g2l, "code_g2g": code_g2g}
    for name, c in codes.items():
        if c is not None and (tuple(c.shape) != shapes[name] or c.dtype != torch.uint8 or c.device != q_l.device
                              or not c.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous uint8 tensor {shapes[name]} on {q_l.device}")
    out_l = torch.empty_like(q_l) if out_l is None else out_l
    out_g = torch.empty_like(q_g) if out_g is None else out_g
    lse_l = torch.empty((B, H, L), dtype=torch.float32, device=q_l.device) if lse_l is None else lse_l
    lse_g = torch.empty((B, H, G), dtype=torch.float32, device=q_l.device) if lse_g is None else lse_g
    _check_out(out_l, q_l.shape, q_l.dtype, q_l.device, "out_l")
    _check_out(out_g, q_g.shape, q_g.dtype, q_g.device, "out_g")
    _check_out(lse_l, (B, H, L), torch.float32, q_l.device, "lse_l")
    _check_out(lse_g, (B, H, G), torch.float32, q_l.device, "lse_g")
    need = int(lib.lg_etc_struct_attn_fwd_workspace_size(B, H, L, G, D, int(radius), n_labels, dt))
    if need == 0:
        raise NotImplementedError("lg_etc_struct_attn_fwd: unsupported shape, dtype or label count")
    ws = _workspace(need, q_l.device, workspace)
    cp = [None if c is None else _ptr(c) for c in codes.values()]
    st = lib.lg_etc_struct_attn_fwd(_ptr(q_l), _ptr(k_l), _ptr(v_l), _ptr(q_g), _ptr(k_g), _ptr(v_g), _ptr(out_l),
                                    _ptr(out_g), _ptr(lse_l), _ptr(lse_g), None if rel_k is None else _ptr(rel_k),
                                    n_labels, *cp, dt, B, H, L, G, D, int(radius),
                                    float(scale) if scale else 0.0, ws.data_ptr(), _nbytes(ws), _stream(stream))
    _check(st, "lg_etc_struct_attn_fwd")
    if workspace is None:
        _keep_for(stream, ws)
    etc_struct_attn_fwd.last_workspace = ws
    return out_l, out_g, lse_l, lse_g


def etc_struct_attn_fwd_workspace_size(B, H, L, G, D, radius, n_labels, dtype=LG_BF16) -> int:
    return int(load().lg_etc_struct_attn_fwd_workspace_size(B, H, L, G, D, radius, n_labels, int(dtype)))


def longnet_attn_fwd(q, k, v, seg_w: Sequence[int], seg_r: Sequence[int], causal: bool = False,
                     scale: Optional[float] = None, out=None, lse=None, workspace=None, stream=None):
    """LongNet mixture of dilated attentions (lg_longnet_attn_fwd): patterns (seg_w[k], seg_r[k]),
    head h offset h mod r.  q, k, v: bf16 CUDA tensors [B, H, N, D].  Returns (out, lse)."""
    import torch
    lib = load()
    if q.dim() != 4 or not q.is_cuda:
        raise ValueError("q must be a CUDA tensor [B, H, N, D]")
    _same(q, "k", k, v)
    B, H, N, D = q.shape
    sw = np.ascontiguousarray(np.asarray(seg_w, dtype=np.int32))
    sr = np.ascontiguousarray(np.asarray(seg_r, dtype=np.int32))
    if sw.size != sr.size:
        raise ValueError("seg_w and seg_r need the same length")
    dt = _dtype_code(q)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_out(out, q.shape, q.dtype, q.device, "out")
    _check_out(lse, (B, H, N), torch.float32, q.device, "lse")
    need = int(lib.lg_longnet_attn_fwd_workspace_size(B, H, N, D, int(sw.size), sw.ctypes.data, sr.ctypes.data, dt))
    if need == 0:
        raise NotImplementedError("lg_longnet_attn_fwd: unsupported shape, dtype or patterns")
    ws = _workspace(need, q.device, workspace)
    st = lib.lg_longnet_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), dt, B, H, N, D, int(sw.size),
                                 sw.ctypes.data, sr.ctypes.data, int(bool(causal)), float(scale) if scale else 0.0,
                                 ws.data_ptr(), _nbytes(ws), _stream(stream))
    _check(st, "lg_longnet_attn_fwd")
    if workspace is None:
        _keep_for(stream, ws)
    longnet_attn_fwd.last_workspace = ws
    return out, lse


def longnet_attn_fwd_workspace_size(B, H, N, D, seg_w, seg_r, dtype=LG_BF16) -> int:
    sw = np.ascontiguousarray(np.asarray(seg_w, dtype=np.int32))
    sr = np.ascontiguousarray(np.asarray(seg_r, dtype=np.int32))
    return int(load().lg_longnet_attn_fwd_workspace_size(B, H, N, D, int(sw.size), sw.ctypes.data, sr.ctypes.data,
                                                          int(dtype)))


def longnet_count_pairs(N, seg_w, seg_r, causal, head) -> int:
    sw = np.ascontiguousarray(np.asarray(seg_w, dtype=np.int32))
    sr = np.ascontiguousarray(np.asarray(seg_r, dtype=np.int32))
    r = load().lg_longnet_count_pairs(int(N), int(sw.size), sw.ctypes.data, sr.ctypes.data, int(bool(causal)),
                                      int(head))
    if r < 0:
        raise ValueError("invalid arguments to lg_longnet_count_pairs")
    return int(r)


def query_status(workspace, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status of the last call."""
    return int(load().lg_query_status(workspace.data_ptr(), _stream(stream)))


def count_pairs(N, w_left, w_right, dilation, causal, global_idx_host=None) -> int:
    """Allowed pairs of one head (host computation in the library)."""
    g = np.ascontiguousarray(np.asarray([] if global_idx_host is None else global_idx_host, dtype=np.int32))
    r = load().lg_count_pairs(int(N), int(w_left), int(w_right), int(dilation), int(bool(causal)),
                              g.ctypes.data if g.size else None, int(g.size))
    if r < 0:
        raise ValueError("invalid arguments to lg_count_pairs")
    return int(r)


def etc_count_pairs(L, G, radius) -> int:
    r = load().lg_etc_count_pairs(int(L), int(G), int(radius))
    if r < 0:
        raise ValueError("invalid arguments to lg_etc_count_pairs")
    return int(r)


def debug_timeout_test(withhold: bool, wait_cap_cycles: int = 0):
    """Testing aid of the timeout path: with withhold, later bf16 calls issue no
    loads or MMAs, so their first bounded wait runs out (after wait_cap_cycles
    SM cycles; <= 0 restores the default cap) and lg_query_status reports
    LG_ERR_TIMEOUT.  debug_timeout_test(False) restores normal operation."""
    _check(load().lg_debug_timeout_test(int(bool(withhold)), int(wait_cap_cycles)), "lg_debug_timeout_test")


def profile_begin():
    _check(load().lg_profile_begin(), "lg_profile_begin")


def profile_end():
    """Returns (total milliseconds, launches) of the dominant kernel since profile_begin."""
    ms = ctypes.c_float(0.0)
    n = ctypes.c_int(0)
    _check(load().lg_profile_end(ctypes.byref(ms), ctypes.byref(n)), "lg_profile_end")
    return float(ms.value), int(n.value)
