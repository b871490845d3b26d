"""The C-ABI library without a GPU: it loads, exports every declared symbol,
rejects bad arguments before touching CUDA, and its host-side pair count
agrees with the CPU oracle's (independently written) counts."""
import ctypes
import os
import re

import numpy as np
import pytest

import sparse_long_sequence_window_gb300 as lg
from oracle import lg_oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lg_attn.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(lg.LIB_PATH):
        from sparse_long_sequence_window_gb300 import _build
        _build.build()
    return lg.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lg_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(7):
        assert lg.status_string(s).startswith("LG_")
    assert b"sm_103a" in lib.lg_version()


FAKE = 1 << 20  # a 16-byte-aligned non-null address; never dereferenced on these paths


def call_fwd(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=FAKE, dt=lg.LG_BF16, B=1, H=2, N=256, D=64, wl=8, wr=8,
             dil=(ctypes.c_int32 * 2)(1, 1), causal=0, gidx=None, ng=0, scale=0.0, ws=FAKE,
             wsb=1 << 30, stream=None)
    a.update(over)
    return lib.lg_attn_fwd(a["q"], a["k"], a["v"], a["out"], a["lse"], a["dt"], a["B"], a["H"], a["N"],
                           a["D"], a["wl"], a["wr"], ctypes.cast(a["dil"], ctypes.c_void_p) if a["dil"] else None,
                           a["causal"], a["gidx"], a["ng"], a["scale"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("over,expect", [
    (dict(q=None), lg.LG_ERR_INVALID_ARG),
    (dict(out=FAKE + 8), lg.LG_ERR_INVALID_ARG),
    (dict(N=0), lg.LG_ERR_INVALID_ARG),
    (dict(B=0), lg.LG_ERR_INVALID_ARG),
    (dict(wl=-1), lg.LG_ERR_INVALID_ARG),
    (dict(causal=2), lg.LG_ERR_INVALID_ARG),
    (dict(dil=(ctypes.c_int32 * 2)(1, 0)), lg.LG_ERR_INVALID_ARG),
    (dict(dil=None), lg.LG_ERR_INVALID_ARG),
    (dict(ng=3, gidx=None), lg.LG_ERR_INVALID_ARG),
    (dict(ng=300), lg.LG_ERR_INVALID_ARG),
    (dict(dt=7), lg.LG_ERR_INVALID_ARG),
    (dict(D=96), lg.LG_ERR_UNSUPPORTED),
    (dict(dt=lg.LG_F32, D=130), lg.LG_ERR_UNSUPPORTED),
    (dict(dil=(ctypes.c_int32 * 2)(1, 9)), lg.LG_ERR_UNSUPPORTED),
    (dict(H=200, dil=(ctypes.c_int32 * 200)(*([1] * 200))), lg.LG_ERR_UNSUPPORTED),
    (dict(ws=None), lg.LG_ERR_WORKSPACE),
    (dict(ws=FAKE + 16), lg.LG_ERR_WORKSPACE),
    (dict(wsb=16), lg.LG_ERR_WORKSPACE),
])
def test_argument_errors_return_before_launch(lib, over, expect):
    assert call_fwd(lib, **over) == expect


def test_etc_argument_errors(lib):
    args = [FAKE] * 10 + [lg.LG_BF16, 1, 2, 100, 8, 64, 4, 0.0, FAKE, 1 << 30, None]
    bad = list(args); bad[0] = None
    assert lib.lg_etc_attn_fwd(*bad) == lg.LG_ERR_INVALID_ARG
    bad = list(args); bad[13] = 0        # L = 0
    assert lib.lg_etc_attn_fwd(*bad) == lg.LG_ERR_INVALID_ARG
    bad = list(args); bad[16] = -1       # radius
    assert lib.lg_etc_attn_fwd(*bad) == lg.LG_ERR_INVALID_ARG
    bad = list(args); bad[15] = 32       # D
    assert lib.lg_etc_attn_fwd(*bad) == lg.LG_ERR_UNSUPPORTED
    bad = list(args); bad[19] = 64       # workspace bytes
    assert lib.lg_etc_attn_fwd(*bad) == lg.LG_ERR_WORKSPACE


def test_workspace_sizes(lib):
    assert lg.attn_fwd_workspace_size(1, 2, 512, 64, 0, lg.LG_F32) == 256
    base = lg.attn_fwd_workspace_size(1, 12, 4096, 64, 0, lg.LG_BF16)
    with_g = lg.attn_fwd_workspace_size(1, 12, 4096, 64, 65, lg.LG_BF16)
    # bf16: the status word and a table of 64-byte work-unit records (at least
    # one per pair of 128-row query tiles of every head)
    assert base >= 256 + 64 * 12 * (4096 // 256) and base % 256 == 0
    assert with_g > base
    # the partial statistics grow with the number of key splits (linear in N)
    a = lg.attn_fwd_workspace_size(1, 16, 8192, 128, 128, lg.LG_BF16)
    b = lg.attn_fwd_workspace_size(1, 16, 32768, 128, 128, lg.LG_BF16)
    assert b > a
    # the partials have room for the finest split a launch may choose: rows of
    # up to 64 key tiles may be cut into 8-tile pieces, two partials per piece
    # of D + 2 floats (acc and (m, l)) for every (head, global row)
    assert with_g - base >= 12 * 65 * (2 * (4096 // 128 // 8)) * (64 + 2) * 4
    assert lg.attn_fwd_workspace_size(0, 1, 1, 64, 0, lg.LG_BF16) == 0
    assert lg.etc_attn_fwd_workspace_size(2, 12, 4096, 256, 64, lg.LG_BF16) > 256


def test_count_pairs_agrees_with_oracle(lib):
    rng = np.random.default_rng(21)
    for _ in range(150):
        N = int(rng.integers(1, 90))
        wl, wr = int(rng.integers(0, 15)), int(rng.integers(0, 15))
        d = int(rng.integers(1, 7)); causal = bool(rng.integers(0, 2))
        ng = int(rng.integers(0, min(N, 7) + 1))
        g = sorted(rng.choice(N, size=ng, replace=False).tolist()) if ng else []
        expect = lg_oracle.count_pairs_bruteforce(N, wl, wr, d, causal, g)
        assert lg.count_pairs(N, wl, wr, d, causal, g) == expect
    # large sizes: against the oracle's closed form
    for N, wl, wr, d, causal, g in [(4096, 256, 256, 1, False, list(range(65))),
                                    (16384, 512, 0, 3, True, []),
                                    (131072, 512, 512, 1, False, list(range(0, 131072, 1024)))]:
        assert lg.count_pairs(N, wl, wr, d, causal, g) == lg_oracle.count_pairs_closed(N, wl, wr, d, causal, g)


def test_etc_count_pairs(lib):
    for L, G, r in [(6, 2, 1), (4, 3, 0), (4096, 256, 84), (100, 7, 200)]:
        assert lg.etc_count_pairs(L, G, r) == lg_oracle.etc_count_pairs(L, G, r)
        assert lg.etc_count_pairs(L, G, r) == int(lg_oracle.etc_mask(L, G, r).sum()) or L > 1000


def _i32(*xs):
    return (ctypes.c_int32 * len(xs))(*xs)


def call_longnet(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=FAKE, dt=lg.LG_BF16, B=1, H=2, N=256, D=64, n=2,
             w=_i32(64, 256), r=_i32(1, 6), causal=0, scale=0.0, ws=FAKE, wsb=1 << 30, stream=None)
    a.update(over)
    return lib.lg_longnet_attn_fwd(a["q"], a["k"], a["v"], a["out"], a["lse"], a["dt"], a["B"], a["H"], a["N"],
                                   a["D"], a["n"], ctypes.cast(a["w"], ctypes.c_void_p) if a["w"] else None,
                                   ctypes.cast(a["r"], ctypes.c_void_p) if a["r"] else None, a["causal"],
                                   a["scale"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("over,expect", [
    (dict(q=None), lg.LG_ERR_INVALID_ARG),
    (dict(lse=FAKE + 2), lg.LG_ERR_INVALID_ARG),
    (dict(N=0), lg.LG_ERR_INVALID_ARG),
    (dict(causal=3), lg.LG_ERR_INVALID_ARG),
    (dict(n=0), lg.LG_ERR_INVALID_ARG),
    (dict(w=None), lg.LG_ERR_INVALID_ARG),
    (dict(w=_i32(64, 0)), lg.LG_ERR_INVALID_ARG),
    (dict(r=_i32(0, 1)), lg.LG_ERR_INVALID_ARG),
    (dict(n=17, w=_i32(*([64] * 17)), r=_i32(*([1] * 17))), lg.LG_ERR_UNSUPPORTED),
    (dict(dt=lg.LG_F32), lg.LG_ERR_UNSUPPORTED),
    (dict(D=96), lg.LG_ERR_UNSUPPORTED),
    (dict(ws=None), lg.LG_ERR_WORKSPACE),
    (dict(wsb=1024), lg.LG_ERR_WORKSPACE),
])
def test_longnet_argument_errors_return_before_launch(lib, over, expect):
    assert call_longnet(lib, **over) == expect


def test_longnet_workspace_and_counts(lib):
    ws_, rs_ = _i32(2048, 4096, 8192, 16384, 32768), _i32(1, 2, 4, 6, 12)
    size = lib.lg_longnet_attn_fwd_workspace_size(1, 12, 32768, 64, 5, ctypes.cast(ws_, ctypes.c_void_p),
                                                  ctypes.cast(rs_, ctypes.c_void_p), lg.LG_BF16)
    # at least one bf16 output and fp32 LSE per pattern kept in strided layout (r divides w, r <= 8)
    assert size >= 3 * 12 * 32768 * (64 * 2 + 4) and size % 256 == 0
    assert lib.lg_longnet_attn_fwd_workspace_size(1, 12, 32768, 64, 5, ctypes.cast(ws_, ctypes.c_void_p),
                                                  ctypes.cast(rs_, ctypes.c_void_p), lg.LG_F32) == 0
    rng = np.random.default_rng(5)
    for _ in range(60):
        N = int(rng.integers(1, 400)); k = int(rng.integers(1, 5))
        ws = [int(x) for x in rng.integers(1, 300, size=k)]; rs = [int(x) for x in rng.integers(1, 14, size=k)]
        causal = bool(rng.integers(0, 2)); h = int(rng.integers(0, 20))
        assert lg.longnet_count_pairs(N, ws, rs, causal, h) == lg_oracle.longnet_count_pairs(N, ws, rs, causal, h)
    for h in range(12):
        assert lg.longnet_count_pairs(32768, list(ws_), list(rs_), True, h) == \
            lg_oracle.longnet_count_pairs(32768, list(ws_), list(rs_), True, h)
    with pytest.raises(ValueError):
        lg.longnet_count_pairs(100, [0], [1], False, 0)


def call_etc_struct(lib, **over):
    a = dict(t=[FAKE] * 10, rel=FAKE, V=8, codes=[FAKE, None, FAKE, None], dt=lg.LG_BF16, B=1, H=2, L=300, G=4,
             D=64, r=8, scale=0.0, ws=FAKE, wsb=1 << 30, stream=None)
    a.update(over)
    return lib.lg_etc_struct_attn_fwd(*a["t"], a["rel"], a["V"], *a["codes"], a["dt"], a["B"], a["H"], a["L"],
                                      a["G"], a["D"], a["r"], a["scale"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("over,expect", [
    (dict(t=[None] + [FAKE] * 9), lg.LG_ERR_INVALID_ARG),
    (dict(t=[FAKE] * 7 + [FAKE + 8] + [FAKE] * 2), lg.LG_ERR_INVALID_ARG),
    (dict(t=[FAKE] * 9 + [FAKE + 2]), lg.LG_ERR_INVALID_ARG),
    (dict(G=0), lg.LG_ERR_INVALID_ARG),
    (dict(r=-1), lg.LG_ERR_INVALID_ARG),
    (dict(rel=None), lg.LG_ERR_INVALID_ARG),          # labels without vectors
    (dict(V=0), lg.LG_ERR_INVALID_ARG),               # vectors without labels
    (dict(V=65), lg.LG_ERR_UNSUPPORTED),
    (dict(dt=lg.LG_F32), lg.LG_ERR_UNSUPPORTED),
    (dict(D=32), lg.LG_ERR_UNSUPPORTED),
    (dict(ws=None), lg.LG_ERR_WORKSPACE),
    (dict(wsb=4096), lg.LG_ERR_WORKSPACE),
])
def test_etc_struct_argument_errors_return_before_launch(lib, over, expect):
    assert call_etc_struct(lib, **over) == expect


def test_etc_struct_workspace_size(lib):
    f = lib.lg_etc_struct_attn_fwd_workspace_size
    base = f(2, 12, 4096, 256, 64, 84, 0, lg.LG_BF16)
    # one 16 KB code block per (query tile, key tile) visited: per instance 2 global query tiles x
    # (2 + 32) key tiles and 32 long query tiles x (3 band + 2 global) key tiles
    assert base >= 256 + 2 * (2 * 34 + 32 * 5) * 16384
    # q . a^K is formed inside the attention kernel (tensor memory), so labels add no workspace
    assert f(2, 12, 4096, 256, 64, 84, 32, lg.LG_BF16) == base
    assert f(2, 12, 4096, 256, 64, 84, 0, lg.LG_F32) == 0 and f(2, 12, 4096, 0, 64, 84, 0, lg.LG_BF16) == 0


def test_count_pairs_rejects_bad_lists(lib):
    with pytest.raises(ValueError):
        lg.count_pairs(10, 1, 1, 1, False, [3, 3])
    with pytest.raises(ValueError):
        lg.count_pairs(10, 1, 1, 1, False, [11])


def test_host_entry_rejects_bad_arguments(lib):
    """lg_attn_fwd_host checks its arguments before queueing anything (no GPU needed)."""
    dil = (ctypes.c_int32 * 2)(1, 1)

    def call(**over):
        a = dict(ptrs=[FAKE] * 10, dt=lg.LG_BF16, B=1, H=2, N=256, D=64, wl=8, wr=8, dil=dil, causal=0,
                 gidx=None, ng=0, scale=0.0, ws=FAKE, wsb=1 << 30, groups=2)
        a.update(over)
        return lib.lg_attn_fwd_host(*a["ptrs"], a["dt"], a["B"], a["H"], a["N"], a["D"], a["wl"], a["wr"],
                                    a["dil"], a["causal"], a["gidx"], a["ng"], a["scale"], a["ws"], a["wsb"],
                                    a["groups"], None)

    assert call(ptrs=[FAKE] * 9 + [None]) == lg.LG_ERR_INVALID_ARG
    assert call(groups=0) == lg.LG_ERR_INVALID_ARG
    assert call(N=0) == lg.LG_ERR_INVALID_ARG
    assert call(dil=(ctypes.c_int32 * 2)(1, 0)) == lg.LG_ERR_INVALID_ARG
    assert call(wsb=64) == lg.LG_ERR_WORKSPACE
    assert call(ws=None) == lg.LG_ERR_WORKSPACE
    # Checks of the whole problem come before the first copy is queued (the
    # FAKE pointers would fault any copy): a bf16 dilation beyond the limit on
    # the last head, with the heads split over two groups; D unsupported by the
    # tensor cores; a misaligned staging buffer; a missing global list.
    assert call(dil=(ctypes.c_int32 * 2)(1, 9), groups=2) == lg.LG_ERR_UNSUPPORTED
    assert call(D=96, groups=2) == lg.LG_ERR_UNSUPPORTED
    assert call(ptrs=[FAKE] * 6 + [FAKE + 8] + [FAKE] * 3) == lg.LG_ERR_INVALID_ARG
    assert call(ng=4, gidx=None, groups=2) == lg.LG_ERR_INVALID_ARG
    assert call(causal=3) == lg.LG_ERR_INVALID_ARG


def test_debug_timeout_switch_checks_its_argument(lib):
    assert lib.lg_debug_timeout_test(2, 0) == lg.LG_ERR_INVALID_ARG
    assert lib.lg_debug_timeout_test(0, 0) == lg.LG_OK


def test_binding_checks_tensors_before_the_library(lib):
    """The binding refuses tensors whose sizes the library would trust blindly."""
    import torch
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        lg.attn_fwd(q, q, q, 4, 4)                  # host tensors on the device entry point
    k_bad = torch.zeros(1, 2, 7, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        lg.attn_fwd_host(q, k_bad, q, 4, 4)         # k shorter than q
    v_bad = torch.zeros(1, 2, 8, 64, dtype=torch.float32)
    with pytest.raises(ValueError):
        lg.attn_fwd_host(q, q, v_bad, 4, 4)         # v of another dtype
    with pytest.raises(ValueError):
        lg.etc_attn_fwd(q, q, q, q, q, q, 2)        # host tensors on the device entry point
