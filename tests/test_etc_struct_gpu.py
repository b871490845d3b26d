"""ETC attention with relation labels and per-instance masks: the CUDA path
against the CPU oracle (needs a GB300).

Small cases compare every element (random labels and blocked edges, the
page's long-document recipe, rows whose every edge is blocked, two global
tiles, radius 0 and radius beyond L, D 64 and 128, an explicit scale); the
ETC-base shape with the recipe's structure compares sampled long rows and
every global row.  Tolerances as for the other bf16 outputs: max |dO| <=
2e-2, mean |dO| <= 2e-3, |dLSE| <= 1e-3.  A label outside the vocabulary is
reported through lg_query_status and the next call is clean.
"""
import numpy as np
import pytest
import torch

from oracle import lg_oracle
from sparse_long_sequence_window_gb300 import workloads
from sparse_long_sequence_window_gb300.workloads import Workload
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


def E(name, B, H, L, G, D, r, seed=400):
    return Workload(name, "bf16", B, H, L, D, etc_G=G, radius=r, seed=seed)


def random_codes(w, V, p_block, seed):
    rng = np.random.default_rng(seed)

    def c(*shape):
        lab = rng.integers(0, V, size=shape).astype(np.uint8)
        return lab | ((rng.random(shape) < p_block).astype(np.uint8) << 7)
    B, L, G, r = w.B, w.N, w.etc_G, w.radius
    return {"code_l2l": c(B, L, 2 * r + 1), "code_l2g": c(B, L, G), "code_g2l": c(B, G, L), "code_g2g": c(B, G, G)}


def run_case(lg, w, codes, rel, rows=None, scale=None, key_ramp=None):
    inp = workloads.make_inputs(w)
    if key_ramp is not None:
        # long key n times 1 + key_ramp * n / L, global key i times 1 + key_ramp * i / G (both
        # sides get the same keys): the row maximum keeps growing along the key tiles
        for n, cnt in (("k", w.N), ("k_g", w.etc_G)):
            ramp = 1.0 + key_ramp * torch.arange(cnt, dtype=torch.float32) / cnt
            inp[n] = (inp[n].float() * ramp[None, None, :, None]).to(inp[n].dtype)
    dev = torch.device("cuda")
    t = {n: inp[n].to(dev) for n in ("q", "k", "v", "q_g", "k_g", "v_g")}
    cd = {n: (None if c is None else torch.from_numpy(np.ascontiguousarray(c)).to(dev)) for n, c in codes.items()}
    rel_d = None if rel is None else rel.to(dev)
    out_l, out_g, lse_l, lse_g = lg.etc_struct_attn_fwd(t["q"], t["k"], t["v"], t["q_g"], t["k_g"], t["v_g"],
                                                        w.radius, rel_d, **cd, scale=scale)
    torch.cuda.synchronize()
    st = lg.query_status(lg.etc_struct_attn_fwd.last_workspace)
    assert st == 0, lg.status_string(st)
    a = [pu.to_np32(inp[n]) for n in ("q", "k", "v", "q_g", "k_g", "v_g")]
    reln = None if rel is None else rel.float().numpy()
    if rows is None:
        ref = lg_oracle.etc_struct_attn_fwd(*a, w.radius, reln, *codes.values(), scale=scale)
        pu.compare(w.name + " long", "bf16", out_l.cpu(), lse_l.cpu(), ref[0], ref[2])
    else:
        ref = lg_oracle.etc_struct_attn_fwd_rows(*a, w.radius, rows, reln, *codes.values(), scale=scale)
        pu.compare(w.name + " long rows", "bf16", out_l.cpu()[:, :, rows], lse_l.cpu()[:, :, rows], ref[0], ref[2])
    pu.compare(w.name + " global", "bf16", out_g.cpu(), lse_g.cpu(), ref[1], ref[3])
    return out_l, out_g, lse_l, lse_g


def rel_for(w, V, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.standard_normal((w.H, V, w.D), dtype=np.float32)).to(torch.bfloat16)


NONE = {"code_l2l": None, "code_l2g": None, "code_g2l": None, "code_g2g": None}

CASES = [
    (E("random labels D64 ragged", 2, 3, 300, 5, 64, 7), 8, 0.2),
    (E("random labels D128", 1, 2, 450, 40, 128, 30), 20, 0.1),
    (E("two global tiles", 1, 2, 200, 130, 64, 12), 5, 0.3),
    (E("radius 0", 1, 2, 260, 3, 64, 0), 4, 0.1),
    (E("radius beyond L", 1, 2, 150, 4, 64, 400), 6, 0.2),
    (E("64 labels", 1, 2, 333, 9, 64, 20), 64, 0.25),
    (E("40 labels D128 two global tiles", 1, 2, 260, 140, 128, 9), 40, 0.25),
    (E("single token", 1, 1, 1, 1, 64, 3), 2, 0.0),
    # rows of l2g, g2l and g2g codes that are multiples of 16 bytes (packed 16 at a time)
    (E("16-byte code rows", 2, 2, 512, 32, 64, 20), 8, 0.2),
]


@pytest.mark.parametrize("w,V,p_block", CASES, ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_etc_struct_small(cuda_lib, w, V, p_block):
    run_case(cuda_lib, w, random_codes(w, V, p_block, w.seed + 1), rel_for(w, V, w.seed + 2))


def test_etc_struct_masks_only(cuda_lib):
    """No relative term (rel_k NULL): the masks alone; and no codes at all is plain ETC."""
    w = E("masks only", 2, 2, 400, 6, 64, 16)
    run_case(cuda_lib, w, random_codes(w, 1, 0.3, 5), None)
    run_case(cuda_lib, w, dict(NONE), None)


def test_etc_struct_fully_blocked_rows(cuda_lib):
    """Rows whose every edge is blocked keep their unblocked weights and an LSE lower by C."""
    w = E("fully blocked rows", 1, 2, 260, 4, 64, 10)
    codes = random_codes(w, 6, 0.2, 7)
    for c in ("code_l2l", "code_l2g"):
        codes[c][0, [0, 5, 130, 259]] |= 128
    for c in ("code_g2l", "code_g2g"):
        codes[c][0, [1, 3]] |= 128
    run_case(cuda_lib, w, codes, rel_for(w, 6, 8))


def test_etc_struct_recipe_small(cuda_lib):
    """The page's long-document recipe (sentences, summary tokens, documents, hard g2l) at L = 700."""
    w = E("recipe small", 2, 3, 700, 24, 64, 16, seed=41)
    st = workloads.make_etc_structure(w)
    codes = {n: st[n] for n in NONE}
    run_case(cuda_lib, w, codes, st["rel_k"])
    run_case(cuda_lib, w, codes, st["rel_k"], scale=0.21)


def test_etc_struct_base_full_size_sampled(cuda_lib):
    """ETC-base shape (B2 H12 L4096 G256 D64 r84) with the recipe's structure: sampled long rows
    (document and sentence edges, both ends) and every global row."""
    w = workloads.PRESETS["etc_struct"]
    st = workloads.make_etc_structure(w)
    codes = {n: st[n] for n in NONE}
    rng = np.random.default_rng(23)
    rows = sorted(set([0, 1, 83, 84, 85, 127, 128, 2047, 2048, 4010, 4095] + rng.integers(0, w.N, 24).tolist()))
    run_case(cuda_lib, w, codes, st["rel_k"], rows=rows)


# The packing kernel reads a code row byte by byte, or 16 bytes at once where the row's
# length is a multiple of 16 (G = 32 here): a label past the vocabulary is reported on
# either path.
@pytest.mark.parametrize("L,G,name,at", [(200, 4, "code_l2g", (0, 17, 2)), (256, 32, "code_l2g", (0, 17, 18)),
                                          (256, 32, "code_g2l", (0, 3, 40))])
def test_etc_struct_bad_label_is_reported(cuda_lib, L, G, name, at):
    lg = cuda_lib
    w = E("bad label", 1, 2, L, G, 64, 8)
    codes = random_codes(w, 4, 0.1, 9)
    codes[name][at] = 4 | 128     # label 4 with a vocabulary of 4
    inp = workloads.make_inputs(w)
    t = {n: inp[n].cuda() for n in ("q", "k", "v", "q_g", "k_g", "v_g")}
    cd = {n: torch.from_numpy(c).cuda() for n, c in codes.items()}
    rel = rel_for(w, 4, 10).cuda()
    ws = torch.empty(lg.etc_struct_attn_fwd_workspace_size(1, 2, L, G, 64, 8, 4), dtype=torch.uint8, device="cuda")
    lg.etc_struct_attn_fwd(t["q"], t["k"], t["v"], t["q_g"], t["k_g"], t["v_g"], w.radius, rel, **cd, workspace=ws)
    assert lg.query_status(ws) == lg.LG_ERR_INVALID_ARG
    codes[name][at] = 3
    cd[name] = torch.from_numpy(codes[name]).cuda()
    lg.etc_struct_attn_fwd(t["q"], t["k"], t["v"], t["q_g"], t["k_g"], t["v_g"], w.radius, rel, **cd, workspace=ws)
    assert lg.query_status(ws) == 0


def test_etc_struct_running_max_rescales(cuda_lib):
    """Keys growing 30-fold along both key sequences, labels and blocked edges at random: the
    running maximum passes the rescale threshold on most key tiles, so O is rescaled in TMEM
    (a path N(0, 1) inputs rarely take), in long and global rows, at D 64 and 128."""
    for w, V, p_block in ((E("rising keys D64", 1, 2, 520, 150, 64, 60, seed=470), 12, 0.2),
                          (E("rising keys D128", 1, 2, 400, 40, 128, 90, seed=471), 9, 0.1)):
        codes = random_codes(w, V, p_block, seed=w.seed + 1)
        run_case(cuda_lib, w, codes, rel_for(w, V, w.seed + 2), key_ramp=30.0)
