"""Pin checks for the CPU oracle.

Each ``pin_*`` takes an oracle module and raises AssertionError when the
oracle disagrees with something fixed outside it: hand-derived key sets and
counts (tests/golden), closed forms, a library softmax-attention routine, or
an invariant of the definition.  ``test_oracle_pins.py`` runs them on the real
oracle; ``test_oracle_mutants.py`` runs them on copies with a planted mistake
and expects at least one pin to fail for each.
"""
from __future__ import annotations

import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


def _parse_list(s):
    return [] if s == "-" else [int(x) for x in s.split(",")]


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- golden

def pin_golden_windows(O):
    for case, N, wl, wr, d, causal, glist, row, keys in _golden_lines("window_keys.txt"):
        N, wl, wr, d, row = int(N), int(wl), int(wr), int(d), int(row)
        g = _parse_list(glist)
        mask = O.allowed_mask(N, wl, wr, d, bool(int(causal)), g)
        got = np.nonzero(mask[row])[0].tolist()
        assert got == _parse_list(keys), (case, got, keys)
        gflags = O.global_flags(N, g)
        got_row = np.nonzero(O.allowed_row(row, N, wl, wr, d, bool(int(causal)), gflags))[0].tolist()
        assert got_row == _parse_list(keys), (case, "row", got_row, keys)


def pin_golden_etc(O):
    for case, L, G, r, query, keys in _golden_lines("etc_keys.txt"):
        L, G, r = int(L), int(G), int(r)
        mask = O.etc_mask(L, G, r)
        qi = int(query[1:]) + (0 if query[0] == "g" else G)
        names = [f"g{j}" for j in range(G)] + [f"l{j}" for j in range(L)]
        got = [names[j] for j in np.nonzero(mask[qi])[0]]
        assert got == keys.split(","), (case, got, keys)


def pin_golden_counts(O):
    for parts in _golden_lines("pair_counts.txt"):
        if parts[0] == "etc":
            L, G, r, count = map(int, parts[1:])
            assert O.etc_count_pairs(L, G, r) == count, parts
            assert int(O.etc_mask(L, G, r).sum()) == count, parts
            continue
        case, N, wl, wr, d, causal, glist, count = parts
        args = (int(N), int(wl), int(wr), int(d), bool(int(causal)), _parse_list(glist))
        assert O.count_pairs_bruteforce(*args) == int(count), (case, "brute")
        assert O.count_pairs_closed(*args) == int(count), (case, "closed")


# ---------------------------------------------------------------- closed forms

def pin_closed_form_counts(O, trials=120, seed=11):
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        N = int(rng.integers(1, 70))
        wl = int(rng.integers(0, 12)); wr = int(rng.integers(0, 12))
        d = int(rng.integers(1, 6)); causal = bool(rng.integers(0, 2))
        ng = int(rng.integers(0, min(N, 6) + 1))
        g = sorted(rng.choice(N, size=ng, replace=False).tolist()) if ng else []
        a = O.count_pairs_bruteforce(N, wl, wr, d, causal, g)
        b = O.count_pairs_closed(N, wl, wr, d, causal, g)
        assert a == b, (N, wl, wr, d, causal, g, a, b)
    # interior rows keep exactly w_left + w_right + 1 keys (w + 1 in the page's notation)
    mask = O.band_mask(200, 7, 5, 3, False)
    assert (mask[60:140].sum(axis=1) == 13).all()


def pin_linear_in_n(O):
    """Longformer page: cost O(n*w) + O(n*g) -> the count is affine in N once N exceeds the span."""
    g = list(range(5))
    c = [O.count_pairs_closed(n, 16, 16, 2, False, g) for n in (400, 800, 1200, 1600)]
    assert c[1] - c[0] == c[2] - c[1] == c[3] - c[2]
    per_row = (c[1] - c[0]) / 400
    assert per_row == 33 + 2 * len(g)   # w + 1 band keys plus a global row and column per global


# ---------------------------------------------------------------- library routine

def _sdpa64(q, k, v, scale):
    qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(x)) for x in (q, k, v))
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale).numpy()


def pin_full_attention(O, seed=3):
    """A window that covers the sequence (d = 1, non-causal) is full softmax attention."""
    rng = np.random.default_rng(seed)
    B, H, N, D = 2, 3, 37, 16
    q, k, v = _rand(rng, B, H, N, D), _rand(rng, B, H, N, D), _rand(rng, B, H, N, D)
    for scale in (None, 0.37):
        s = 1 / np.sqrt(D) if scale is None else scale
        out, lse = O.attn_fwd(q, k, v, N - 1, N - 1, [1] * H, False, [], scale)
        ref = _sdpa64(q, k, v, s)
        assert np.abs(out - ref).max() < 1e-12
        logits = torch.from_numpy(s * np.einsum("bhid,bhjd->bhij", q, k))
        assert np.abs(lse - torch.logsumexp(logits, dim=-1).numpy()).max() < 1e-12
    # ETC with a radius that covers the long input is full attention over [global; long]
    G, L = 5, 23
    ql, kl, vl = _rand(rng, 1, 2, L, D), _rand(rng, 1, 2, L, D), _rand(rng, 1, 2, L, D)
    qg, kg, vg = _rand(rng, 1, 2, G, D), _rand(rng, 1, 2, G, D), _rand(rng, 1, 2, G, D)
    ol, og, _, _ = O.etc_attn_fwd(ql, kl, vl, qg, kg, vg, L, None)
    cat = lambda a, b: np.concatenate([a, b], axis=2)
    ref = _sdpa64(cat(qg, ql), cat(kg, kl), cat(vg, vl), 1 / np.sqrt(D))
    assert np.abs(og - ref[:, :, :G]).max() < 1e-12
    assert np.abs(ol - ref[:, :, G:]).max() < 1e-12


def pin_global_rows_are_full_rows(O, seed=4):
    """Longformer page, "Global Attention": a global query attends to every token."""
    rng = np.random.default_rng(seed)
    B, H, N, D = 1, 2, 50, 8
    q, k, v = _rand(rng, B, H, N, D), _rand(rng, B, H, N, D), _rand(rng, B, H, N, D)
    g = [0, 17, 49]
    out, lse = O.attn_fwd(q, k, v, 3, 2, [1, 3], True, g)
    ref = _sdpa64(q, k, v, 1 / np.sqrt(D))
    assert np.abs(out[:, :, g] - ref[:, :, g]).max() < 1e-12


# ---------------------------------------------------------------- invariants

def pin_rows_sum_to_one(O, seed=5):
    rng = np.random.default_rng(seed)
    N, D = 41, 8
    q, k, v = _rand(rng, N, D), _rand(rng, N, D), _rand(rng, N, D)
    mask = O.allowed_mask(N, 4, 2, 3, False, [7, 40])
    _, _, probs = O.masked_attention(q, k, v, mask, 0.5)
    assert np.abs(probs.sum(axis=1) - 1).max() < 1e-12
    assert (probs[~mask] == 0).all()
    assert (probs[mask] > 0).all()


def pin_identity_window(O, seed=6):
    """w_left = w_right = 0 without globals: each row sees only itself -> O = V, LSE = s<q_i, k_i>."""
    rng = np.random.default_rng(seed)
    B, H, N, D = 1, 2, 19, 8
    q, k, v = _rand(rng, B, H, N, D), _rand(rng, B, H, N, D), _rand(rng, B, H, N, D)
    out, lse = O.attn_fwd(q, k, v, 0, 0, [1, 4], False, [])
    assert np.abs(out - v).max() < 1e-14
    assert np.abs(lse - np.einsum("bhnd,bhnd->bhn", q, k) / np.sqrt(D)).max() < 1e-13
    # causal first row sees only itself
    out, _ = O.attn_fwd(q, k, v, 5, 5, [1, 2], True, [])
    assert np.abs(out[:, :, 0] - v[:, :, 0]).max() < 1e-14


def pin_dilation_residues(O, seed=7):
    """A dilated head equals an undilated window applied to each residue class {c + d*t}."""
    rng = np.random.default_rng(seed)
    N, D, d = 47, 8, 3
    q, k, v = _rand(rng, 1, 1, N, D), _rand(rng, 1, 1, N, D), _rand(rng, 1, 1, N, D)
    for causal in (False, True):
        out, lse = O.attn_fwd(q, k, v, 2, 3, [d], causal, [])
        for c in range(d):
            idx = np.arange(c, N, d)
            o2, l2 = O.attn_fwd(q[:, :, idx], k[:, :, idx], v[:, :, idx], 2, 3, [1], causal, [])
            assert np.abs(out[:, :, idx] - o2).max() < 1e-13
            assert np.abs(lse[:, :, idx] - l2).max() < 1e-13


def pin_key_shift(O, seed=8):
    """Adding u to every key leaves O unchanged and shifts LSE_i by s<q_i, u>."""
    rng = np.random.default_rng(seed)
    N, D = 33, 8
    q, k, v = _rand(rng, 1, 2, N, D), _rand(rng, 1, 2, N, D), _rand(rng, 1, 2, N, D)
    u = _rand(rng, D)
    o1, l1 = O.attn_fwd(q, k, v, 3, 5, [1, 2], False, [4, 30])
    o2, l2 = O.attn_fwd(q, k + u, v, 3, 5, [1, 2], False, [4, 30])
    assert np.abs(o1 - o2).max() < 1e-12
    assert np.abs((l2 - l1) - np.einsum("bhnd,d->bhn", q, u) / np.sqrt(D)).max() < 1e-12


def pin_constant_values(O, seed=9):
    rng = np.random.default_rng(seed)
    N, D = 29, 4
    q, k = _rand(rng, 1, 1, N, D), _rand(rng, 1, 1, N, D)
    c = np.array([1.5, -2.0, 0.25, 3.0])
    v = np.broadcast_to(c, (1, 1, N, D)).copy()
    out, _ = O.attn_fwd(q, k, v, 2, 2, [2], False, [3])
    assert np.abs(out - c).max() < 1e-13


def pin_etc_permutation(O, seed=10):
    """Permuting the global tokens permutes out_g and leaves out_l unchanged (no positional term)."""
    rng = np.random.default_rng(seed)
    L, G, D = 21, 6, 8
    t = [_rand(rng, 1, 2, L, D) for _ in range(3)] + [_rand(rng, 1, 2, G, D) for _ in range(3)]
    perm = rng.permutation(G)
    a = O.etc_attn_fwd(*t, 2)
    b = O.etc_attn_fwd(*t[:3], *(x[:, :, perm] for x in t[3:]), 2)
    assert np.abs(a[0] - b[0]).max() < 1e-12
    assert np.abs(a[1][:, :, perm] - b[1]).max() < 1e-12
    assert np.abs(a[3][:, :, perm] - b[3]).max() < 1e-12


def pin_etc_rows(O, seed=12):
    """The sampled-row ETC oracle agrees with the dense one."""
    rng = np.random.default_rng(seed)
    L, G, D = 30, 4, 8
    t = [_rand(rng, 2, 1, L, D) for _ in range(3)] + [_rand(rng, 2, 1, G, D) for _ in range(3)]
    ol, og, ll, lg = O.etc_attn_fwd(*t, 3)
    rows = [0, 1, 14, 28, 29]
    rl, rg, rll, rlg = O.etc_attn_fwd_rows(*t, 3, rows)
    assert np.abs(ol[:, :, rows] - rl).max() < 1e-12 and np.abs(og - rg).max() < 1e-12
    assert np.abs(ll[:, :, rows] - rll).max() < 1e-12 and np.abs(lg - rlg).max() < 1e-12


def pin_rows_vs_dense(O, seed=13):
    rng = np.random.default_rng(seed)
    B, H, N, D = 2, 3, 45, 8
    q, k, v = _rand(rng, B, H, N, D), _rand(rng, B, H, N, D), _rand(rng, B, H, N, D)
    g = [2, 44]
    for causal in (False, True):
        out, lse = O.attn_fwd(q, k, v, 3, 4, [1, 2, 5], causal, g)
        rows = [0, 2, 3, 20, 43, 44]
        ro, rl = O.attn_fwd_rows(q, k, v, 3, 4, [1, 2, 5], causal, g, rows)
        assert np.abs(out[:, :, rows] - ro).max() < 1e-12
        assert np.abs(lse[:, :, rows] - rl).max() < 1e-12


def pin_merge(O, seed=14):
    """LongNet page: weighting partial outputs by softmax denominators equals one joint softmax."""
    rng = np.random.default_rng(seed)
    n, nk, D = 9, 40, 8
    q, k, v = _rand(rng, n, D), _rand(rng, nk, D), _rand(rng, nk, D)
    mask = rng.random((n, nk)) < 0.6
    mask[:, 0] = True
    full_o, full_l, _ = O.masked_attention(q, k, v, mask, 0.7)
    for parts in (1, 2, 3, 7):
        cuts = np.sort(rng.choice(np.arange(1, nk), size=parts - 1, replace=False)) if parts > 1 else []
        bounds = [0, *cuts, nk]
        ms, ls, accs = [], [], []
        for a, b in zip(bounds[:-1], bounds[1:]):
            sub = np.zeros_like(mask); sub[:, a:b] = mask[:, a:b]
            m, l, acc = O.partial_stats(q, k, v, sub, 0.7)
            ms.append(m); ls.append(l); accs.append(acc)
        o, lse = O.merge_partials(ms, ls, accs)
        assert np.abs(o - full_o).max() < 1e-12
        assert np.abs(lse - full_l).max() < 1e-12


# ---------------------------------------------------------------- backward

def _loss(O, q, k, v, args, dout, dlse):
    """Scalar L = sum(dO * O) + sum(dLSE * LSE); its gradients are the backward pass."""
    out, lse = O.attn_fwd(q, k, v, *args)
    return float((dout * out).sum() + (dlse * lse).sum())


def pin_bwd_finite_differences(O, seed=15):
    """Central differences of the forward oracle reproduce dQ, dK, dV (incl. a dLSE term)."""
    rng = np.random.default_rng(seed)
    B, H, N, D = 1, 2, 11, 3
    q, k, v = _rand(rng, B, H, N, D), _rand(rng, B, H, N, D), _rand(rng, B, H, N, D)
    dout, dlse = _rand(rng, B, H, N, D), _rand(rng, B, H, N)
    for args in ((2, 1, [1, 2], False, [4]), (3, 0, [2, 1], True, [])):
        dq, dk, dv = O.attn_bwd(q, k, v, dout, *args, dlse=dlse)
        eps = 1e-6
        for x, g in ((q, dq), (k, dk), (v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + eps; up = _loss(O, q, k, v, args, dout, dlse)
                x[idx] = old - eps; dn = _loss(O, q, k, v, args, dout, dlse)
                x[idx] = old
                num[idx] = (up - dn) / (2 * eps)
            assert np.abs(num - g).max() < 1e-6 * (1 + np.abs(g).max())


def pin_bwd_autograd(O, seed=16):
    """torch autograd of a masked fp64 softmax attention (library routine) gives the same gradients."""
    rng = np.random.default_rng(seed)
    B, H, N, D = 2, 2, 19, 8
    q, k, v = _rand(rng, B, H, N, D), _rand(rng, B, H, N, D), _rand(rng, B, H, N, D)
    dout, dlse = _rand(rng, B, H, N, D), _rand(rng, B, H, N)
    wl, wr, dil, causal, g = 3, 2, [1, 3], False, [0, 9]
    masks = torch.from_numpy(np.stack([O.allowed_mask(N, wl, wr, d, causal, g) for d in dil]))[None]
    qt, kt, vt = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
    s = 1 / np.sqrt(D)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=masks, scale=s)
    logits = (s * qt @ kt.transpose(-1, -2)).masked_fill(~masks, float("-inf"))
    loss = (out * torch.from_numpy(dout)).sum() + (torch.logsumexp(logits, dim=-1) * torch.from_numpy(dlse)).sum()
    loss.backward()
    dq, dk, dv = O.attn_bwd(q, k, v, dout, wl, wr, dil, causal, g, dlse=dlse)
    for mine, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        assert np.abs(mine - ref.numpy()).max() < 1e-11


def pin_bwd_invariants(O, seed=17):
    """Shifting every key leaves O unchanged, so sum_j dK_j = 0; rows of P sum to 1, so sum_j dV_j = sum_i dO_i."""
    rng = np.random.default_rng(seed)
    B, H, N, D = 2, 3, 40, 6
    q, k, v, dout = (_rand(rng, B, H, N, D) for _ in range(4))
    dq, dk, dv = O.attn_bwd(q, k, v, dout, 5, 4, [1, 2, 3], True, [7, 30])
    assert np.abs(dk.sum(axis=2)).max() < 1e-11
    assert np.abs(dv.sum(axis=2) - dout.sum(axis=2)).max() < 1e-11
    # identity window (w = 0, no globals): O = V, so dV = dO and dQ = dK = 0
    dq, dk, dv = O.attn_bwd(q, k, v, dout, 0, 0, [1, 1, 1], False, [])
    assert np.abs(dv - dout).max() < 1e-14 and np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14


def pin_etc_bwd_finite_differences(O, seed=18):
    """Central differences of the ETC forward reproduce the gradients of the long and global inputs."""
    rng = np.random.default_rng(seed)
    B, H, L, G, D, r = 1, 1, 7, 2, 3, 1
    xs = [_rand(rng, B, H, L, D) for _ in range(3)] + [_rand(rng, B, H, G, D) for _ in range(3)]
    dl, dg = _rand(rng, B, H, L, D), _rand(rng, B, H, G, D)

    def loss():
        ol, og, _, _ = O.etc_attn_fwd(*xs, r)
        return float((dl * ol).sum() + (dg * og).sum())

    grads = O.etc_attn_bwd(*xs, r, dl, dg)
    eps = 1e-6
    for x, g in zip(xs, grads):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps; up = loss()
            x[idx] = old - eps; dn = loss()
            x[idx] = old
            num[idx] = (up - dn) / (2 * eps)
        assert np.abs(num - g).max() < 1e-6 * (1 + np.abs(g).max())


def pin_bwd_rows_cols_vs_dense(O, seed=19):
    """The sampled-row dQ and sampled-key dK, dV equal the dense backward (dilation, causal, globals)."""
    rng = np.random.default_rng(seed)
    B, H, N, D = 2, 3, 41, 5
    q, k, v, dout = (_rand(rng, B, H, N, D) for _ in range(4))
    g = [0, 17, 40]
    for causal in (False, True):
        args = (4, 3, [1, 2, 5], causal, g)
        dq, dk, dv = O.attn_bwd(q, k, v, dout, *args)
        rows = [0, 1, 9, 17, 33, 40]
        assert np.abs(O.attn_bwd_rows(q, k, v, dout, *args, rows) - dq[:, :, rows]).max() < 1e-12
        cols = [0, 2, 17, 25, 39, 40]
        ck, cv = O.attn_bwd_cols(q, k, v, dout, *args, cols)
        assert np.abs(ck - dk[:, :, cols]).max() < 1e-12 and np.abs(cv - dv[:, :, cols]).max() < 1e-12


def pin_gproj(O, seed=20):
    """Separate global projections: equal projections reduce to attn_fwd; a global row is the
    full-attention row of (q_glob, k_glob, v_glob) (library SDPA); other rows ignore the global projections."""
    rng = np.random.default_rng(seed)
    B, H, N, D = 1, 2, 30, 8
    q, k, v, qg, kg, vg = (_rand(rng, B, H, N, D) for _ in range(6))
    args = (3, 2, [1, 2], False, [0, 11, 29])
    o1, l1 = O.attn_fwd_gproj(q, k, v, q, k, v, *args)
    o0, l0 = O.attn_fwd(q, k, v, *args)
    assert np.abs(o1 - o0).max() < 1e-13 and np.abs(l1 - l0).max() < 1e-13
    o2, l2 = O.attn_fwd_gproj(q, k, v, qg, kg, vg, *args)
    ref = _sdpa64(qg, kg, vg, 1 / np.sqrt(D))
    for i in (0, 11, 29):
        assert np.abs(o2[:, :, i] - ref[:, :, i]).max() < 1e-12
    rest = [i for i in range(N) if i not in (0, 11, 29)]
    assert np.abs(o2[:, :, rest] - o0[:, :, rest]).max() < 1e-13 and np.abs(l2[:, :, rest] - l0[:, :, rest]).max() < 1e-13


def pin_golden_longnet(O):
    """Hand-worked LongNet kept rows and mixtures (tests/golden/longnet.txt)."""
    for parts in _golden_lines("longnet.txt"):
        if parts[0] == "rows":
            N, w, r, head, seg = (int(x) for x in parts[1:6])
            assert O.longnet_rows(N, w, r, head % r, seg).tolist() == _parse_list(parts[6]), parts
        else:
            N = int(parts[1]); ws = _parse_list(parts[2]); rs = _parse_list(parts[3]); causal = bool(int(parts[4]))
            row, o_ref, s_ref = int(parts[5]), float(parts[6]), float(parts[7])
            z = np.zeros((1, 1, N, 1)); v = (np.arange(N, dtype=np.float64) + 1).reshape(1, 1, N, 1)
            o, l = O.longnet_attn_fwd(z, z, v, ws, rs, causal)
            assert abs(o[0, 0, row, 0] - o_ref) < 1e-12 and abs(l[0, 0, row] - np.log(s_ref)) < 1e-12, parts


def pin_longnet_reductions(O, seed=21):
    """One pattern with w >= N, r = 1 is full attention; one pattern (w, r) on head h is dense
    attention on the gathered rows of each segment (library SDPA), zero elsewhere."""
    rng = np.random.default_rng(seed)
    B, H, N, D = 1, 3, 37, 8
    q, k, v = (_rand(rng, B, H, N, D) for _ in range(3))
    s = 1 / np.sqrt(D)
    o, l = O.longnet_attn_fwd(q, k, v, [64], [1])
    assert np.abs(o - _sdpa64(q, k, v, s)).max() < 1e-12
    for w, r in ((12, 3), (16, 4), (8, 2), (10, 3), (16, 6), (5, 7)):   # r need not divide w; r > w
        o, l = O.longnet_attn_fwd(q, k, v, [w], [r])
        for h in range(H):
            covered = np.zeros(N, dtype=bool)
            for seg in range((N + w - 1) // w):
                rows = [p for p in range(seg * w + h % r, min(seg * w + w, N), r)]
                if not rows:
                    continue
                covered[rows] = True
                ref = _sdpa64(q[:, h:h + 1, rows], k[:, h:h + 1, rows], v[:, h:h + 1, rows], s)
                assert np.abs(o[:, h:h + 1, rows] - ref).max() < 1e-12
            assert np.abs(o[:, h, ~covered]).max() == 0.0 and np.isneginf(l[:, h, ~covered]).all()


def pin_longnet_rows_vs_full(O, seed=23):
    """The row-at-a-time LongNet oracle equals the whole-sequence one (several patterns, causal, r not dividing w)."""
    rng = np.random.default_rng(seed)
    B, H, N, D = 2, 5, 53, 8
    q, k, v = (_rand(rng, B, H, N, D) for _ in range(3))
    rows = [0, 1, 6, 17, 30, 31, 52]
    for ws, rs, causal in (([8, 24, 53], [1, 3, 7], False), ([10, 32], [2, 5], True), ([4, 64], [6, 4], False)):
        o, l = O.longnet_attn_fwd(q, k, v, ws, rs, causal)
        o2, l2 = O.longnet_attn_fwd_rows(q, k, v, ws, rs, causal, rows)
        assert np.abs(o2 - o[:, :, rows]).max() < 1e-13
        assert np.array_equal(np.isneginf(l2), np.isneginf(l[:, :, rows]))
        fin = np.isfinite(l2)
        assert np.abs(l2[fin] - l[:, :, rows][fin]).max() < 1e-13


def pin_longnet_counts(O):
    """Pair count of the patterns: (w/r)^2 per full segment (non-causal), against brute force."""
    assert O.longnet_count_pairs(4096, [2048, 4096], [1, 2], False, 0) == 2 * 2048 ** 2 + 2048 ** 2
    for N, ws, rs, causal, h in ((37, [8, 16], [1, 4], False, 3), (50, [10, 20], [2, 5], True, 1)):
        brute = 0
        for w, r in zip(ws, rs):
            for seg in range((N + w - 1) // w):
                n = len(range(seg * w + h % r, min(seg * w + w, N), r))
                brute += n * (n + 1) // 2 if causal else n * n
        assert O.longnet_count_pairs(N, ws, rs, causal, h) == brute


# ---------------------------------------------------------------- ETC structured attention

def pin_golden_etc_struct(O):
    """Hand-worked ETC relative labels and masks (tests/golden/etc_struct.txt)."""
    one = lambda *x: np.array(x, dtype=np.float64).reshape(1, 1, -1, 1)
    q_l, k_l, v_l = one(1, 1), one(0, 0), one(1, 3)
    q_g, k_g, v_g = one(1), one(0), one(5)
    rel = np.array([[[0.0], [np.log(2.0)]]])
    n = 0
    for case, l2l, l2g, g2l, g2g, row, o_ref, lse_a, lse_b in _golden_lines("etc_struct.txt"):
        c_l2l = np.array([[int(x) for x in r.split(",")] for r in l2l.split("/")], dtype=np.uint8)[None]
        c_l2g = np.array([[int(x)] for x in l2g.split("/")], dtype=np.uint8)[None]
        c_g2l = np.array([[int(x) for x in g2l.split(",")]], dtype=np.uint8)[None]
        c_g2g = np.array([[int(g2g)]], dtype=np.uint8)[None]
        out_l, out_g, lse_l, lse_g = O.etc_struct_attn_fwd(q_l, k_l, v_l, q_g, k_g, v_g, 1, rel, c_l2l, c_l2g,
                                                           c_g2l, c_g2g, scale=1.0)
        o, l = (out_g[0, 0, 0, 0], lse_g[0, 0, 0]) if row == "g0" else (out_l[0, 0, int(row[1]), 0],
                                                                        lse_l[0, 0, int(row[1])])
        assert abs(o - float(o_ref)) < 1e-12, (case, row, o)
        assert abs(l - (np.log(float(lse_a)) + float(lse_b))) < 1e-9, (case, row, l)
        n += 1
    assert n == 4


def _etc_inputs(rng, B=2, H=3, L=23, G=5, D=8):
    x = lambda *s: _rand(rng, *s)
    return x(B, H, L, D), x(B, H, L, D), x(B, H, L, D), x(B, H, G, D), x(B, H, G, D), x(B, H, G, D)


def _etc_codes(rng, B, L, G, r, V, p_block=0.0):
    def c(*shape):
        lab = rng.integers(0, V, size=shape).astype(np.uint8)
        return lab | ((rng.random(shape) < p_block).astype(np.uint8) << 7)
    return c(B, L, 2 * r + 1), c(B, L, G), c(B, G, L), c(B, G, G)


def pin_etc_struct_reductions(O, seed=31):
    """No relative term and no blocked edge is plain ETC; one label on every edge of a row shifts
    its logits by the same s q_i . a_l, which leaves O unchanged and adds s q_i . a_l to LSE."""
    rng = np.random.default_rng(seed)
    B, H, L, G, D, r = 2, 3, 23, 5, 8, 3
    args = _etc_inputs(rng, B, H, L, G, D)
    ref = O.etc_attn_fwd(*args, r)
    got = O.etc_struct_attn_fwd(*args, r)
    assert all(np.abs(a - b).max() < 1e-13 for a, b in zip(ref, got))
    codes = _etc_codes(rng, B, L, G, r, 4)
    got = O.etc_struct_attn_fwd(*args, r, np.zeros((H, 4, D)), *codes)
    assert all(np.abs(a - b).max() < 1e-13 for a, b in zip(ref, got))
    rel = _rand(rng, H, 4, D)
    for lab in (0, 3):
        codes = tuple(np.full_like(c, lab) for c in _etc_codes(rng, B, L, G, r, 4))
        out_l, out_g, lse_l, lse_g = O.etc_struct_attn_fwd(*args, r, rel, *codes)
        s = 1 / np.sqrt(D)
        sh_l = s * np.einsum("bhid,hd->bhi", args[0], rel[:, lab])
        sh_g = s * np.einsum("bhid,hd->bhi", args[3], rel[:, lab])
        assert np.abs(out_l - ref[0]).max() < 1e-12 and np.abs(out_g - ref[1]).max() < 1e-12
        assert np.abs(lse_l - ref[2] - sh_l).max() < 1e-12 and np.abs(lse_g - ref[3] - sh_g).max() < 1e-12


def pin_etc_struct_unexpanded_form(O, seed=32):
    """The page's unexpanded logit q_i (k_j + a_ij)^T, with a per-edge key materialised, blocked
    edges minus C and the band by -inf, through torch softmax / logsumexp, equals the oracle."""
    rng = np.random.default_rng(seed)
    B, H, L, G, D, r, V = 2, 2, 19, 4, 8, 2, 6
    args = _etc_inputs(rng, B, H, L, G, D)
    codes = _etc_codes(rng, B, L, G, r, V, p_block=0.2)
    rel = _rand(rng, H, V, D)
    s = 0.37
    out_l, out_g, lse_l, lse_g = O.etc_struct_attn_fwd(*args, r, rel, *codes, scale=s)
    n = G + L
    for b in range(B):
        dense = np.zeros((n, n), dtype=np.int64)   # codes over [global; long], written out piece by piece
        dense[:G, :G] = codes[3][b]; dense[:G, G:] = codes[2][b]; dense[G:, :G] = codes[1][b]
        inband = np.zeros((n, n), dtype=bool); inband[:G, :] = True; inband[G:, :G] = True
        for i in range(L):
            for j in range(max(0, i - r), min(L, i + r + 1)):
                dense[G + i, G + j] = codes[0][b, i, j - i + r]; inband[G + i, G + j] = True
        for h in range(H):
            q = torch.from_numpy(np.concatenate([args[3][b, h], args[0][b, h]]))
            k = torch.from_numpy(np.concatenate([args[4][b, h], args[1][b, h]]))
            v = torch.from_numpy(np.concatenate([args[5][b, h], args[2][b, h]]))
            lab = torch.from_numpy(dense & 0x7F)
            key_ij = k[None, :, :] + torch.from_numpy(rel[h])[lab]          # [n, n, D]: k_j + a_label(i, j)
            e = s * torch.einsum("id,ijd->ij", q, key_ij) - O.ETC_MASK_C * torch.from_numpy((dense >> 7) & 1)
            e = e.masked_fill(~torch.from_numpy(inband), float("-inf"))
            o = (torch.softmax(e, dim=1) @ v).numpy()
            l = torch.logsumexp(e, dim=1).numpy()
            assert np.abs(o[:G] - out_g[b, h]).max() < 1e-12 and np.abs(o[G:] - out_l[b, h]).max() < 1e-12
            assert np.abs(l[:G] - lse_g[b, h]).max() < 1e-10 and np.abs(l[G:] - lse_l[b, h]).max() < 1e-10


def pin_etc_struct_masks(O, seed=33):
    """A blocked edge (in a row that keeps an allowed key) weighs exactly nothing: the output equals
    library SDPA over the allowed edges only.  A row whose every edge is blocked keeps the weights
    it would have with none blocked (the -C is common to its logits), and its LSE is lower by C."""
    rng = np.random.default_rng(seed)
    B, H, L, G, D, r = 1, 2, 21, 4, 8, 3
    args = _etc_inputs(rng, B, H, L, G, D)
    codes = list(_etc_codes(rng, B, L, G, r, 1, p_block=0.35))
    codes[3][0, :, 0] = 0           # every global row keeps global key 0
    codes[1][0, :, 0] = 0           # every long row keeps global key 0
    out_l, out_g, lse_l, lse_g = O.etc_struct_attn_fwd(*args, r, None, *codes)
    n = G + L
    allowed = O.etc_mask(L, G, r).copy()
    blocked = (O.etc_dense_codes(L, G, r, codes[0][0], codes[1][0], codes[2][0], codes[3][0]) >> 7) == 1
    allowed &= ~blocked
    for h in range(H):
        q = np.concatenate([args[3][0, h], args[0][0, h]]); k = np.concatenate([args[4][0, h], args[1][0, h]])
        v = np.concatenate([args[5][0, h], args[2][0, h]])
        o = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
            attn_mask=torch.from_numpy(allowed)[None], scale=1 / np.sqrt(D))[0].numpy()
        assert np.abs(o[:G] - out_g[0, h]).max() < 1e-12 and np.abs(o[G:] - out_l[0, h]).max() < 1e-12
    # long row 7 and global row 1: every edge blocked
    full = [np.zeros_like(c) for c in codes]
    blk = [c.copy() for c in full]
    blk[0][0, 7, :] = 128; blk[1][0, 7, :] = 128; blk[2][0, 1, :] = 128; blk[3][0, 1, :] = 128
    a = O.etc_struct_attn_fwd(*args, r, None, *full)
    b = O.etc_struct_attn_fwd(*args, r, None, *blk)
    assert np.abs(a[0] - b[0]).max() < 1e-9 and np.abs(a[1] - b[1]).max() < 1e-9
    assert np.abs(b[2][:, :, 7] - a[2][:, :, 7] + O.ETC_MASK_C).max() < 1e-9
    assert np.abs(b[3][:, :, 1] - a[3][:, :, 1] + O.ETC_MASK_C).max() < 1e-9


def pin_etc_struct_rows_vs_full(O, seed=34):
    """The sampled-row ETC structured oracle equals the whole-instance one."""
    rng = np.random.default_rng(seed)
    B, H, L, G, D, r, V = 2, 2, 29, 6, 8, 4, 5
    args = _etc_inputs(rng, B, H, L, G, D)
    codes = _etc_codes(rng, B, L, G, r, V, p_block=0.2)
    rel = _rand(rng, H, V, D)
    full = O.etc_struct_attn_fwd(*args, r, rel, *codes)
    rows = [0, 3, 4, 17, 28]
    got = O.etc_struct_attn_fwd_rows(*args, r, rows, rel, *codes)
    assert np.abs(got[0] - full[0][:, :, rows]).max() < 1e-12 and np.abs(got[1] - full[1]).max() < 1e-12
    assert np.abs(got[2] - full[2][:, :, rows]).max() < 1e-10 and np.abs(got[3] - full[3]).max() < 1e-10


ALL_PINS = [
    pin_golden_windows, pin_golden_etc, pin_golden_counts, pin_closed_form_counts,
    pin_linear_in_n, pin_full_attention, pin_global_rows_are_full_rows, pin_rows_sum_to_one,
    pin_identity_window, pin_dilation_residues, pin_key_shift, pin_constant_values,
    pin_etc_permutation, pin_etc_rows, pin_rows_vs_dense, pin_merge,
    pin_bwd_finite_differences, pin_bwd_autograd, pin_bwd_invariants, pin_etc_bwd_finite_differences,
    pin_bwd_rows_cols_vs_dense, pin_gproj, pin_golden_longnet, pin_longnet_reductions, pin_longnet_counts,
    pin_longnet_rows_vs_full, pin_golden_etc_struct, pin_etc_struct_reductions, pin_etc_struct_unexpanded_form,
    pin_etc_struct_masks, pin_etc_struct_rows_vs_full,
]
