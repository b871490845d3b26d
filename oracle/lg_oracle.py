"""fp64 CPU oracle for window + dilation + global sparse self-attention
(forward; and its backward, the next row after the forward).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check in
``__graft_entry__.smoke`` and the CPU-baseline leg of ``bench.py`` may import
this module.  The library's product path never calls it, and this module
shares no code with the CUDA path: it materialises the attention mask from
the method's definition and runs a plain masked softmax in float64.

Sources (each function names the passage it follows):

* "Longformer: The Long-Document Transformer" (arXiv 2004.05150), commentary
  page, section 3.4 "Detailed, sentence-based technical breakdown":
  - "Sliding Window Attention": a token attends to w/2 tokens on its left,
    w/2 on its right and itself (w + 1 keys).
  - "Dilated Sliding Window Attention": with dilation d the keys are
    i - d*w/2, ..., i - d, i, i + d, ..., i + d*w/2 (same key count, span x d).
  - "Global Attention": a global token attends to every token and every token
    attends to it; its row and column of the attention matrix are full.
  - "Separate Linear Projections for Local vs. Global Attention": positions
    outside the window get -inf before the softmax.
  - "Autoregressive Language Modeling Configuration": causal mode keeps only
    the left half of the window (the upper triangle of the band is masked).
* "ETC: Encoding Long and Structured Inputs in Transformers" (arXiv
  2004.08483), commentary page, section 3.4, "Global-Local Attention: The Core
  Sparse Mechanism": g2g, g2l and l2g are full; l2l is the band |i - j| <= r
  clamped to valid indices; g2g+g2l share one softmax and l2g+l2l share another
  ("Softmax unification").
* ETC page, "Relative Position Encoding" and the four pieces' logits of
  "Global-Local Attention": a learnable vector a^K_l per relation label and
  head is added to the key, e_ij = x_i W^Q (x_j W^K + a^K_ij)^T / sqrt(d_z) -
  (1 - M_ij) C with per-instance binary masks M and C = 10000.
* "LONGNET: Scaling Transformers to 1,000,000,000 Tokens" (arXiv 2307.02486),
  commentary page, section 3.4, "Standard Self-Attention and Sparse Attention"
  (a binary mask S sends disallowed logits to -inf), "Dilated Attention: Core
  Mechanism" (segments of w, every r-th row kept, dense attention among the
  kept rows), "Multi-Head Dilated Attention: Offset Mechanism" (head j starts
  at offset j mod r) and "Mixture of Dilated Attentions" (outputs computed
  over parts of the key set, weighted by their softmax denominators, equal
  one joint softmax over the union of the keys).

Readings taken where the pages are silent or ambiguous (window counted in
steps of the dilation; stride-style dilation; keys outside [0, N) dropped; a
global key inside the band counted once; causal limits only the band; natural
log LSE of the scaled logits) are stated on each function.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
hand-derived key sets from the passages above, closed forms, a library
softmax-attention routine, and invariants of the definition.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# Mask predicates
# --------------------------------------------------------------------------

def band_mask(N: int, w_left: int, w_right: int, dilation: int, causal: bool) -> np.ndarray:
    """Boolean [N, N] matrix: key j lies in the (dilated, optionally causal) window of query i.

    Longformer page, "Sliding Window Attention" and "Dilated Sliding Window
    Attention": query i sees the keys i + d*t for integer steps t running from
    -w_left to +w_right (w_left = w_right = w/2 in the page's notation), so the
    key count stays w_left + w_right + 1 while the span grows by d.  Reading:
    w_left / w_right count steps, not positions; d is a stride (d = 1 is the
    contiguous window).  Keys outside [0, N) are dropped (ETC page: "clamped
    to valid indices").  Causal ("Autoregressive Language Modeling
    Configuration"): only the left half of the window remains, i.e. t <= 0.
    """
    if dilation < 1:
        raise ValueError("dilation must be >= 1")
    i = np.arange(N, dtype=np.int64)[:, None]
    j = np.arange(N, dtype=np.int64)[None, :]
    diff = j - i
    right = 0 if causal else w_right
    on_stride = (diff % dilation) == 0
    steps = diff // dilation  # exact wherever on_stride holds
    return on_stride & (steps >= -w_left) & (steps <= right)


def global_flags(N: int, global_idx) -> np.ndarray:
    """Boolean [N]: position p is a global token."""
    flags = np.zeros(N, dtype=bool)
    g = np.asarray(global_idx, dtype=np.int64).reshape(-1)
    if g.size:
        if g.min() < 0 or g.max() >= N:
            raise ValueError("global index out of range")
        flags[g] = True
    return flags


def allowed_mask(N: int, w_left: int, w_right: int, dilation: int, causal: bool, global_idx) -> np.ndarray:
    """Boolean [N, N] attention mask of one head.

    Longformer page, "Global Attention": a global token's row and column of the
    attention matrix are both full.  The mask is the boolean union of the band
    and those rows/columns, so a global key that also falls in the band counts
    once.  Reading: causal restricts only the band; global rows and columns
    stay full.
    """
    mask = band_mask(N, w_left, w_right, dilation, causal)
    g = global_flags(N, global_idx)
    mask |= g[:, None]
    mask |= g[None, :]
    return mask


def allowed_row(i: int, N: int, w_left: int, w_right: int, dilation: int, causal: bool, gflags: np.ndarray) -> np.ndarray:
    """Boolean [N]: row i of ``allowed_mask`` evaluated from the same predicate.

    Used for sampled-row checks at sizes where the N x N mask does not fit.
    """
    j = np.arange(N, dtype=np.int64)
    diff = j - i
    right = 0 if causal else w_right
    inband = ((diff % dilation) == 0) & (diff // dilation >= -w_left) & (diff // dilation <= right)
    if gflags[i]:
        return np.ones(N, dtype=bool)
    return inband | gflags


# --------------------------------------------------------------------------
# Masked softmax attention (one head)
# --------------------------------------------------------------------------

def masked_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: np.ndarray, scale: float):
    """O, LSE and the probability matrix P of softmax(scale * q k^T masked) v, in float64.

    LongNet page, "Standard Self-Attention and Sparse Attention": logits where
    the mask is 0 are sent to -inf before the softmax, so they get weight 0.
    LSE (a reading; no page fixes it) is the natural log of the sum of
    exp(scale * q.k) over the allowed keys of each row.
    q: [n_q, D]; k, v: [n_k, D]; mask: [n_q, n_k] bool.  Every row must allow
    at least one key.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if not mask.any(axis=1).all():
        raise ValueError("a row allows no key")
    logits = scale * (q @ k.T)
    logits = np.where(mask, logits, -np.inf)
    row_max = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - row_max)          # masked entries become exactly 0
    denom = e.sum(axis=1, keepdims=True)
    probs = e / denom
    out = probs @ v
    lse = (row_max + np.log(denom))[:, 0]
    return out, lse, probs


def default_scale(D: int, scale) -> float:
    """1/sqrt(D) unless a positive scale is given (the pages' 1/sqrt(d_k))."""
    if scale is None or scale <= 0:
        return 1.0 / np.sqrt(D)
    return float(scale)


# --------------------------------------------------------------------------
# Longformer-style call: [B, H, N, D]
# --------------------------------------------------------------------------

def attn_fwd(q, k, v, w_left, w_right, dilation, causal, global_idx, scale=None):
    """Dense-mask oracle.  q, k, v: [B, H, N, D]; dilation: H ints.

    Materialises ``allowed_mask`` for each head and applies
    ``masked_attention``.  Returns O [B, H, N, D] and LSE [B, H, N] (float64).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, D = q.shape
    s = default_scale(D, scale)
    out = np.empty((B, H, N, D), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    for h in range(H):
        mask = allowed_mask(N, w_left, w_right, int(dilation[h]), bool(causal), global_idx)
        for b in range(B):
            out[b, h], lse[b, h], _ = masked_attention(q[b, h], k[b, h], v[b, h], mask, s)
    return out, lse


def attn_fwd_gproj(q, k, v, q_glob, k_glob, v_glob, w_left, w_right, dilation, causal, global_idx, scale=None):
    """Longformer attention with separate projections for global attention.

    Longformer page, "Separate Linear Projections for Local vs. Global
    Attention": local attention is softmax(Q_s K_s^T / sqrt(d_k) + mask_local)
    V_s, global attention is softmax(Q_g K_g^T / sqrt(d_k)) V_g with no mask,
    "applied to the designated global tokens".  Reading (the page does not say
    which projection a local row uses for the global columns): a global row i
    takes the global formula over every token, q_glob[i] against k_glob, with
    v_glob; every other row takes the local formula over its allowed keys
    (band plus global columns) with q, k, v.  With q_glob = q, k_glob = k,
    v_glob = v this is ``attn_fwd``.  All tensors [B, H, N, D]; returns
    O [B, H, N, D], LSE [B, H, N].
    """
    out, lse = attn_fwd(q, k, v, w_left, w_right, dilation, causal, global_idx, scale=scale)
    B, H, N, D = np.asarray(q).shape
    s = default_scale(D, scale)
    g = sorted(set(int(x) for x in np.asarray(global_idx).reshape(-1)))
    for b in range(B):
        for h in range(H):
            for i in g:
                o, l, _ = masked_attention(np.asarray(q_glob[b, h, i], np.float64)[None, :], k_glob[b, h], v_glob[b, h],
                                           np.ones((1, N), dtype=bool), s)
                out[b, h, i], lse[b, h, i] = o[0], l[0]
    return out, lse


def attn_fwd_rows(q, k, v, w_left, w_right, dilation, causal, global_idx, rows, scale=None):
    """Sampled-row oracle.  Same definition as ``attn_fwd`` for the listed rows only.

    For each (b, h) and each row i in ``rows`` the mask row is evaluated with
    ``allowed_row`` over all N keys; the allowed keys are then softmaxed.
    Returns O [B, H, len(rows), D] and LSE [B, H, len(rows)].
    """
    B, H, N, D = q.shape
    s = default_scale(D, scale)
    rows = np.asarray(rows, dtype=np.int64)
    gflags = global_flags(N, global_idx)
    out = np.empty((B, H, rows.size, D), dtype=np.float64)
    lse = np.empty((B, H, rows.size), dtype=np.float64)
    for h in range(H):
        d = int(dilation[h])
        for r, i in enumerate(rows):
            keys = np.nonzero(allowed_row(int(i), N, w_left, w_right, d, bool(causal), gflags))[0]
            for b in range(B):
                qi = np.asarray(q[b, h, i], dtype=np.float64)[None, :]
                kk = np.asarray(k[b, h, keys], dtype=np.float64)
                vv = np.asarray(v[b, h, keys], dtype=np.float64)
                o, l, _ = masked_attention(qi, kk, vv, np.ones((1, keys.size), dtype=bool), s)
                out[b, h, r] = o[0]
                lse[b, h, r] = l[0]
    return out, lse


# --------------------------------------------------------------------------
# ETC global-local call
# --------------------------------------------------------------------------

def etc_mask(L: int, G: int, radius: int) -> np.ndarray:
    """Boolean [(G+L), (G+L)] mask over the concatenation (global tokens first, then long).

    ETC page, "Global-Local Attention": the g2g, g2l and l2g blocks are full;
    the l2l block allows |i - j| <= r, clamped to valid indices.  The
    per-instance masks M are all ones (no structure given), and no relative
    position term is added.
    """
    n = G + L
    mask = np.zeros((n, n), dtype=bool)
    mask[:G, :] = True          # g2g and g2l
    mask[G:, :G] = True         # l2g
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    mask[G:, G:] = np.abs(i - j) <= radius   # l2l
    return mask


def etc_attn_fwd(q_l, k_l, v_l, q_g, k_g, v_g, radius, scale=None):
    """ETC oracle.  Long tensors [B, H, L, D], global tensors [B, H, G, D].

    "Softmax unification": a global query takes one softmax over the
    concatenation of its g2g and g2l logits; a long query takes one softmax
    over its l2g and l2l logits.  Implemented as one masked softmax over the
    concatenated token list [global; long] with ``etc_mask``.
    Returns (out_l, out_g, lse_l, lse_g), float64.
    """
    q_l = np.asarray(q_l, dtype=np.float64)
    B, H, L, D = q_l.shape
    G = np.asarray(q_g).shape[2]
    s = default_scale(D, scale)
    mask = etc_mask(L, G, radius)
    out_l = np.empty((B, H, L, D)); out_g = np.empty((B, H, G, D))
    lse_l = np.empty((B, H, L)); lse_g = np.empty((B, H, G))
    for b in range(B):
        for h in range(H):
            qq = np.concatenate([np.asarray(q_g[b, h], np.float64), q_l[b, h]], axis=0)
            kk = np.concatenate([np.asarray(k_g[b, h], np.float64), np.asarray(k_l[b, h], np.float64)], axis=0)
            vv = np.concatenate([np.asarray(v_g[b, h], np.float64), np.asarray(v_l[b, h], np.float64)], axis=0)
            o, l, _ = masked_attention(qq, kk, vv, mask, s)
            out_g[b, h], out_l[b, h] = o[:G], o[G:]
            lse_g[b, h], lse_l[b, h] = l[:G], l[G:]
    return out_l, out_g, lse_l, lse_g


def etc_attn_fwd_rows(q_l, k_l, v_l, q_g, k_g, v_g, radius, long_rows, scale=None):
    """Sampled long rows of ``etc_attn_fwd`` (l2g + l2l in one softmax); global rows are all computed.

    Returns (out_l_rows [B, H, R, D], out_g [B, H, G, D], lse_l_rows, lse_g).
    """
    B, H, L, D = q_l.shape
    G = q_g.shape[2]
    s = default_scale(D, scale)
    long_rows = np.asarray(long_rows, dtype=np.int64)
    out_l = np.empty((B, H, long_rows.size, D)); lse_l = np.empty((B, H, long_rows.size))
    out_g = np.empty((B, H, G, D)); lse_g = np.empty((B, H, G))
    for b in range(B):
        for h in range(H):
            kk = np.concatenate([np.asarray(k_g[b, h], np.float64), np.asarray(k_l[b, h], np.float64)], axis=0)
            vv = np.concatenate([np.asarray(v_g[b, h], np.float64), np.asarray(v_l[b, h], np.float64)], axis=0)
            o, l, _ = masked_attention(np.asarray(q_g[b, h], np.float64), kk, vv, np.ones((G, G + L), bool), s)
            out_g[b, h], lse_g[b, h] = o, l
            j = np.arange(L)
            for r, i in enumerate(long_rows):
                row_mask = np.concatenate([np.ones(G, bool), np.abs(j - i) <= radius])
                o, l, _ = masked_attention(np.asarray(q_l[b, h, i], np.float64)[None, :], kk, vv, row_mask[None, :], s)
                out_l[b, h, r], lse_l[b, h, r] = o[0], l[0]
    return out_l, out_g, lse_l, lse_g


# --------------------------------------------------------------------------
# ETC structured attention: relative-position labels and per-instance masks
# --------------------------------------------------------------------------

ETC_MASK_C = 10000.0   # ETC page, "Global-Local Attention": C = 10000


def etc_dense_codes(L, G, radius, code_l2l=None, code_l2g=None, code_g2l=None, code_g2g=None):
    """One instance's per-pair codes over the concatenation [global; long], uint8 [G+L, G+L].

    A code byte holds the relative-position label of the edge i -> j in bits
    0..6 and 1 - M_ij (1: blocked by the instance mask) in bit 7.  The four
    pieces come as code_g2g [G, G], code_g2l [G, L], code_l2g [L, G] and
    code_l2l [L, 2 radius + 1] (entry [i, t + radius] for the long key j = i + t);
    a piece given as None has code 0 on every edge (label 0, allowed).  Edges
    outside the l2l band keep code 0 here; they are not part of any softmax.
    """
    n = G + L
    codes = np.zeros((n, n), dtype=np.uint8)
    if code_g2g is not None:
        codes[:G, :G] = np.asarray(code_g2g, dtype=np.uint8)
    if code_g2l is not None:
        codes[:G, G:] = np.asarray(code_g2l, dtype=np.uint8)
    if code_l2g is not None:
        codes[G:, :G] = np.asarray(code_l2g, dtype=np.uint8)
    if code_l2l is not None:
        c = np.asarray(code_l2l, dtype=np.uint8)
        for t in range(-radius, radius + 1):
            i = np.arange(max(0, -t), min(L, L - t))
            codes[G + i, G + i + t] = c[i, t + radius]
    return codes


def _etc_struct_row_block(qq, kk, vv, member, codes, rel_k_h, s):
    """Softmax rows of e_ij = s q_i (k_j + a_label)^T - C (1 - M_ij) over the member keys."""
    logits = s * (qq @ kk.T)
    lab = (codes & 0x7F).astype(np.int64)
    if rel_k_h is not None:
        qa = qq @ np.asarray(rel_k_h, np.float64).T              # [rows, V]: q_i . a_l for every label
        if lab.size and lab[member].max(initial=0) >= qa.shape[1]:
            raise ValueError("a label is outside the relative-position vocabulary")
        logits = logits + s * np.take_along_axis(qa, np.minimum(lab, qa.shape[1] - 1), axis=1)
    logits = logits - ETC_MASK_C * ((codes >> 7) & 1)
    logits = np.where(member, logits, -np.inf)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    den = e.sum(axis=1, keepdims=True)
    return (e / den) @ vv, (m + np.log(den))[:, 0]


def etc_struct_attn_fwd(q_l, k_l, v_l, q_g, k_g, v_g, radius, rel_k=None, code_l2l=None, code_l2g=None,
                        code_g2l=None, code_g2g=None, scale=None):
    """ETC global-local attention with relative-position labels and per-instance masks.

    ETC page, "Relative Position Encoding" (label l_ij per edge, one learnable
    vector a^K_l per label and head) and "Global-Local Attention" (the four
    pieces' logits e_ij = x_i W^Q (x_j W^K + a^K_ij)^T / sqrt(d_z) - (1 - M_ij) C
    with C = 10000, l2l only for |i - j| <= r clamped to valid indices, and one
    softmax over g2g + g2l for a global query and one over l2g + l2l for a long
    query).  Here q_i = x_i W^Q etc. are the inputs, s the scale (1/sqrt(D) by
    default), and e_ij = s q_i . (k_j + a_l) - C blocked_ij.  rel_k: [H, V, D]
    (None: no relative term); codes per instance: code_l2l [B, L, 2r+1],
    code_l2g [B, L, G], code_g2l [B, G, L], code_g2g [B, G, G] (see
    ``etc_dense_codes``; None: all 0).  Returns (out_l, out_g, lse_l, lse_g), float64.
    """
    q_l = np.asarray(q_l, dtype=np.float64)
    B, H, L, D = q_l.shape
    G = np.asarray(q_g).shape[2]
    s = default_scale(D, scale)
    member = etc_mask(L, G, radius)
    out_l = np.empty((B, H, L, D)); out_g = np.empty((B, H, G, D))
    lse_l = np.empty((B, H, L)); lse_g = np.empty((B, H, G))
    pick = lambda c, b: None if c is None else np.asarray(c)[b]
    for b in range(B):
        codes = etc_dense_codes(L, G, radius, pick(code_l2l, b), pick(code_l2g, b), pick(code_g2l, b),
                                pick(code_g2g, b))
        for h in range(H):
            qq = np.concatenate([np.asarray(q_g[b, h], np.float64), q_l[b, h]], axis=0)
            kk = np.concatenate([np.asarray(k_g[b, h], np.float64), np.asarray(k_l[b, h], np.float64)], axis=0)
            vv = np.concatenate([np.asarray(v_g[b, h], np.float64), np.asarray(v_l[b, h], np.float64)], axis=0)
            o, l = _etc_struct_row_block(qq, kk, vv, member, codes, None if rel_k is None else rel_k[h], s)
            out_g[b, h], out_l[b, h] = o[:G], o[G:]
            lse_g[b, h], lse_l[b, h] = l[:G], l[G:]
    return out_l, out_g, lse_l, lse_g


def etc_struct_attn_fwd_rows(q_l, k_l, v_l, q_g, k_g, v_g, radius, long_rows, rel_k=None, code_l2l=None,
                             code_l2g=None, code_g2l=None, code_g2g=None, scale=None):
    """``etc_struct_attn_fwd`` at sampled long rows (every global row is computed).

    A long row i takes the G global keys (codes code_l2g[b, i]) and the long
    keys j in [i - r, i + r] inside [0, L) (codes code_l2l[b, i, j - i + r]).
    Returns (out_l_rows [B, H, R, D], out_g [B, H, G, D], lse_l_rows, lse_g).
    """
    q_l = np.asarray(q_l, dtype=np.float64)
    B, H, L, D = q_l.shape
    G = np.asarray(q_g).shape[2]
    s = default_scale(D, scale)
    long_rows = np.asarray(long_rows, dtype=np.int64)
    out_l = np.empty((B, H, long_rows.size, D)); lse_l = np.empty((B, H, long_rows.size))
    out_g = np.empty((B, H, G, D)); lse_g = np.empty((B, H, G))
    for b in range(B):
        gcodes = np.zeros((G, G + L), dtype=np.uint8)
        if code_g2g is not None:
            gcodes[:, :G] = np.asarray(code_g2g)[b]
        if code_g2l is not None:
            gcodes[:, G:] = np.asarray(code_g2l)[b]
        for h in range(H):
            a_h = None if rel_k is None else rel_k[h]
            kk = np.concatenate([np.asarray(k_g[b, h], np.float64), np.asarray(k_l[b, h], np.float64)], axis=0)
            vv = np.concatenate([np.asarray(v_g[b, h], np.float64), np.asarray(v_l[b, h], np.float64)], axis=0)
            o, l = _etc_struct_row_block(np.asarray(q_g[b, h], np.float64), kk, vv, np.ones((G, G + L), bool),
                                         gcodes, a_h, s)
            out_g[b, h], lse_g[b, h] = o, l
            for x, i in enumerate(long_rows):
                lo, hi = max(0, i - radius), min(L - 1, i + radius)
                keys = np.concatenate([np.arange(G), G + np.arange(lo, hi + 1)])
                rc = np.zeros(keys.size, dtype=np.uint8)
                if code_l2g is not None:
                    rc[:G] = np.asarray(code_l2g)[b, i]
                if code_l2l is not None:
                    rc[G:] = np.asarray(code_l2l)[b, i, lo - i + radius: hi - i + radius + 1]
                o, l = _etc_struct_row_block(q_l[b, h, i][None, :], kk[keys], vv[keys], np.ones((1, keys.size), bool),
                                             rc[None, :], a_h, s)
                out_l[b, h, x], lse_l[b, h, x] = o[0], l[0]
    return out_l, out_g, lse_l, lse_g


# --------------------------------------------------------------------------
# LongNet dilated attention
# --------------------------------------------------------------------------

def longnet_rows(N: int, w: int, r: int, s: int, seg: int) -> np.ndarray:
    """Positions kept by one dilation pattern (w, r) with offset s in segment `seg`.

    LONGNET page, "Dilated Attention: Core Mechanism" and "Multi-Head Dilated
    Attention: Offset Mechanism": segment i covers [i w, (i + 1) w); the
    sparsified rows are i w + s, i w + s + r, i w + s + 2 r, ... (w / r of
    them), clipped to the sequence.
    """
    a = seg * w
    return np.arange(a + s, min(a + w, N), r, dtype=np.int64)


def longnet_pattern(q, k, v, w, r, s, causal, scale):
    """One pattern (w, r, offset s) on one head: O, LSE of the kept rows (zeros / -inf elsewhere).

    Dense softmax attention among the sparsified rows of each segment (the
    page's gather, dense attention, scatter); causal: a kept query sees the
    kept keys at or before its own position.
    """
    N, D = np.asarray(q).shape
    out = np.zeros((N, D), dtype=np.float64)
    lse = np.full(N, -np.inf, dtype=np.float64)
    for seg in range((N + w - 1) // w):
        rows = longnet_rows(N, w, r, s, seg)
        if rows.size == 0:
            continue
        mask = np.ones((rows.size, rows.size), dtype=bool)
        if causal:
            mask = rows[None, :] <= rows[:, None]
        o, l, _ = masked_attention(np.asarray(q)[rows], np.asarray(k)[rows], np.asarray(v)[rows], mask, scale)
        out[rows], lse[rows] = o, l
    return out, lse


def longnet_attn_fwd(q, k, v, seg_w, seg_r, causal=False, scale=None):
    """LongNet mixture of dilated attentions.  q, k, v [B, H, N, D]; patterns (seg_w[i], seg_r[i]).

    LONGNET page, "Mixture of Dilated Attentions": O = sum_i alpha_i O_i with
    alpha_i = s_i / sum_j s_j, s_i the softmax denominator of pattern i for
    the row (0 where the pattern does not keep the row).  Head h uses offset
    s = h mod r_i for pattern i ("Multi-Head Dilated Attention: Offset
    Mechanism").  In terms of each pattern's LSE_i = ln s_i: LSE = ln sum_i
    s_i and O = sum_i exp(LSE_i - LSE) O_i.  A row no pattern keeps gets O = 0
    and LSE = -inf.  Returns O [B, H, N, D], LSE [B, H, N].
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    B, H, N, D = q.shape
    sc = default_scale(D, scale)
    out = np.zeros((B, H, N, D)); lse = np.full((B, H, N), -np.inf)
    for b in range(B):
        for h in range(H):
            os_, ls_ = [], []
            for w, r in zip(seg_w, seg_r):
                o, l = longnet_pattern(q[b, h], k[b, h], v[b, h], int(w), int(r), h % int(r), causal, sc)
                os_.append(o); ls_.append(l)
            out[b, h], lse[b, h] = _longnet_mix(np.stack(os_), np.stack(ls_))
    return out, lse


def _longnet_mix(os_, ls_):
    """Mix per-pattern outputs os_ [k, n, D] with their LSE ls_ [k, n] (-inf: not kept) by softmax denominators."""
    m = ls_.max(axis=0)
    keep = np.isfinite(m)
    wts = np.where(np.isfinite(ls_), np.exp(ls_ - np.where(keep, m, 0.0)[None, :]), 0.0)
    tot = wts.sum(axis=0)
    lse = np.where(keep, m + np.log(np.where(keep, tot, 1.0)), -np.inf)
    out = np.where(keep[:, None], (wts[:, :, None] * os_).sum(axis=0) / np.where(keep, tot, 1.0)[:, None], 0.0)
    return out, lse


def longnet_attn_fwd_rows(q, k, v, seg_w, seg_r, causal, rows, scale=None):
    """``longnet_attn_fwd`` at the given query rows only, one row at a time.

    Row i of head h under pattern (w, r): if the pattern keeps i (i in
    ``longnet_rows`` of its segment i // w with offset h mod r), its keys are
    the kept rows of that segment (those at or before i when causal).
    Returns O [B, H, len(rows), D], LSE [B, H, len(rows)].
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    B, H, N, D = q.shape
    sc = default_scale(D, scale)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((B, H, rows.size, D)); lse = np.full((B, H, rows.size), -np.inf)
    for b in range(B):
        for h in range(H):
            os_ = np.zeros((len(seg_w), rows.size, D)); ls_ = np.full((len(seg_w), rows.size), -np.inf)
            for pi, (w, r) in enumerate(zip(seg_w, seg_r)):
                w, r = int(w), int(r)
                for x, i in enumerate(rows):
                    kept = longnet_rows(N, w, r, h % r, int(i) // w)
                    if not (kept == i).any():
                        continue
                    keys = kept[kept <= i] if causal else kept
                    o, l, _ = masked_attention(q[b, h, i][None, :], k[b, h, keys], v[b, h, keys],
                                               np.ones((1, keys.size), dtype=bool), sc)
                    os_[pi, x], ls_[pi, x] = o[0], l[0]
            out[b, h], lse[b, h] = _longnet_mix(os_, ls_)
    return out, lse


def longnet_count_pairs(N, seg_w, seg_r, causal, h):
    """Query-key pairs head h computes, summed over the patterns (a key kept by two patterns counts twice)."""
    total = 0
    for w, r in zip(seg_w, seg_r):
        for seg in range((N + w - 1) // w):
            n = longnet_rows(N, int(w), int(r), h % int(r), seg).size
            total += n * (n + 1) // 2 if causal else n * n
    return total


# --------------------------------------------------------------------------
# Pair counts (the useful-work measure: allowed query-key pairs)
# --------------------------------------------------------------------------

def count_pairs_bruteforce(N, w_left, w_right, dilation, causal, global_idx) -> int:
    """Number of allowed (i, j) pairs of one head, by summing the materialised mask."""
    return int(allowed_mask(N, w_left, w_right, dilation, causal, global_idx).sum())


def _band_row_count(i, N, w_left, right, d):
    """#{t in [-w_left, right] : 0 <= i + d*t < N}."""
    lo = max(-w_left, -(i // d))            # smallest t with i + d*t >= 0
    hi = min(right, (N - 1 - i) // d)       # largest t with i + d*t <= N-1
    return max(0, hi - lo + 1)


def _band_col_count(j, N, w_left, right, d):
    """#{t in [-w_left, right] : 0 <= j - d*t < N} (queries whose band holds key j)."""
    hi = min(right, j // d)                          # j - d*t >= 0
    lo = max(-w_left, -((N - 1 - j) // d))           # j - d*t <= N-1
    return max(0, hi - lo + 1)


def count_pairs_closed(N, w_left, w_right, dilation, causal, global_idx) -> int:
    """Closed-form allowed-pair count of one head.

    Band: sum over steps t of the number of rows whose key i + d*t stays in
    [0, N): sum_{t=-wl}^{wr'} max(0, N - d*|t|).  Globals add the union of g
    full rows and g full columns, 2gN - g^2 pairs, minus those already in the
    band (inclusion-exclusion over band rows and columns of the global set).
    """
    d = int(dilation)
    right = 0 if causal else w_right
    band = sum(max(0, N - d * abs(t)) for t in range(-w_left, right + 1))
    g = sorted(set(int(x) for x in np.asarray(global_idx).reshape(-1)))
    if not g:
        return band
    n_g = len(g)
    rows_cols = 2 * n_g * N - n_g * n_g
    in_band_rows = sum(_band_row_count(i, N, w_left, right, d) for i in g)
    in_band_cols = sum(_band_col_count(j, N, w_left, right, d) for j in g)
    garr = np.asarray(g, dtype=np.int64)
    diff = garr[None, :] - garr[:, None]
    both = int((((diff % d) == 0) & (diff // d >= -w_left) & (diff // d <= right)).sum())
    overlap = in_band_rows + in_band_cols - both
    return band + rows_cols - overlap


def etc_count_pairs(L, G, radius) -> int:
    """Allowed pairs of one ETC head: l2l band + l2g (L*G) + g2g and g2l (G*(G+L)).

    ETC page, "Global-Local Attention", complexity O(n_g(n_g + n_l) + n_l(n_g + 2r + 1)).
    """
    ll = sum(max(0, L - abs(t)) for t in range(-radius, radius + 1))
    return ll + L * G + G * (G + L)


# --------------------------------------------------------------------------
# Partial softmax statistics and their merge
# --------------------------------------------------------------------------

def partial_stats(q, k, v, mask, scale):
    """Softmax statistics of one key subset: row max m, sum l of exp(x - m), unnormalised acc.

    A row with no allowed key in the subset gets m = -inf, l = 0, acc = 0.
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    logits = np.where(mask, scale * (q @ k.T), -np.inf)
    m = logits.max(axis=1)
    safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(logits - safe[:, None])
    return m, e.sum(axis=1), e @ v


def merge_partials(ms, ls, accs):
    """Joint softmax from per-subset statistics.

    LongNet page, "Mixture of Dilated Attentions": outputs over parts of the
    key set, weighted by their softmax denominators, equal one softmax over the
    union of the keys.  With m = max_p m_p: l = sum_p e^{m_p - m} l_p,
    O = sum_p e^{m_p - m} acc_p / l, LSE = m + ln l.
    ms, ls: [P, n]; accs: [P, n, D].
    """
    ms = np.asarray(ms, np.float64); ls = np.asarray(ls, np.float64); accs = np.asarray(accs, np.float64)
    m = ms.max(axis=0)
    w = np.where(np.isfinite(ms), np.exp(ms - m[None, :]), 0.0)
    l = (w * ls).sum(axis=0)
    out = (w[:, :, None] * accs).sum(axis=0) / l[:, None]
    return out, m + np.log(l)


# --------------------------------------------------------------------------
# Backward pass (the row after the forward: gradients of the same function)
# --------------------------------------------------------------------------

def masked_attention_bwd(q, k, v, mask, scale, dout, dlse=None):
    """dQ, dK, dV of one head of ``masked_attention`` for upstream gradients dO (and dLSE).

    The pages train with this attention and take gradients through it
    (Longformer page, "Autoregressive Language Modeling Configuration":
    activations recomputed in the backward pass; LongNet page, "Distributed
    Training Algorithm": the gradients with respect to the keys and values),
    so the backward pass is the derivative of the forward definition above,
    written out by the chain rule in float64:
      P = softmax over the allowed keys of scale * q k^T,  O = P v,
      dV = P^T dO,   dP = dO v^T,
      dS_ij = P_ij (dP_ij - sum_j' P_ij' dP_ij') + P_ij dLSE_i,
      dQ = scale * dS k,   dK = scale * dS^T q.
    Disallowed pairs have P = 0 and so contribute nothing.  q, dout: [n_q, D];
    k, v: [n_k, D]; mask: [n_q, n_k] bool; dlse: [n_q] or None.
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    dout = np.asarray(dout, np.float64)
    _, _, p = masked_attention(q, k, v, mask, scale)
    dv = p.T @ dout
    dp = dout @ v.T
    delta = (p * dp).sum(axis=1, keepdims=True)
    ds = p * (dp - delta)
    if dlse is not None:
        ds = ds + p * np.asarray(dlse, np.float64)[:, None]
    return scale * (ds @ k), scale * (ds.T @ q), dv


def attn_bwd(q, k, v, dout, w_left, w_right, dilation, causal, global_idx, scale=None, dlse=None):
    """Dense-mask backward of ``attn_fwd``: dQ, dK, dV [B, H, N, D] (float64).

    Same mask as the forward (``allowed_mask`` per head); dout: [B, H, N, D];
    dlse: [B, H, N] or None.
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    dout = np.asarray(dout, np.float64)
    B, H, N, D = q.shape
    s = default_scale(D, scale)
    dq = np.empty_like(q); dk = np.empty_like(k); dv = np.empty_like(v)
    for h in range(H):
        mask = allowed_mask(N, w_left, w_right, int(dilation[h]), bool(causal), global_idx)
        for b in range(B):
            dl = None if dlse is None else np.asarray(dlse, np.float64)[b, h]
            dq[b, h], dk[b, h], dv[b, h] = masked_attention_bwd(q[b, h], k[b, h], v[b, h], mask, s,
                                                                dout[b, h], dl)
    return dq, dk, dv


def allowed_col(j: int, N: int, w_left: int, w_right: int, dilation: int, causal: bool, gflags: np.ndarray) -> np.ndarray:
    """Boolean [N]: the rows i with allowed(i, j), column j of ``allowed_mask``.

    Same predicate as ``allowed_row``, read down a column: key j is in row i's
    band when j - i = d*t with -w_left <= t <= w_right (0 if causal); a global
    row allows every key, and a global key is allowed by every row.
    """
    i = np.arange(N, dtype=np.int64)
    diff = j - i
    right = 0 if causal else w_right
    inband = ((diff % dilation) == 0) & (diff // dilation >= -w_left) & (diff // dilation <= right)
    if gflags[j]:
        return np.ones(N, dtype=bool)
    return inband | gflags


def _row_stats(q, k, v, dout, i, keys, s):
    """Row i over its allowed keys: P_i (over `keys`), Delta_i = <dO_i, O_i>."""
    qi = np.asarray(q[i], np.float64)[None, :]
    kk = np.asarray(k[keys], np.float64)
    vv = np.asarray(v[keys], np.float64)
    o, _, p = masked_attention(qi, kk, vv, np.ones((1, keys.size), dtype=bool), s)
    return p[0], float(np.dot(np.asarray(dout[i], np.float64), o[0]))


def attn_bwd_rows(q, k, v, dout, w_left, w_right, dilation, causal, global_idx, rows, scale=None):
    """dQ of the listed query rows, [B, H, len(rows), D]: the backward of ``attn_fwd_rows``.

    dQ_i needs row i alone: its allowed keys, P_i over them, Delta_i =
    <dO_i, O_i>, dS_ij = P_ij (<dO_i, v_j> - Delta_i), dQ_i = s sum_j dS_ij k_j
    (the chain rule of ``masked_attention_bwd`` restricted to one row).
    """
    B, H, N, D = q.shape
    s = default_scale(D, scale)
    rows = np.asarray(rows, dtype=np.int64)
    gflags = global_flags(N, global_idx)
    out = np.empty((B, H, rows.size, D), dtype=np.float64)
    for h in range(H):
        d = int(dilation[h])
        for r, i in enumerate(rows):
            keys = np.nonzero(allowed_row(int(i), N, w_left, w_right, d, bool(causal), gflags))[0]
            for b in range(B):
                p, delta = _row_stats(q[b, h], k[b, h], v[b, h], dout[b, h], int(i), keys, s)
                dp = np.asarray(v[b, h, keys], np.float64) @ np.asarray(dout[b, h, i], np.float64)
                ds = p * (dp - delta)
                out[b, h, r] = s * (ds @ np.asarray(k[b, h, keys], np.float64))
    return out


def attn_bwd_cols(q, k, v, dout, w_left, w_right, dilation, causal, global_idx, cols, scale=None, heads=None):
    """dK and dV of the listed keys, [B, H, len(cols), D] each (heads not in `heads` left 0).

    Key j collects from every row i that allows it (``allowed_col``):
    dV_j = sum_i P_ij dO_i and dK_j = s sum_i dS_ij q_i, where P_i and Delta_i
    come from row i's own allowed keys.  Rows are evaluated once per (b, h).
    """
    B, H, N, D = q.shape
    s = default_scale(D, scale)
    cols = np.asarray(cols, dtype=np.int64)
    gflags = global_flags(N, global_idx)
    dk = np.zeros((B, H, cols.size, D), dtype=np.float64)
    dv = np.zeros((B, H, cols.size, D), dtype=np.float64)
    for h in (range(H) if heads is None else heads):
        d = int(dilation[h])
        for b in range(B):
            cache = {}
            for c, j in enumerate(cols):
                rows = np.nonzero(allowed_col(int(j), N, w_left, w_right, d, bool(causal), gflags))[0]
                for i in rows:
                    i = int(i)
                    if i not in cache:
                        keys = np.nonzero(allowed_row(i, N, w_left, w_right, d, bool(causal), gflags))[0]
                        p, delta = _row_stats(q[b, h], k[b, h], v[b, h], dout[b, h], i, keys, s)
                        cache[i] = (keys, p, delta)
                    keys, p, delta = cache[i]
                    pij = p[np.searchsorted(keys, j)]
                    dij = pij * (float(np.dot(np.asarray(dout[b, h, i], np.float64), np.asarray(v[b, h, j], np.float64))) - delta)
                    dv[b, h, c] += pij * np.asarray(dout[b, h, i], np.float64)
                    dk[b, h, c] += s * dij * np.asarray(q[b, h, i], np.float64)
    return dk, dv


def etc_attn_bwd(q_l, k_l, v_l, q_g, k_g, v_g, radius, dout_l, dout_g, scale=None):
    """Dense-mask backward of ``etc_attn_fwd``: gradients of the long and global inputs.

    The [global; long] sequence with the ``etc_mask`` of the forward; returns
    (dq_l, dk_l, dv_l, dq_g, dk_g, dv_g), each shaped like its input.
    """
    q_l = np.asarray(q_l, np.float64); k_l = np.asarray(k_l, np.float64); v_l = np.asarray(v_l, np.float64)
    q_g = np.asarray(q_g, np.float64); k_g = np.asarray(k_g, np.float64); v_g = np.asarray(v_g, np.float64)
    B, H, L, D = q_l.shape
    G = q_g.shape[2]
    s = default_scale(D, scale)
    mask = etc_mask(L, G, radius)
    out = [np.empty_like(x) for x in (q_l, k_l, v_l, q_g, k_g, v_g)]
    for b in range(B):
        for h in range(H):
            q = np.concatenate([q_g[b, h], q_l[b, h]]); k = np.concatenate([k_g[b, h], k_l[b, h]])
            v = np.concatenate([v_g[b, h], v_l[b, h]])
            do = np.concatenate([np.asarray(dout_g, np.float64)[b, h], np.asarray(dout_l, np.float64)[b, h]])
            dq, dk, dv = masked_attention_bwd(q, k, v, mask, s, do)
            for i, (x, part) in enumerate(((dq, 1), (dk, 1), (dv, 1), (dq, 0), (dk, 0), (dv, 0))):
                out[i][b, h] = x[G:] if part else x[:G]
    return tuple(out)
