"""Plant plausible mistakes in copies of the CPU oracle and check that a pin catches each.

The mutants live only in this test, on the CPU.  Each replaces one function of
a fresh copy of the oracle module with a subtly wrong version (a dropped term,
a swapped sign or index, a transposed operand); the pins must reject it.
"""
import importlib.util
import os

import numpy as np
import pytest

from tests import oracle_pins

ORACLE_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "lg_oracle.py")


def fresh_oracle():
    spec = importlib.util.spec_from_file_location("lg_oracle_mutant", ORACLE_PATH)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def mut_swap_sides(O):
    orig = O.band_mask
    O.band_mask = lambda N, wl, wr, d, causal: orig(N, wr, wl, d, causal)
    orig_row = O.allowed_row
    O.allowed_row = lambda i, N, wl, wr, d, causal, g: orig_row(i, N, wr, wl, d, causal, g)


def mut_ignore_dilation(O):
    orig = O.band_mask
    O.band_mask = lambda N, wl, wr, d, causal: orig(N, wl, wr, 1, causal)


def mut_span_not_steps(O):
    # window counted in positions instead of dilation steps
    orig = O.band_mask
    O.band_mask = lambda N, wl, wr, d, causal: orig(N, wl // d, wr // d, d, causal)


def mut_causal_keeps_right(O):
    orig = O.band_mask
    O.band_mask = lambda N, wl, wr, d, causal: orig(N, wl, wr, d, False)


def mut_no_global_columns(O):
    def allowed_mask(N, wl, wr, d, causal, g):
        m = O.band_mask(N, wl, wr, d, causal)
        m |= O.global_flags(N, g)[:, None]
        return m
    O.allowed_mask = allowed_mask


def mut_no_scale(O):
    orig = O.masked_attention
    O.masked_attention = lambda q, k, v, mask, scale: orig(q, k, v, mask, 1.0)


def mut_transposed_logits(O):
    def masked_attention(q, k, v, mask, scale):
        q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
        logits = scale * (q @ k.T)
        if logits.shape[0] == logits.shape[1]:
            logits = logits.T
        logits = np.where(mask, logits, -np.inf)
        mx = logits.max(axis=1, keepdims=True)
        e = np.exp(logits - mx); den = e.sum(axis=1, keepdims=True)
        return (e / den) @ v, (mx + np.log(den))[:, 0], e / den
    O.masked_attention = masked_attention


def mut_lse_log2(O):
    orig = O.masked_attention
    def masked_attention(q, k, v, mask, scale):
        o, l, p = orig(q, k, v, mask, scale)
        return o, l / np.log(2.0), p
    O.masked_attention = masked_attention


def mut_etc_radius_off_by_one(O):
    orig = O.etc_mask
    O.etc_mask = lambda L, G, r: orig(L, G, r + 1)


def mut_etc_no_l2g(O):
    orig = O.etc_mask
    def etc_mask(L, G, r):
        m = orig(L, G, r); m[G:, :G] = False
        return m
    O.etc_mask = etc_mask


def mut_closed_form_no_overlap(O):
    orig = O.count_pairs_closed
    def count(N, wl, wr, d, causal, g):
        g = list(g)
        if not g:
            return orig(N, wl, wr, d, causal, g)
        band = orig(N, wl, wr, d, causal, [])
        return band + 2 * len(g) * N - len(g) ** 2
    O.count_pairs_closed = count


def mut_merge_no_rescale(O):
    def merge_partials(ms, ls, accs):
        ls = np.asarray(ls); accs = np.asarray(accs); ms = np.asarray(ms)
        l = ls.sum(axis=0)
        return accs.sum(axis=0) / l[:, None], ms.max(axis=0) + np.log(l)
    O.merge_partials = merge_partials


def _bwd_mutant(O, variant):
    def masked_attention_bwd(q, k, v, mask, scale, dout, dlse=None):
        q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
        _, _, p = O.masked_attention(q, k, v, mask, scale)
        dp = dout @ v.T
        delta = 0.0 if variant == "no_delta" else (p * dp).sum(axis=1, keepdims=True)
        ds = p * (dp - delta)
        if dlse is not None:
            ds = ds + p * np.asarray(dlse)[:, None]
        dv = p @ dout if variant == "dv_untransposed" else p.T @ dout
        sc = 1.0 if variant == "no_scale" else scale
        dk = sc * (ds @ q) if variant == "dk_untransposed" else sc * (ds.T @ q)
        return sc * (ds @ k), dk, dv
    O.masked_attention_bwd = masked_attention_bwd


def mut_bwd_no_delta(O):
    _bwd_mutant(O, "no_delta")


def mut_bwd_no_scale(O):
    _bwd_mutant(O, "no_scale")


def mut_bwd_dk_untransposed(O):
    _bwd_mutant(O, "dk_untransposed")


def mut_bwd_dv_untransposed(O):
    _bwd_mutant(O, "dv_untransposed")


def mut_gproj_local_keys(O):
    # global rows scored against the local keys instead of the global projection's
    orig = O.attn_fwd_gproj
    O.attn_fwd_gproj = lambda q, k, v, qg, kg, vg, *a, **kw: orig(q, k, v, qg, k, vg, *a, **kw)


def mut_bwd_cols_drop_global_rows(O):
    # sampled-key backward that forgets the global rows attending every key
    orig_col = O.allowed_col
    O.allowed_col = lambda j, N, wl, wr, d, causal, g: orig_col(j, N, wl, wr, d, causal, g) & ~g | (
        g if g[j] else False)


def mut_longnet_no_offset(O):
    # every head starts its sparsification at offset 0
    orig = O.longnet_rows
    O.longnet_rows = lambda N, w, r, s, seg: orig(N, w, r, 0, seg)


def mut_longnet_plain_average(O):
    # patterns averaged with equal weights instead of their softmax denominators
    orig = O.longnet_pattern

    def pattern(q, k, v, w, r, s, causal, scale):
        o, l = orig(q, k, v, w, r, s, causal, scale)
        return o, np.where(np.isfinite(l), 0.0, l)
    O.longnet_pattern = pattern


def mut_etc_struct_bias_sign(O):
    # relative term subtracted instead of added
    orig = O._etc_struct_row_block
    O._etc_struct_row_block = lambda qq, kk, vv, member, codes, a, s: orig(
        qq, kk, vv, member, codes, None if a is None else -np.asarray(a), s)


def mut_etc_struct_bias_unscaled(O):
    # relative term q . a_l without the 1/sqrt(d) of the content term
    orig = O._etc_struct_row_block
    O._etc_struct_row_block = lambda qq, kk, vv, member, codes, a, s: orig(
        qq, kk, vv, member, codes, None if a is None else np.asarray(a) / s, s)


def mut_etc_struct_mask_excludes(O):
    # a blocked edge dropped from the softmax (-inf) instead of -C
    orig = O._etc_struct_row_block

    def block(qq, kk, vv, member, codes, a, s):
        return orig(qq, kk, vv, member & ((codes >> 7) == 0), codes & 0x7F, a, s)
    O._etc_struct_row_block = block


def mut_etc_struct_l2l_reversed(O):
    # the l2l code of key j = i + t read at offset -t
    orig = O.etc_dense_codes
    O.etc_dense_codes = lambda L, G, r, c_ll=None, c_lg=None, c_gl=None, c_gg=None: orig(
        L, G, r, None if c_ll is None else np.asarray(c_ll)[:, ::-1], c_lg, c_gl, c_gg)


def mut_etc_struct_g2l_as_l2g(O):
    # the global rows' long-key codes taken from the transposed long rows' global-key codes
    orig = O.etc_dense_codes
    O.etc_dense_codes = lambda L, G, r, c_ll=None, c_lg=None, c_gl=None, c_gg=None: orig(
        L, G, r, c_ll, c_lg, None if c_lg is None else np.asarray(c_lg).T, c_gg)


MUTANTS = [mut_swap_sides, mut_ignore_dilation, mut_span_not_steps, mut_causal_keeps_right,
           mut_no_global_columns, mut_no_scale, mut_transposed_logits, mut_lse_log2,
           mut_etc_radius_off_by_one, mut_etc_no_l2g, mut_closed_form_no_overlap, mut_merge_no_rescale,
           mut_bwd_no_delta, mut_bwd_no_scale, mut_bwd_dk_untransposed, mut_bwd_dv_untransposed,
           mut_gproj_local_keys, mut_bwd_cols_drop_global_rows, mut_longnet_no_offset,
           mut_longnet_plain_average, mut_etc_struct_bias_sign, mut_etc_struct_bias_unscaled,
           mut_etc_struct_mask_excludes, mut_etc_struct_l2l_reversed, mut_etc_struct_g2l_as_l2g]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda f: f.__name__)
def test_mutant_is_caught(mutant):
    O = fresh_oracle()
    mutant(O)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(O)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"{mutant.__name__} passed every pin"
