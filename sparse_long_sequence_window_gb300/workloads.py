"""Seeded synthetic inputs and named workload presets.

This module only draws random numbers and rounds them to the input dtype.  It
holds none of the attention arithmetic, so both the CUDA path and the
independent CPU checker can take their inputs from it.

Recipe: Q, K, V are iid N(0, 1) float32 drawn from
``numpy.random.default_rng(seed)`` in the order q, k, v with shape
[B, H, N, D] (for the ETC workload: q_l, k_l, v_l [B, H, L, D], then q_g, k_g,
v_g [B, H, G, D]).  bf16 workloads are rounded to bfloat16 with
round-to-nearest-even before either side sees them, so a comparison measures
kernel error only.  Random global positions are distinct, drawn with
``default_rng(seed + 1000)`` and sorted ascending.  The upstream gradient dO
of the backward pass (and dO_g of the ETC global outputs) is iid N(0, 1)
from ``default_rng(seed + 7919)``, rounded like the inputs.  Separate global
projections (q_glob, k_glob, v_glob) are iid N(0, 1) from
``default_rng(seed + 4243)``, in that order, rounded like the inputs.

The presets mirror the pages' workloads: a Longformer-base QA shape
(CLS + question span global), an ETC-base shape (local radius 84, a few
hundred global tokens), a character-LM shape (causal, dilated heads), a
long-sequence sweep, and the LongNet language-model mixture (12 heads of 64,
32K tokens, causal, segments 2K..32K with rates 1, 2, 4, 6, 12).  The pages evaluate on datasets that are not used here;
these synthetic tensors stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                   # "f32" or "bf16"
    B: int
    H: int
    N: int                       # sequence length (ETC: long length L)
    D: int
    w_left: int = 0
    w_right: int = 0
    dilation: Sequence[int] = ()  # per head; empty means all 1
    causal: bool = False
    global_positions: Optional[Sequence[int]] = None   # explicit positions
    n_random_global: int = 0     # draw this many distinct random positions
    etc_G: int = 0               # > 0 selects the ETC call with a separate global input
    radius: int = 0              # ETC local radius
    seed: int = 0
    seg_w: Sequence[int] = ()    # LongNet: segment lengths of the mixture's patterns
    seg_r: Sequence[int] = ()    # LongNet: their dilation rates

    @property
    def is_etc(self) -> bool:
        return self.etc_G > 0

    @property
    def is_longnet(self) -> bool:
        return len(self.seg_w) > 0

    def dilations(self):
        return list(self.dilation) if self.dilation else [1] * self.H

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The reference workloads.
PRESETS = {
    "tiny_f32": Workload("tiny_f32 B1 H2 N512 D64 w64/64 G={0}", "f32", 1, 2, 512, 64,
                         64, 64, (), False, (0,), seed=1),
    "longformer_base": Workload("longformer_base bf16 B1 H12 N4096 D64 w256/256 G=0..64", "bf16",
                                1, 12, 4096, 64, 256, 256, (), False, tuple(range(65)), seed=2),
    "etc_base": Workload("etc_base bf16 B2 H12 L4096 G256 D64 r84", "bf16", 2, 12, 4096, 64,
                         etc_G=256, radius=84, seed=3),
    "charlm_dilated": Workload("charlm_dilated bf16 B1 H8 N16384 D64 causal wl512 d=[1,1,2,2,3,3,4,4]",
                               "bf16", 1, 8, 16384, 64, 512, 0, (1, 1, 2, 2, 3, 3, 4, 4), True, (), seed=4),
    "long_8k": Workload("long_scale bf16 B1 H16 N8192 D128 w512/512 G=128 random", "bf16",
                        1, 16, 8192, 128, 512, 512, (), False, None, 128, seed=5),
    "long_32k": Workload("long_scale bf16 B1 H16 N32768 D128 w512/512 G=128 random", "bf16",
                         1, 16, 32768, 128, 512, 512, (), False, None, 128, seed=5),
    "etc_struct": Workload("etc_struct bf16 B2 H12 L4096 G256 D64 r84, 32 relation labels, 4 documents, hard g2l",
                           "bf16", 2, 12, 4096, 64, etc_G=256, radius=84, seed=7),
    "longnet_lm": Workload("longnet_lm bf16 B1 H12 N32768 D64 causal w=2K..32K r=1,2,4,6,12", "bf16",
                           1, 12, 32768, 64, causal=True, seg_w=(2048, 4096, 8192, 16384, 32768),
                           seg_r=(1, 2, 4, 6, 12), seed=6),
    "long_128k": Workload("long_scale bf16 B1 H16 N131072 D128 w512/512 G=128 random", "bf16",
                          1, 16, 131072, 128, 512, 512, (), False, None, 128, seed=5),
}


def global_positions(w: Workload) -> np.ndarray:
    """Sorted distinct int32 global positions of a (non-ETC) workload."""
    if w.global_positions is not None:
        return np.asarray(sorted(set(int(x) for x in w.global_positions)), dtype=np.int32)
    if w.n_random_global > 0:
        rng = np.random.default_rng(w.seed + 1000)
        pos = rng.choice(w.N, size=w.n_random_global, replace=False)
        return np.sort(pos).astype(np.int32)
    return np.zeros(0, dtype=np.int32)


def _round(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(x)
    if dtype == "bf16":
        return t.to(torch.bfloat16)
    return t.contiguous()


def make_inputs(w: Workload) -> dict:
    """Host tensors of the workload in its input dtype, plus global positions.

    Returns a dict with q, k, v (and q_g, k_g, v_g for ETC) as CPU torch
    tensors of dtype float32 or bfloat16, and ``global_idx`` (int32 numpy).
    """
    rng = np.random.default_rng(w.seed)
    shape = (w.B, w.H, w.N, w.D)
    out = {}
    for name in ("q", "k", "v"):
        out[name] = _round(rng.standard_normal(shape, dtype=np.float32), w.dtype)
    if w.is_etc:
        gshape = (w.B, w.H, w.etc_G, w.D)
        for name in ("q_g", "k_g", "v_g"):
            out[name] = _round(rng.standard_normal(gshape, dtype=np.float32), w.dtype)
        out["global_idx"] = np.zeros(0, dtype=np.int32)
    else:
        out["global_idx"] = global_positions(w)
    return out


def as_f64(t: torch.Tensor) -> np.ndarray:
    """The exact values of an input tensor as float64 (bf16 and f32 upcast exactly)."""
    return t.to(torch.float64).numpy()


def make_grad_out(w: Workload) -> dict:
    """The upstream gradient of the outputs for the backward pass: dout
    [B, H, N, D] (and dout_g [B, H, G, D] for ETC), iid N(0, 1) from
    default_rng(seed + 7919), in the workload's dtype."""
    rng = np.random.default_rng(w.seed + 7919)
    out = {"dout": _round(rng.standard_normal((w.B, w.H, w.N, w.D), dtype=np.float32), w.dtype)}
    if w.is_etc:
        out["dout_g"] = _round(rng.standard_normal((w.B, w.H, w.etc_G, w.D), dtype=np.float32), w.dtype)
    return out


# Relation labels of the structured ETC workload (a vocabulary of 32): the
# clipped relative distances -k..k (k = 12) within a sentence, then a few
# structural relations.
ETC_REL_K = 12
ETC_LABEL_OTHER_SENTENCE = 2 * ETC_REL_K + 1   # l2l: key in another sentence
ETC_LABEL_OWN_SUMMARY = 26                     # l2g: the summary token of the query's sentence
ETC_LABEL_OTHER_SUMMARY = 27                   # l2g: another sentence's summary token
ETC_LABEL_CLS = 28                             # edges to or from the global CLS token (global 0)
ETC_LABEL_OWN_TOKEN = 29                       # g2l: a token of the summary's own sentence
ETC_LABEL_OTHER_TOKEN = 30                     # g2l: a token of another sentence
ETC_N_LABELS = 32


def make_etc_structure(w: Workload, n_docs: int = 4, hard_g2l: bool = True) -> dict:
    """Per-instance structure for ETC attention with relation labels and masks, following the ETC
    page's recipe for long documents: the long input split into sentences, one summary token per
    sentence in the global input after a CLS token (global 0), several documents per instance.

    Sentence lengths are drawn from ``default_rng(seed + 5557)`` (uniform in [4, 2 L / (G - 1)],
    the last sentence taking the rest); sentences are dealt to ``n_docs`` documents in order.  Codes
    (uint8, label in bits 0..6, 128 = blocked):
      * l2l: clip(j - i, -k, k) + k inside a sentence, ETC_LABEL_OTHER_SENTENCE across sentences;
        blocked across documents;
      * l2g: CLS label to global 0, own / other summary label; blocked to summaries of other documents;
      * g2l: CLS label from global 0; own / other token label; with hard_g2l a summary token is
        blocked from every token outside its sentence, else only from other documents;
      * g2g: clip(j - i, -k, k) + k; blocked between summaries of different documents.
    rel_k [H, 32, D] is iid N(0, 1) from the same generator, rounded like the inputs.
    Returns numpy arrays code_l2l [B, L, 2r+1], code_l2g [B, L, G], code_g2l [B, G, L],
    code_g2g [B, G, G], rel_k, and the per-instance sentence and document ids.
    """
    B, H, L, G, D, r = w.B, w.H, w.N, w.etc_G, w.D, w.radius
    k = ETC_REL_K
    rng = np.random.default_rng(w.seed + 5557)
    n_sent = max(1, G - 1)
    c_ll = np.zeros((B, L, 2 * r + 1), np.uint8); c_lg = np.zeros((B, L, G), np.uint8)
    c_gl = np.zeros((B, G, L), np.uint8); c_gg = np.zeros((B, G, G), np.uint8)
    sent_ids = np.zeros((B, L), np.int64); doc_of_sent = np.zeros((B, n_sent), np.int64)
    for b in range(B):
        hi = max(4, 2 * L // n_sent)
        lens = rng.integers(4, hi + 1, size=n_sent)
        starts = np.minimum(np.concatenate([[0], np.cumsum(lens)[:-1]]), L)
        sent = np.searchsorted(starts, np.arange(L), side="right") - 1    # sentence of each token
        doc_s = (np.arange(n_sent) * n_docs) // n_sent                    # document of each sentence
        doc_t = doc_s[sent]
        sent_ids[b], doc_of_sent[b] = sent, doc_s
        i = np.arange(L)[:, None]; t = np.arange(-r, r + 1)[None, :]; j = i + t
        jc = np.clip(j, 0, L - 1)
        same_s = sent[i[:, 0]][:, None] == sent[jc]
        lab = np.where(same_s, np.clip(t, -k, k) + k, ETC_LABEL_OTHER_SENTENCE)
        blk = doc_t[i[:, 0]][:, None] != doc_t[jc]
        c_ll[b] = (lab | (blk.astype(np.int64) << 7)).astype(np.uint8)
        gs = np.arange(G) - 1                                             # sentence of each global (-1: CLS)
        own = sent[:, None] == gs[None, :]
        lab = np.where(own, ETC_LABEL_OWN_SUMMARY, ETC_LABEL_OTHER_SUMMARY); lab[:, 0] = ETC_LABEL_CLS
        gdoc = np.where(gs >= 0, doc_s[np.clip(gs, 0, n_sent - 1)], -1)
        blk = (gdoc[None, :] != doc_t[:, None]) & (gs[None, :] >= 0)
        c_lg[b] = (lab | (blk.astype(np.int64) << 7)).astype(np.uint8)
        lab = np.where(own.T, ETC_LABEL_OWN_TOKEN, ETC_LABEL_OTHER_TOKEN); lab[0, :] = ETC_LABEL_CLS
        blk = (~own.T if hard_g2l else (gdoc[:, None] != doc_t[None, :])) & (gs[:, None] >= 0)
        c_gl[b] = (lab | (blk.astype(np.int64) << 7)).astype(np.uint8)
        tg = np.arange(G)[None, :] - np.arange(G)[:, None]
        lab = np.clip(tg, -k, k) + k
        blk = (gdoc[:, None] != gdoc[None, :]) & (gs[:, None] >= 0) & (gs[None, :] >= 0)
        c_gg[b] = (lab | (blk.astype(np.int64) << 7)).astype(np.uint8)
    rel = _round(rng.standard_normal((H, ETC_N_LABELS, D), dtype=np.float32), w.dtype)
    return {"code_l2l": c_ll, "code_l2g": c_lg, "code_g2l": c_gl, "code_g2g": c_gg, "rel_k": rel,
            "sent_ids": sent_ids, "doc_of_sent": doc_of_sent}


def make_global_projections(w: Workload) -> dict:
    """Separate projections for global attention, [B, H, N, D] each: q_glob,
    k_glob, v_glob iid N(0, 1) from default_rng(seed + 4243), in the
    workload's dtype."""
    rng = np.random.default_rng(w.seed + 4243)
    shape = (w.B, w.H, w.N, w.D)
    return {n: _round(rng.standard_normal(shape, dtype=np.float32), w.dtype) for n in ("q_glob", "k_glob", "v_glob")}
