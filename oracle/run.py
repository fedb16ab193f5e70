"""Oracle over a synthetic workload (test infrastructure only).

Builds the oracle's own cache state from the seeded inputs of `workloads`
and evaluates the explicit definition for a subset of sequences.
"""
from __future__ import annotations

import numpy as np

import workloads as W

from . import qkmla_oracle as O


def sequence_cache(w: W.Workload, b: int, plain: bool = False, host_seq=None):
    """(c^, r^, alpha^k) of sequence b in token order, fp64."""
    wk, _, _, _, grk = W.weights(w)
    c, r = W.sequence(w, b) if host_seq is None else host_seq
    return O.append_tokens(c, r, wk, grk, w.eps, w.cache_dtype, plain=plain, alpha_dtype=w.alpha_dtype)


def reference(w: W.Workload, seqs=None, plain: bool = False, heads=None, host_seqs=None):
    """Explicit-definition outputs for sequences `seqs` (default: all).

    Returns (o [n, s_q, H, d_c], lse [n, s_q, H]) for the selected sequences.
    `heads` restricts the evaluation to the KV groups of those heads (others 0).
    """
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    wk, gq, gk, grq, _ = W.weights(w)
    q, qr = W.queries(w)
    caches = []
    for b in seqs:
        c, r = W.sequence(w, b) if host_seqs is None else host_seqs[b]
        # the explicit form needs only the stored latent and RoPE key
        caches.append((O.cache_cast(c, w.cache_dtype), O.rope_key(r, W.weights(w)[4], w.eps, w.cache_dtype, plain)))
    if heads is None:
        return O.decode_explicit(q[seqs], qr[seqs], gq, gk, grq, wk, caches, w.s_q, w.scale, w.eps, plain=plain)
    hpg = w.H // w.G
    groups = sorted({h // hpg for h in heads})
    o = np.zeros((len(seqs), w.s_q, w.H, w.d_c))
    lse = np.zeros((len(seqs), w.s_q, w.H))
    for g in groups:
        hs = slice(g * hpg, (g + 1) * hpg)
        og, lg = O.decode_explicit(q[seqs][:, :, hs], qr[seqs][:, :, hs], gq, gk, grq, wk[g:g + 1], caches,
                                   w.s_q, w.scale, w.eps, plain=plain)
        o[:, :, hs] = og
        lse[:, :, hs] = lg
    return o, lse


def reference_absorbed(w: W.Workload, seqs=None, plain: bool = False):
    """Absorbed-form outputs for sequences `seqs` (default: all), from the
    oracle's own cache state -- including alpha^k in the workload's A^k_cache
    element type (fp16 rounding when alpha_dtype is "f16").

    Returns (o [n, s_q, H, d_c], lse [n, s_q, H]).
    """
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    wk, gq, gk, grq, _ = W.weights(w)
    q, qr = W.queries(w)
    qs = q[seqs]
    qt, aq = O.absorb_query(qs.reshape(-1, w.H, w.d_h), gq, gk, wk, w.eps, plain=plain)
    qt = qt.reshape(len(seqs), w.s_q, w.H, w.d_c)
    aq = aq.reshape(len(seqs), w.s_q, w.H)
    caches = [sequence_cache(w, b, plain=plain) for b in seqs]
    return O.decode_absorbed(qt, aq, qr[seqs], grq, caches, w.G, w.s_q, w.scale, w.eps, plain=plain)
