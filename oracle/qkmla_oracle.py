"""CPU oracle for QK-Normed MLA decode attention (fp64, numpy).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module; only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference legs use it.  It shares no code with the CUDA
library: its only inputs are the seeded arrays of the `workloads` module.

Sources (all from the web pages on "QK-Normed MLA: QK normalization without
full key caching", arXiv 2606.16310):

  [PS]   gist.science Technical Summary, "Problem Statement": MLA caches the
         latent c_t and recovers the key as k_{t,g} = c_t W^K_g; post-projection
         QK RMSNorm seemingly needs that full key for every cached token.
  [RMS]  same page, "Methodology", RMSNorm decomposition equation:
         RMSNorm(z) = z (.) gamma / S(z), gamma static, S(z) a dynamic RMS scalar.
  [ABS]  "Methodology", Static Weight Absorption: gamma_k (and gamma_q)
         pre-multiply the query before the latent dot product.
  [DYN]  "Methodology", Dynamic Scalar Caching: one inverse-RMS scalar
         alpha_{t,g} = 1/S_{t,g} per token and KV group.
  [LAY]  "Methodology", Cache Layout: keep c_t, add the scalar cache A^k_cache,
         never store full normalised keys.
  [BLK]  "Methodology", Blockwise Normalization: the content and RoPE parts are
         normalised separately; RoPE uses standard materialised vectors.
  [LOG]  "Methodology", decode-logit equation:
         l_{i,t,h} = (q~_{i,h} . c_t) alpha^q_{i,h} alpha^k_{t,g(h)}, the scalars
         applied as a row/column scaling before the softmax.
  [EXACT] thelatestinai.com abstract: the absorbed form is exactly equivalent
         to explicit post-projection QK RMSNorm in exact arithmetic and keeps
         MLA's latent decode path.
  [UP]   Technical Summary, "Problem Statement": MLA keeps the latent and
         recovers per-head quantities through up-projections (W^K_g for keys).
  [QPROJ] thelatestinai.com abstract: the static key weight is absorbed into
         the MLA query-side projection -- the query comes from the layer input
         x through W^Q before the absorption.

Readings where the pages are silent:
  * g(h) = h // (H/G) (contiguous head groups).
  * gamma_q, gamma_k are one [d_h] vector each, shared by all heads/groups.
  * S(z) = sqrt(mean(z^2) + eps) over the d_h entries of one head/group
    (eps inside the root).
  * The RoPE block: one post-RoPE key r_t per token shared by all groups,
    normalised with its own gamma (ones by default) and stored normalised;
    the query RoPE part is normalised per head inside decode.
  * alpha^k is computed from the stored (cache-dtype-rounded) latent.
  * Values are the latents: o = sum_t p_t c^_t (latent-space output).  Per-head
    values come from o by a value up-projection W^V_{g(h)} (per group, like
    W^K_g; G_v = H is one matrix per head), stored in bf16.
  * s_q > 1: query i of the step sees tokens t < seq_len - s_q + i + 1.
  * lse is the natural log of sum_t exp(l_t) with the logit scale included.
  * Plain-MLA mode (comparator): no norms, l = scale (q W^K_g^T . c^ + q_r . r^).
  * RoPE (the pages name none): the original rotary formulation on interleaved
    pairs, (x_2i, x_2i+1) rotated by pos * theta^(-2i/d_r); rotation comes
    before the RMS normalisation of the RoPE block (the normalised vectors are
    the rotated ones, as the post-RoPE inputs of the decode path).
  * Reduced-precision scalar cache (the scalar cache is the method's whole
    storage overhead: Technical Summary, Key Contributions and Results): alpha^k
    stored in IEEE half precision is the round-to-nearest-even fp16 of the fp32
    alpha^k, and decode uses the stored value.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_rne", "cache_cast", "inv_rms", "group_of_head",
    "absorb_query", "append_tokens", "rope_key", "full_keys",
    "decode_explicit", "decode_absorbed", "combine_partials",
    "valid_length", "cache_write", "cache_gather", "up_project",
    "rope_rotate", "project_query",
]


# ----------------------------------------------------------------------------
# storage rounding
# ----------------------------------------------------------------------------
def bf16_rne(x) -> np.ndarray:
    """Round fp32 values to bfloat16 (round to nearest, ties to even) and return
    them as fp32.  Textbook bit arithmetic on the IEEE-754 binary32 pattern:
    add 0x7FFF plus the lowest kept bit, then clear the low 16 bits.  NaNs are
    kept as (quiet) NaNs."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    keep = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep) & np.uint64(0xFFFF0000)).astype(np.uint32)
    out = r.view(np.float32).copy()
    nan = np.isnan(a)
    if nan.any():
        out[nan] = np.float32(np.nan)
    return out


def cache_cast(x, cache_dtype: str) -> np.ndarray:
    """Value held by the cache for an fp32 input, returned in fp64."""
    x32 = np.asarray(x, dtype=np.float32)
    if cache_dtype == "f32":
        return x32.astype(np.float64)
    if cache_dtype == "bf16":
        return bf16_rne(x32).astype(np.float64)
    raise ValueError(cache_dtype)


# ----------------------------------------------------------------------------
# RMS statistic and grouping
# ----------------------------------------------------------------------------
def inv_rms(z, eps: float) -> np.ndarray:
    """alpha = 1 / S(z) with S(z) = sqrt(mean_j z_j^2 + eps) over the last axis
    ([RMS] decomposition; [DYN] inverse-RMS scalar)."""
    z = np.asarray(z, dtype=np.float64)
    return 1.0 / np.sqrt(np.mean(z * z, axis=-1) + eps)


def group_of_head(H: int, G: int) -> np.ndarray:
    """g(h) for every head: contiguous groups of H/G heads."""
    assert H % G == 0
    return np.arange(H) // (H // G)


# ----------------------------------------------------------------------------
# the three calls, stated directly
# ----------------------------------------------------------------------------
def absorb_query(q, gamma_q, gamma_k, w_k, eps: float, plain: bool = False):
    """Query side of the absorbed formulation ([ABS], [LOG]).

    q [R, H, d_h] (R = B*s_q rows), gamma_q/gamma_k [d_h], w_k [G, d_c, d_h].
    Returns q~ [R, H, d_c] = W^K_{g(h)} (q (.) gamma_q (.) gamma_k), i.e. the
    vector whose dot with a latent c gives (q (.) gamma_q (.) gamma_k) . (c W^K_g),
    and alpha^q [R, H] = 1/S(q).  Plain mode: q~ = W^K_g q, alpha^q = 1.
    """
    q = np.asarray(q, dtype=np.float64)
    w = np.asarray(w_k, dtype=np.float64)
    R, H, d_h = q.shape
    G = w.shape[0]
    g_of = group_of_head(H, G)
    if plain:
        qp = q
        aq = np.ones((R, H))
    else:
        qp = q * np.asarray(gamma_q, np.float64) * np.asarray(gamma_k, np.float64)
        aq = inv_rms(q, eps)
    qt = np.empty((R, H, w.shape[1]))
    for h in range(H):
        qt[:, h, :] = qp[:, h, :] @ w[g_of[h]].T
    return qt, aq


def append_tokens(c_new, r_new, w_k, gamma_rk, eps: float, cache_dtype: str, plain: bool = False,
                  alpha_dtype: str = "f32"):
    """Cache entries of new tokens ([LAY], [DYN], [BLK]).

    c_new [N, d_c], r_new [N, d_r] (post-RoPE), w_k [G, d_c, d_h].
    Returns (c^ [N, d_c], r^ [N, d_r], alpha^k [N, G]), all fp64:
      c^      = latent rounded to the cache dtype (the stored state),
      alpha^k = 1 / S(c^ W^K_g) for every group g,
      r^      = RoPE key normalised with its own statistic and gamma, then
                rounded to the cache dtype.
    Plain mode: r^ = rounded raw r, alpha^k = 1.  alpha_dtype "f16": the
    stored alpha^k is the fp16 rounding of its fp32 value ([DYN], [LAY]).
    """
    c_hat = cache_cast(c_new, cache_dtype)
    w = np.asarray(w_k, dtype=np.float64)
    G = w.shape[0]
    N = c_hat.shape[0]
    r = np.asarray(r_new, dtype=np.float64)
    if plain:
        ak = np.ones((N, G))
        return c_hat, rope_key(r_new, gamma_rk, eps, cache_dtype, plain=True), ak
    ak = np.empty((N, G))
    for g in range(G):
        ak[:, g] = inv_rms(c_hat @ w[g], eps)
    if alpha_dtype == "f16":
        # IEEE binary32 -> binary16, round to nearest even (numpy's cast)
        ak = ak.astype(np.float32).astype(np.float16).astype(np.float64)
    elif alpha_dtype != "f32":
        raise ValueError(alpha_dtype)
    return c_hat, rope_key(r_new, gamma_rk, eps, cache_dtype), ak


def rope_key(r_new, gamma_rk, eps: float, cache_dtype: str, plain: bool = False) -> np.ndarray:
    """Stored RoPE key ([BLK]): r (.) gamma_rk / S(r), rounded to the cache dtype
    (plain mode: the rounded raw key)."""
    if plain:
        return cache_cast(np.asarray(r_new, np.float32), cache_dtype)
    r = np.asarray(r_new, dtype=np.float64)
    gr = np.ones(r.shape[1]) if gamma_rk is None else np.asarray(gamma_rk, np.float64)
    beta = inv_rms(r, eps)
    return cache_cast((r * gr * beta[:, None]).astype(np.float32), cache_dtype)


def full_keys(c_hat, w_k) -> np.ndarray:
    """k_{t,g} = c^_t W^K_g for every token and group, [N, G, d_h] ([PS]).
    This is the materialisation the method avoids; only the oracle does it."""
    c = np.asarray(c_hat, dtype=np.float64)
    w = np.asarray(w_k, dtype=np.float64)
    return np.stack([c @ w[g] for g in range(w.shape[0])], axis=1)


def valid_length(seq_len: int, s_q: int, i: int) -> int:
    """Tokens visible to query i of a step with s_q queries (causal in the step)."""
    return int(seq_len) - s_q + i + 1


def _softmax_out(logits, values):
    """Standard softmax over tokens and the latent-space output.
    logits [L, n], values [L, d_c] -> (o [n, d_c], lse [n])."""
    m = logits.max(axis=0)
    e = np.exp(logits - m)
    s = e.sum(axis=0)
    p = e / s
    return p.T @ values, m + np.log(s)


def decode_explicit(q, q_rope, gamma_q, gamma_k, gamma_rq, w_k, seqs, s_q: int,
                    scale: float, eps: float, plain: bool = False):
    """Attention with explicit post-projection QK RMSNorm: the plain definition
    that the absorbed form must equal ([PS], [RMS], [EXACT]).

    q [B, s_q, H, d_h], q_rope [B, s_q, H, d_r] (raw, post-RoPE), w_k [G, d_c, d_h].
    seqs: list over b of (c^ [L_b, d_c], r^ [L_b, d_r]) -- the cache state of
    each sequence in token order (stored values, rope key already normalised).
    For every head the full key k = c^ W^K_g is materialised, RMS-normalised with
    gamma_k, the query RMS-normalised with gamma_q, the RoPE query normalised
    with gamma_rq; logits l = scale (q^ . k^ + q^_r . r^); softmax; o = sum p c^.
    Returns o [B, s_q, H, d_c], lse [B, s_q, H].
    """
    q = np.asarray(q, np.float64)
    qr = np.asarray(q_rope, np.float64)
    w = np.asarray(w_k, np.float64)
    gq = np.asarray(gamma_q, np.float64)
    gk = np.asarray(gamma_k, np.float64)
    B, _, H, d_h = q.shape
    G = w.shape[0]
    hpg = H // G
    d_c = w.shape[1]
    d_r = qr.shape[-1]
    grq = np.ones(d_r) if gamma_rq is None else np.asarray(gamma_rq, np.float64)
    o = np.zeros((B, s_q, H, d_c))
    lse = np.zeros((B, s_q, H))
    for b in range(B):
        c_hat, r_hat = seqs[b]
        c_hat = np.asarray(c_hat, np.float64)
        r_hat = np.asarray(r_hat, np.float64)
        for g in range(G):
            k = c_hat @ w[g]                                        # [L, d_h]
            if plain:
                k_hat = k
            else:
                k_hat = k * gk * inv_rms(k, eps)[:, None]
            for i in range(s_q):
                L = valid_length(c_hat.shape[0], s_q, i)
                hs = slice(g * hpg, (g + 1) * hpg)
                qh = q[b, i, hs]                                    # [hpg, d_h]
                qrh = qr[b, i, hs]
                if plain:
                    q_hat, qr_hat = qh, qrh
                else:
                    q_hat = qh * gq * inv_rms(qh, eps)[:, None]
                    qr_hat = qrh * grq * inv_rms(qrh, eps)[:, None]
                logits = scale * (k_hat[:L] @ q_hat.T + r_hat[:L] @ qr_hat.T)
                oo, ll = _softmax_out(logits, c_hat[:L])
                o[b, i, hs] = oo
                lse[b, i, hs] = ll
    return o, lse


def decode_absorbed(q_tilde, alpha_q, q_rope, gamma_rq, seqs, G: int, s_q: int,
                    scale: float, eps: float, plain: bool = False, token_range=None):
    """Absorbed decode ([LOG], [BLK]): l = scale (alpha^q alpha^k_{t,g(h)} (q~ . c^_t)
    + q^_r . r^_t), softmax, o = sum_t p_t c^_t.  Never forms a full key.

    q_tilde [B, s_q, H, d_c], alpha_q [B, s_q, H], q_rope [B, s_q, H, d_r] raw.
    seqs: list over b of (c^ [L_b, d_c], r^ [L_b, d_r], alpha^k [L_b, G]).
    token_range: optional (lo, hi) restricting the tokens (a split-KV part; the
    causal limit still applies).  Plain mode: l = scale (q~ . c^ + q_r . r^).
    Returns o [B, s_q, H, d_c], lse [B, s_q, H]; a part with no tokens gives
    o = 0, lse = -inf.
    """
    qt = np.asarray(q_tilde, np.float64)
    aq = np.asarray(alpha_q, np.float64)
    qr = np.asarray(q_rope, np.float64)
    B, _, H, d_c = qt.shape
    d_r = qr.shape[-1]
    g_of = group_of_head(H, G)
    grq = np.ones(d_r) if gamma_rq is None else np.asarray(gamma_rq, np.float64)
    o = np.zeros((B, s_q, H, d_c))
    lse = np.full((B, s_q, H), -np.inf)
    for b in range(B):
        c_hat, r_hat, ak = (np.asarray(a, np.float64) for a in seqs[b])
        for i in range(s_q):
            L = valid_length(c_hat.shape[0], s_q, i)
            lo, hi = (0, L) if token_range is None else (max(0, token_range[0]), min(L, token_range[1]))
            if hi <= lo:
                continue
            content = c_hat[lo:hi] @ qt[b, i].T                     # [n, H]
            if plain:
                rope = r_hat[lo:hi] @ qr[b, i].T
                logits = scale * (content + rope)
            else:
                qr_hat = qr[b, i] * grq * inv_rms(qr[b, i], eps)[:, None]
                rope = r_hat[lo:hi] @ qr_hat.T
                logits = scale * (aq[b, i][None, :] * ak[lo:hi][:, g_of] * content + rope)
            oo, ll = _softmax_out(logits, c_hat[lo:hi])
            o[b, i] = oo
            lse[b, i] = ll
    return o, lse


def combine_partials(o_parts, lse_parts):
    """Merge split-KV parts: lse = log sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s.
    o_parts [S, ..., d_c] (each normalised over its own tokens), lse_parts [S, ...]."""
    o_parts = np.asarray(o_parts, np.float64)
    lse_parts = np.asarray(lse_parts, np.float64)
    m = np.max(lse_parts, axis=0)
    w = np.exp(lse_parts - m)
    s = w.sum(axis=0)
    lse = m + np.log(s)
    o = np.einsum("s...,s...d->...d", w / s, o_parts)
    return o, lse


def up_project(o, w_v):
    """Per-head values from the latent output ([UP]): out[..., h, :] = o[..., h, :] W^V_{g(h)}.
    o [..., H, d_c], w_v [G_v, d_c, d_v] (the stored weights).  Returns [..., H, d_v]."""
    o = np.asarray(o, np.float64)
    w = np.asarray(w_v, np.float64)
    H = o.shape[-2]
    g_of = group_of_head(H, w.shape[0])
    out = np.empty(o.shape[:-1] + (w.shape[2],))
    for h in range(H):
        out[..., h, :] = o[..., h, :] @ w[g_of[h]]
    return out


def rope_rotate(x, pos, theta: float):
    """Rotary position embedding on interleaved pairs: (x_2i, x_2i+1) rotated by
    the angle pos * theta^(-2i/d), d = x.shape[-1].  x [..., d]; pos broadcasts
    against x[..., 0] (one position per vector).  fp64."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    inv_freq = np.power(float(theta), -np.arange(0, d, 2, dtype=np.float64) / d)      # [d/2]
    ang = np.asarray(pos, np.float64)[..., None] * inv_freq                          # [..., d/2]
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 0::2] * s + x[..., 1::2] * c
    return out


def project_query(x, w_q, d_h: int, pos, theta: float):
    """The query side before the absorption ([QPROJ]): q_h = x W^Q_h for every head.
    x [R, d_x], w_q [H, d_h + d_r, d_x] (row j of W^Q_h holds output j's weights),
    pos [R].  Returns q [R, H, d_h] (the content part) and q_rope [R, H, d_r]
    (the RoPE part, rotated by each row's position; not normalised)."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w_q, np.float64)
    full = np.einsum("rk,hjk->rhj", x, w)
    pos = np.asarray(pos)
    return full[..., :d_h], rope_rotate(full[..., d_h:], pos[:, None], theta)


# ----------------------------------------------------------------------------
# paged cache state
# ----------------------------------------------------------------------------
def cache_write(kv, ak, slots, c_hat, r_hat, alpha_k):
    """Write appended entries into flat cache arrays: kv[slot] = [c^ | r^],
    ak[slot] = alpha^k[0..G-1]; a negative slot is skipped."""
    slots = np.asarray(slots, np.int64)
    ok = slots >= 0
    d_c = c_hat.shape[1]
    kv[slots[ok], :d_c] = c_hat[ok]
    kv[slots[ok], d_c:] = r_hat[ok]
    ak[slots[ok]] = alpha_k[ok]


def cache_gather(kv, ak, page_table, page_size: int, b: int, L: int, d_c: int):
    """Token-ordered (c^, r^, alpha^k) of sequence b from the flat cache:
    slot(t) = page_table[b][t // page_size] * page_size + t % page_size."""
    t = np.arange(L, dtype=np.int64)
    slots = page_table[b, t // page_size].astype(np.int64) * page_size + t % page_size
    rows = kv[slots]
    return rows[:, :d_c], rows[:, d_c:], ak[slots]
