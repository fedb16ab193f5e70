"""Seeded synthetic inputs for QK-Normed MLA decode.

This module only draws random numbers and lays out shapes.  It holds none of
the method's arithmetic (no RMS statistic, no projection, no softmax), so that
both the CPU oracle and the CUDA path can take their inputs from it without
sharing any of the computation under test.

Workloads follow the five decode configurations of this project:

  0  tiny fp32          B=1,   s_q=1, H=16,  G=4, d_c=128, d_h=64,  d_r=32, T=256
  1  small bf16         B=16,  s_q=1, H=16,  G=4, d_c=256, d_h=64,  d_r=32, T~U[1024,8192]
  2  DeepSeek-V3 shape  B=64,  s_q=1, H=128, G=8, d_c=512, d_h=128, d_r=64, T=4096, paged 64
  3  long context       B=4,   s_q=1, same heads, T=262144, paged 64, 1% outliers x50
  4  mixed serving      B=128, s_q=2, same heads, T log-uniform [512,131072], paged 64

Value distributions: latents c_t, raw RoPE keys r_t, queries q and q_rope are
N(0,1) fp32; W^K_g ~ N(0, 1/d_c); gamma_q, gamma_k = 1 + 0.1 N(0,1); the RoPE
gammas are ones; eps = 1e-6.  A fixed fraction of each sequence's tokens (drawn
without replacement) has both c_t and r_t multiplied by the outlier factor.

Every stream is keyed by (seed, purpose[, sequence]) so one sequence can be
regenerated alone (the oracle samples single sequences of the large workloads).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

TILE_ALIGN = 64  # page size of the paged workloads


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    s_q: int
    H: int
    G: int
    d_c: int
    d_h: int
    d_r: int
    cache_dtype: str          # "f32" or "bf16"
    lens: tuple               # ("fixed", T) | ("uniform", lo, hi) | ("loguniform", lo, hi)
    outlier_frac: float
    outlier_scale: float
    page_size: Optional[int]  # None: contiguous cache, slot = b * max_seq + t
    n_append: int             # new latents appended per sequence inside one step
    seed: int
    eps: float = 1e-6
    rope_gamma_std: float = 0.0   # RoPE gammas = 1 + std * N(0,1) (0: ones, the pages name none)
    alpha_dtype: str = "f32"      # A^k_cache element type: "f32" or "f16"

    @property
    def scale(self) -> float:
        # logit scale 1/sqrt(d_h + d_r) for every workload
        return 1.0 / math.sqrt(self.d_h + self.d_r)

    @property
    def rows(self) -> int:
        return self.B * self.s_q

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = [
    Workload("tiny_fp32_B1_T256", 1, 1, 16, 4, 128, 64, 32, "f32", ("fixed", 256),
             0.05, 30.0, None, 0, 1000),
    Workload("small_bf16_B16_T1k-8k", 16, 1, 16, 4, 256, 64, 32, "bf16", ("uniform", 1024, 8192),
             0.05, 30.0, None, 1, 1001),
    Workload("dsv3_bf16_B64_T4096_paged", 64, 1, 128, 8, 512, 128, 64, "bf16", ("fixed", 4096),
             0.05, 30.0, 64, 0, 1002),
    Workload("dsv3_bf16_B4_T256k_paged", 4, 1, 128, 8, 512, 128, 64, "bf16", ("fixed", 262144),
             0.01, 50.0, 64, 0, 1003),
    Workload("dsv3_bf16_B128_sq2_T512-128k_paged", 128, 2, 128, 8, 512, 128, 64, "bf16",
             ("loguniform", 512, 131072), 0.05, 30.0, 64, 2, 1004),
]


def _rng(*key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(list(key)))


def seq_lens(w: Workload) -> np.ndarray:
    """Context length of every sequence (tokens, including this step's s_q)."""
    kind = w.lens[0]
    if kind == "list":
        return np.array(w.lens[1:], dtype=np.int64)
    if kind == "fixed":
        return np.full(w.B, w.lens[1], dtype=np.int64)
    g = _rng(w.seed, 3)
    if kind == "uniform":
        return g.integers(w.lens[1], w.lens[2], size=w.B, endpoint=True).astype(np.int64)
    if kind == "loguniform":
        lo, hi = math.log(w.lens[1]), math.log(w.lens[2])
        return np.clip(np.round(np.exp(g.uniform(lo, hi, size=w.B))), w.lens[1], w.lens[2]).astype(np.int64)
    raise ValueError(kind)


def weights(w: Workload):
    """W^K [G, d_c, d_h] ~ N(0, 1/d_c); gamma_q, gamma_k [d_h] = 1 + 0.1 N(0,1);
    RoPE gammas [d_r] = ones, or 1 + rope_gamma_std N(0,1) from a stream of
    their own (so the other draws do not change).  All fp32."""
    g = _rng(w.seed, 0)
    wk = (g.standard_normal((w.G, w.d_c, w.d_h), dtype=np.float32) / np.float32(math.sqrt(w.d_c))).astype(np.float32)
    gq = (1.0 + 0.1 * g.standard_normal(w.d_h, dtype=np.float32)).astype(np.float32)
    gk = (1.0 + 0.1 * g.standard_normal(w.d_h, dtype=np.float32)).astype(np.float32)
    if w.rope_gamma_std > 0:
        gr = _rng(w.seed, 5)
        grq = (1.0 + w.rope_gamma_std * gr.standard_normal(w.d_r, dtype=np.float32)).astype(np.float32)
        grk = (1.0 + w.rope_gamma_std * gr.standard_normal(w.d_r, dtype=np.float32)).astype(np.float32)
    else:
        grq = np.ones(w.d_r, dtype=np.float32)
        grk = np.ones(w.d_r, dtype=np.float32)
    return wk, gq, gk, grq, grk


def value_weights(w: Workload, d_v: Optional[int] = None, G_v: Optional[int] = None) -> np.ndarray:
    """W^V [G_v, d_c, d_v] ~ N(0, 1/d_c), fp32 (d_v defaults to d_h, G_v to G)."""
    d_v = w.d_h if d_v is None else d_v
    G_v = w.G if G_v is None else G_v
    g = _rng(w.seed, 6)
    return (g.standard_normal((G_v, w.d_c, d_v), dtype=np.float32) / np.float32(math.sqrt(w.d_c))).astype(np.float32)


def query_inputs(w: Workload, d_x: int):
    """The layer input of the step's query rows x [B, s_q, d_x] ~ N(0,1) and the query
    projection W^Q [H, d_h + d_r, d_x] ~ N(0, 1/d_x) (content rows, then RoPE rows), fp32."""
    g = _rng(w.seed, 7)
    x = g.standard_normal((w.B, w.s_q, d_x), dtype=np.float32)
    wq = (g.standard_normal((w.H, w.d_h + w.d_r, d_x), dtype=np.float32) / np.float32(math.sqrt(d_x))).astype(np.float32)
    return x, wq


def sequence(w: Workload, b: int, length: Optional[int] = None):
    """Latents c [L, d_c] and raw post-RoPE keys r [L, d_r] of sequence b (fp32),
    with the outlier tokens already scaled."""
    L = int(seq_lens(w)[b]) if length is None else int(length)
    g = _rng(w.seed, 1, b)
    c = g.standard_normal((L, w.d_c), dtype=np.float32)
    r = g.standard_normal((L, w.d_r), dtype=np.float32)
    n_out = int(round(w.outlier_frac * L))
    if n_out:
        idx = g.choice(L, size=n_out, replace=False)
        c[idx] *= np.float32(w.outlier_scale)
        r[idx] *= np.float32(w.outlier_scale)
    return c, r


def queries(w: Workload):
    """q [B, s_q, H, d_h] and q_rope [B, s_q, H, d_r], fp32 N(0,1)."""
    g = _rng(w.seed, 2)
    q = g.standard_normal((w.B, w.s_q, w.H, w.d_h), dtype=np.float32)
    qr = g.standard_normal((w.B, w.s_q, w.H, w.d_r), dtype=np.float32)
    return q, qr


def page_layout(w: Workload, lens: Optional[np.ndarray] = None):
    """Page geometry of the cache.

    Returns (page_size, max_pages, num_slots, page_table [B, max_pages] int32).
    Paged workloads draw one random permutation of all physical pages; the
    contiguous ones use page b*max_pages + p, i.e. slot = b*max_seq + t.
    Unused table entries are -1 on paged workloads.
    """
    lens = seq_lens(w) if lens is None else np.asarray(lens)
    if w.page_size is None:
        ps = TILE_ALIGN
        max_pages = int(-(-int(lens.max()) // ps))
        table = (np.arange(w.B, dtype=np.int64)[:, None] * max_pages
                 + np.arange(max_pages, dtype=np.int64)[None, :]).astype(np.int32)
        return ps, max_pages, w.B * max_pages * ps, table
    ps = w.page_size
    pages = [int(-(-int(L) // ps)) for L in lens]
    max_pages = max(pages)
    total = sum(pages)
    perm = _rng(w.seed, 4).permutation(total)
    table = np.full((w.B, max_pages), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(pages):
        table[b, :n] = perm[k:k + n]
        k += n
    return ps, max_pages, total * ps, table


def slots_of(page_table: np.ndarray, page_size: int, b: int, t: np.ndarray) -> np.ndarray:
    """Physical slot of tokens t of sequence b: page_table[b][t // ps] * ps + t % ps."""
    t = np.asarray(t, dtype=np.int64)
    return page_table[b, t // page_size].astype(np.int64) * page_size + t % page_size


def small(w: Workload, B: int, lens, **kw) -> Workload:
    """A reduced copy of a workload (same heads and dims) with explicit lengths."""
    lens = tuple(int(x) for x in lens)
    assert len(lens) == B
    return w.with_(B=B, lens=("list",) + lens, **kw)
