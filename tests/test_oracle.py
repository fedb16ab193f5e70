"""Pins of the fp64 CPU oracle against facts fixed outside it.

Each test ties the oracle to something it does not compute itself: library
routines it does not use (torch RMSNorm, torch scaled-dot-product attention,
torch's bfloat16 cast), closed forms, invariants of the method, the exact
equivalence the pages claim between the absorbed and the explicit form, and
the cache-overhead figures the pages print.  Mutation tests at the end plant
plausible mistakes into copies of oracle functions and check that a pin fails.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand_case(seed, B=2, s_q=1, H=8, G=2, d_c=48, d_h=24, d_r=16, lens=(37, 70), cache="f32",
               outliers=True):
    g = np.random.default_rng(seed)
    wk = (g.standard_normal((G, d_c, d_h)) / math.sqrt(d_c)).astype(np.float32)
    gq = (1 + 0.1 * g.standard_normal(d_h)).astype(np.float32)
    gk = (1 + 0.1 * g.standard_normal(d_h)).astype(np.float32)
    grk = (1 + 0.1 * g.standard_normal(d_r)).astype(np.float32)
    grq = (1 + 0.1 * g.standard_normal(d_r)).astype(np.float32)
    q = g.standard_normal((B, s_q, H, d_h)).astype(np.float32)
    qr = g.standard_normal((B, s_q, H, d_r)).astype(np.float32)
    seqs_raw = []
    for b in range(B):
        c = g.standard_normal((lens[b], d_c)).astype(np.float32)
        r = g.standard_normal((lens[b], d_r)).astype(np.float32)
        if outliers:
            idx = g.choice(lens[b], size=max(1, lens[b] // 20), replace=False)
            c[idx] *= 30
            r[idx] *= 30
        seqs_raw.append((c, r))
    return dict(wk=wk, gq=gq, gk=gk, grk=grk, grq=grq, q=q, qr=qr, seqs_raw=seqs_raw,
                B=B, s_q=s_q, H=H, G=G, d_c=d_c, d_h=d_h, d_r=d_r, cache=cache,
                scale=1 / math.sqrt(d_h + d_r), eps=1e-6)


def _build(case, plain=False):
    exp_seqs, abs_seqs = [], []
    for c, r in case["seqs_raw"]:
        ch, rh, ak = O.append_tokens(c, r, case["wk"], case["grk"], case["eps"], case["cache"], plain=plain)
        exp_seqs.append((ch, rh))
        abs_seqs.append((ch, rh, ak))
    return exp_seqs, abs_seqs


# --------------------------------------------------------------------------
# storage rounding
# --------------------------------------------------------------------------
def test_bf16_rne_matches_torch_cast():
    g = np.random.default_rng(0)
    x = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * 10.0 ** g.integers(-30, 30, 20000),
        np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.0e38, -3.0e38, 1e-40, -1e-40,
                  1.00390625, 1.01171875, 1.0078125 + 2 ** -9], dtype=np.float32),
    ]).astype(np.float32)
    # exact ties: low 16 bits == 0x8000 with both parities of the kept bit
    ties = (np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x40498000], dtype=np.uint32)).view(np.float32)
    x = np.concatenate([x, ties])
    ours = O.bf16_rne(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_bf16_rne_keeps_nan():
    x = np.array([np.nan, 1.0], dtype=np.float32)
    y = O.bf16_rne(x)
    assert np.isnan(y[0]) and y[1] == 1.0


# --------------------------------------------------------------------------
# RMS statistic: closed forms and torch's RMSNorm
# --------------------------------------------------------------------------
def test_inv_rms_closed_forms():
    d = 64
    for c in [0.5, 3.0, 30.0]:
        assert O.inv_rms(np.full(d, c), 1e-6) == pytest.approx(1 / math.sqrt(c * c + 1e-6), rel=1e-15)
    e = np.zeros(d)
    e[5] = math.sqrt(d)
    assert O.inv_rms(e, 0.0) == pytest.approx(1.0, rel=1e-15)
    assert O.inv_rms(np.zeros(d), 0.25) == pytest.approx(2.0, rel=1e-15)


def test_inv_rms_matches_torch_rms_norm():
    g = np.random.default_rng(1)
    z = g.standard_normal((50, 128)) * 7
    gamma = 1 + 0.1 * g.standard_normal(128)
    ref = F.rms_norm(torch.from_numpy(z), (128,), torch.from_numpy(gamma), eps=1e-6).numpy()
    ours = z * gamma * O.inv_rms(z, 1e-6)[:, None]
    np.testing.assert_allclose(ours, ref, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# explicit definition vs torch library attention (textbook reduction)
# --------------------------------------------------------------------------
def _torch_cache(x, cache):
    """A value as the cache stores it, by torch's own casts (fp64 -> fp32 -> cache dtype)."""
    t = torch.as_tensor(x).to(torch.float32)
    if cache == "bf16":
        t = t.to(torch.bfloat16)
    return t.to(torch.float64)


def _torch_rope_key(r, gamma, eps, cache, plain=False):
    """Stored RoPE key built with torch's rms_norm from the raw key (not from the oracle)."""
    rt = torch.from_numpy(np.asarray(r, np.float64))
    if not plain:
        rt = F.rms_norm(rt, (rt.shape[-1],), torch.from_numpy(np.asarray(gamma, np.float64)), eps=eps)
    return _torch_cache(rt, cache)


def _torch_reference(case, plain=False):
    """Post-projection QK RMSNorm attention with torch's rms_norm and
    scaled_dot_product_attention (fp64, CPU), built from the raw inputs: the
    stored latent and RoPE key come from torch's casts and rms_norm, not from
    the oracle's append."""
    B, s_q, H, G = case["B"], case["s_q"], case["H"], case["G"]
    hpg = H // G
    o_all = np.zeros((B, s_q, H, case["d_c"]))
    for b in range(B):
        c_raw, r_raw = case["seqs_raw"][b]
        ch = _torch_cache(torch.from_numpy(c_raw), case["cache"])
        rh = _torch_rope_key(r_raw, case["grk"], case["eps"], case["cache"], plain)
        T = ch.shape[0]
        for h in range(H):
            g_ = h // hpg
            k = ch @ torch.from_numpy(case["wk"][g_].astype(np.float64))
            qh = torch.from_numpy(case["q"][b, :, h].astype(np.float64))      # [s_q, d_h]
            qrh = torch.from_numpy(case["qr"][b, :, h].astype(np.float64))
            if not plain:
                k = F.rms_norm(k, (case["d_h"],), torch.from_numpy(case["gk"].astype(np.float64)), eps=case["eps"])
                qh = F.rms_norm(qh, (case["d_h"],), torch.from_numpy(case["gq"].astype(np.float64)), eps=case["eps"])
                qrh = F.rms_norm(qrh, (case["d_r"],), torch.from_numpy(case["grq"].astype(np.float64)), eps=case["eps"])
            Q = torch.cat([qh, qrh], dim=-1)[None, None]           # [1,1,s_q,d]
            K = torch.cat([k, rh], dim=-1)[None, None]             # [1,1,T,d]
            V = ch[None, None]
            mask = torch.ones(s_q, T, dtype=torch.bool)
            for i in range(s_q):
                mask[i, O.valid_length(T, s_q, i):] = False
            out = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=case["scale"])
            o_all[b, :, h] = out[0, 0].numpy()
    return o_all


@pytest.mark.parametrize("s_q", [1, 2, 3])
@pytest.mark.parametrize("plain", [False, True])
def test_explicit_matches_torch_sdpa(s_q, plain):
    case = _rand_case(10 + s_q, s_q=s_q, cache="bf16")
    exp_seqs, _ = _build(case, plain=plain)
    o, _ = O.decode_explicit(case["q"], case["qr"], case["gq"], case["gk"], case["grq"], case["wk"],
                             exp_seqs, s_q, case["scale"], case["eps"], plain=plain)
    ref = _torch_reference(case, plain=plain)
    np.testing.assert_allclose(o, ref, rtol=1e-11, atol=1e-11)


# --------------------------------------------------------------------------
# exact equivalence of the absorbed and explicit forms (the pages' claim)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("cache", ["f32", "bf16"])
@pytest.mark.parametrize("s_q", [1, 2])
@pytest.mark.parametrize("plain", [False, True])
def test_absorbed_equals_explicit_fp64(cache, s_q, plain):
    case = _rand_case(20 + s_q, s_q=s_q, cache=cache, H=16, G=4, d_c=64, d_h=32, d_r=16, lens=(130, 257))
    exp_seqs, abs_seqs = _build(case, plain=plain)
    o_e, l_e = O.decode_explicit(case["q"], case["qr"], case["gq"], case["gk"], case["grq"], case["wk"],
                                 exp_seqs, s_q, case["scale"], case["eps"], plain=plain)
    R = case["B"] * s_q
    qt, aq = O.absorb_query(case["q"].reshape(R, case["H"], case["d_h"]), case["gq"], case["gk"],
                            case["wk"], case["eps"], plain=plain)
    o_a, l_a = O.decode_absorbed(qt.reshape(case["B"], s_q, case["H"], -1), aq.reshape(case["B"], s_q, -1),
                                 case["qr"], case["grq"], abs_seqs, case["G"], s_q, case["scale"],
                                 case["eps"], plain=plain)
    tol = 1e-10
    assert np.max(np.abs(l_a - l_e) / np.maximum(1, np.abs(l_e))) <= tol
    assert np.max(np.abs(o_a - o_e) / np.maximum(1, np.abs(o_e))) <= tol


# --------------------------------------------------------------------------
# brute-force tiny cases and closed forms
# --------------------------------------------------------------------------
def test_single_token_returns_its_latent():
    case = _rand_case(30, B=1, lens=(1,))
    exp_seqs, _ = _build(case)
    o, lse = O.decode_explicit(case["q"], case["qr"], case["gq"], case["gk"], case["grq"], case["wk"],
                               exp_seqs, 1, case["scale"], case["eps"])
    c_raw, r_raw = case["seqs_raw"][0]
    c0 = c_raw[0].astype(np.float64)                      # fp32 cache: the stored latent is the input
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(c0, o[0, 0].shape), rtol=0, atol=1e-14)
    # the stored RoPE key, by hand: r gamma_rk / sqrt(mean r^2 + eps), stored in fp32
    r0 = r_raw[0].astype(np.float64)
    rk = (r0 * case["grk"] / math.sqrt(np.mean(r0 * r0) + case["eps"])).astype(np.float32).astype(np.float64)
    # lse = the single logit, computed by hand for head 0 (group 0)
    k = c0 @ case["wk"][0].astype(np.float64)
    kh = k * case["gk"] / math.sqrt(np.mean(k * k) + case["eps"])
    qh = case["q"][0, 0, 0].astype(np.float64)
    qh = qh * case["gq"] / math.sqrt(np.mean(qh * qh) + case["eps"])
    qrh = case["qr"][0, 0, 0].astype(np.float64)
    qrh = qrh * case["grq"] / math.sqrt(np.mean(qrh * qrh) + case["eps"])
    ell = case["scale"] * (float(qh @ kh) + float(qrh @ rk))
    assert lse[0, 0, 0] == pytest.approx(ell, rel=1e-13, abs=1e-13)


def test_two_tokens_logistic_weight():
    case = _rand_case(31, B=1, lens=(2,), outliers=False)
    _, abs_seqs = _build(case)
    qt, aq = O.absorb_query(case["q"][:, 0], case["gq"], case["gk"], case["wk"], case["eps"])
    o, lse = O.decode_absorbed(qt[:, None], aq[:, None], case["qr"], case["grq"], abs_seqs, case["G"], 1,
                               case["scale"], case["eps"])
    ch = abs_seqs[0][0]
    # o = p0 c0 + (1-p0) c1 with p0 = sigmoid(l0 - l1); recover p0 from coordinate 0
    # and check every other coordinate and lse = l1 + log(1 + exp(l0 - l1)).
    for h in range(case["H"]):
        p0 = (o[0, 0, h, 0] - ch[1, 0]) / (ch[0, 0] - ch[1, 0])
        np.testing.assert_allclose(o[0, 0, h], p0 * ch[0] + (1 - p0) * ch[1], rtol=1e-10, atol=1e-12)
        d = math.log(p0 / (1 - p0))            # l0 - l1
        l1 = lse[0, 0, h] - math.log1p(math.exp(d))
        l0 = l1 + d
        assert math.exp(lse[0, 0, h]) == pytest.approx(math.exp(l0) + math.exp(l1), rel=1e-10)


def test_zero_queries_give_uniform_average():
    case = _rand_case(32, B=2, lens=(17, 40))
    case["q"][:] = 0
    case["qr"][:] = 0
    exp_seqs, _ = _build(case)
    o, lse = O.decode_explicit(case["q"], case["qr"], case["gq"], case["gk"], case["grq"], case["wk"],
                               exp_seqs, 1, case["scale"], case["eps"])
    for b in range(2):
        ch = exp_seqs[b][0]
        np.testing.assert_allclose(o[b, 0], np.broadcast_to(ch.mean(0), o[b, 0].shape), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[b, 0], math.log(ch.shape[0]), rtol=1e-14)


def test_equal_latents_return_that_latent():
    case = _rand_case(33, B=1, lens=(50,), outliers=False)
    c, r = case["seqs_raw"][0]
    c[:] = c[0]
    _, abs_seqs = _build(case)
    qt, aq = O.absorb_query(case["q"][:, 0], case["gq"], case["gk"], case["wk"], case["eps"])
    o, _ = O.decode_absorbed(qt[:, None], aq[:, None], case["qr"], case["grq"], abs_seqs, case["G"], 1,
                             case["scale"], case["eps"])
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(abs_seqs[0][0][0], o[0, 0].shape), rtol=1e-12)


# --------------------------------------------------------------------------
# invariants of the method
# --------------------------------------------------------------------------
def test_alpha_k_scale_invariance():
    """With eps = 0, scaling a token's latent and RoPE key by s > 0 leaves every
    normalised logit (hence lse) unchanged: alpha^k absorbs the scale."""
    case = _rand_case(40, B=1, lens=(64,), outliers=False)
    case["eps"] = 0.0
    _, s1 = _build(case)
    c, r = case["seqs_raw"][0]
    c2, r2 = c.copy(), r.copy()
    c2[::3] *= 32.0            # powers of two keep the cache rounding exact
    r2[::3] *= 32.0
    case2 = dict(case, seqs_raw=[(c2, r2)])
    _, s2 = _build(case2)
    qt, aq = O.absorb_query(case["q"][:, 0], case["gq"], case["gk"], case["wk"], 0.0)
    _, l1 = O.decode_absorbed(qt[:, None], aq[:, None], case["qr"], case["grq"], s1, case["G"], 1, case["scale"], 0.0)
    _, l2 = O.decode_absorbed(qt[:, None], aq[:, None], case["qr"], case["grq"], s2, case["G"], 1, case["scale"], 0.0)
    np.testing.assert_allclose(l1, l2, rtol=1e-12)
    # query scale invariance too
    qt3, aq3 = O.absorb_query(case["q"][:, 0] * 8.0, case["gq"], case["gk"], case["wk"], 0.0)
    _, l3 = O.decode_absorbed(qt3[:, None], aq3[:, None], case["qr"] * 8.0, case["grq"], s1, case["G"], 1,
                              case["scale"], 0.0)
    np.testing.assert_allclose(l1, l3, rtol=1e-12)


def test_logits_bounded_by_cauchy_schwarz():
    """|q^ . k^| <= d_h max|gamma_q gamma_k| since ||z / S(z)|| <= sqrt(d): normalised
    logits stay bounded even with outlier tokens."""
    case = _rand_case(41, B=1, lens=(300,), outliers=True)
    exp_seqs, _ = _build(case)
    ch, rh = exp_seqs[0]
    bound = case["scale"] * (case["d_h"] * np.max(np.abs(case["gq"] * case["gk"]))
                             + case["d_r"] * np.max(np.abs(case["grq"] * case["grk"])) * 1.01)
    _, lse = O.decode_explicit(case["q"], case["qr"], case["gq"], case["gk"], case["grq"], case["wk"],
                               exp_seqs, 1, case["scale"], case["eps"])
    # every logit <= bound  =>  lse <= bound + log L ; and >= -bound
    assert np.all(lse <= bound + math.log(300) + 1e-9)
    assert np.all(lse >= -bound - 1e-9)


def test_output_in_convex_hull():
    case = _rand_case(42, B=2, lens=(33, 91))
    exp_seqs, _ = _build(case)
    o, _ = O.decode_explicit(case["q"], case["qr"], case["gq"], case["gk"], case["grq"], case["wk"],
                             exp_seqs, 1, case["scale"], case["eps"])
    for b in range(2):
        ch = exp_seqs[b][0]
        assert np.all(o[b] <= ch.max(0) + 1e-12) and np.all(o[b] >= ch.min(0) - 1e-12)


# --------------------------------------------------------------------------
# split-KV combine and causal masking
# --------------------------------------------------------------------------
@pytest.mark.parametrize("cuts", [(0, 50, 51, 200), (0, 1, 199, 200), (0, 64, 128, 192, 200)])
def test_combine_of_parts_equals_whole(cuts):
    case = _rand_case(50, B=1, lens=(200,))
    _, abs_seqs = _build(case)
    qt, aq = O.absorb_query(case["q"][:, 0], case["gq"], case["gk"], case["wk"], case["eps"])
    args = (qt[:, None], aq[:, None], case["qr"], case["grq"], abs_seqs, case["G"], 1, case["scale"], case["eps"])
    o_full, l_full = O.decode_absorbed(*args)
    parts = [O.decode_absorbed(*args, token_range=(cuts[k], cuts[k + 1])) for k in range(len(cuts) - 1)]
    o_c, l_c = O.combine_partials([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(o_c, o_full, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l_c, l_full, rtol=1e-12)


def test_causal_query_sees_prefix():
    """Query i of an s_q-token step equals a one-token step on the first
    seq_len - s_q + i + 1 tokens."""
    case = _rand_case(51, B=1, s_q=3, lens=(77,))
    exp_seqs, _ = _build(case)
    o, lse = O.decode_explicit(case["q"], case["qr"], case["gq"], case["gk"], case["grq"], case["wk"],
                               exp_seqs, 3, case["scale"], case["eps"])
    for i in range(3):
        L = 77 - 3 + i + 1
        sub = [(exp_seqs[0][0][:L], exp_seqs[0][1][:L])]
        o1, l1 = O.decode_explicit(case["q"][:, i:i + 1], case["qr"][:, i:i + 1], case["gq"], case["gk"],
                                   case["grq"], case["wk"], sub, 1, case["scale"], case["eps"])
        np.testing.assert_array_equal(o[:, i], o1[:, 0])
        np.testing.assert_array_equal(lse[:, i], l1[:, 0])


# --------------------------------------------------------------------------
# cache layout
# --------------------------------------------------------------------------
def test_paged_write_gather_roundtrip():
    w = W.small(W.WORKLOADS[2], 3, (130, 64, 1), page_size=64)
    ps, max_pages, num_slots, table = W.page_layout(w)
    lens = W.seq_lens(w)
    d_c, d_r, G = w.d_c, w.d_r, w.G
    kv = np.full((num_slots, d_c + d_r), np.nan)
    ak = np.full((num_slots, G), np.nan)
    wk = W.weights(w)[0]
    want = []
    for b in range(w.B):
        c, r = W.sequence(w, b)
        ch, rh, a = O.append_tokens(c, r, wk, None, w.eps, "bf16")
        O.cache_write(kv, ak, W.slots_of(table, ps, b, np.arange(lens[b])), ch, rh, a)
        want.append((ch, rh, a))
    # every page is used exactly once and no slot is written twice
    used = table[table >= 0]
    assert len(np.unique(used)) == len(used) == num_slots // ps
    for b in range(w.B):
        got = O.cache_gather(kv, ak, table, ps, b, int(lens[b]), d_c)
        for x, y in zip(got, want[b]):
            np.testing.assert_array_equal(x, y)
    # negative slots are skipped
    kv2 = kv.copy()
    O.cache_write(kv2, ak.copy(), np.array([-1]), want[0][0][:1], want[0][1][:1], want[0][2][:1])
    np.testing.assert_array_equal(np.isnan(kv2), np.isnan(kv))


def test_cache_overhead_matches_printed_figures():
    gold = json.load(open(os.path.join(HERE, "golden", "cache_overhead.json")))
    s = gold["shapes"]
    # bytes of one cache slot: latent + RoPE row in bf16, and the alpha row
    kv_row_bytes = (s["d_c"] + s["d_r"]) * s["latent_bytes_per_elem"]
    ak_row_bytes = s["G"] * s["alpha_bytes"]
    elems_pct = 100.0 * s["G"] / s["d_c"]
    bytes_pct = 100.0 * ak_row_bytes / kv_row_bytes
    for got, key in [(elems_pct, "elements_ratio_pct"), (bytes_pct, "bytes_ratio_pct")]:
        p = gold["printed"][key]
        assert abs(got - p["value"]) <= 0.5 * 10 ** (-p["decimals"]), (key, got)
    # and the oracle's cache rows have exactly that shape
    _, _, a = O.append_tokens(np.zeros((3, s["d_c"]), np.float32) + 1, np.ones((3, s["d_r"]), np.float32),
                              np.ones((s["G"], s["d_c"], 4), np.float32), None, 1e-6, "bf16")
    assert a.shape == (3, s["G"])


def test_workload_streams_are_reproducible():
    w = W.WORKLOADS[1]
    c1, r1 = W.sequence(w, 3)
    c2, r2 = W.sequence(w, 3)
    np.testing.assert_array_equal(c1, c2)
    assert c1.shape == (W.seq_lens(w)[3], w.d_c)
    n_out = int(round(w.outlier_frac * c1.shape[0]))
    assert np.sum(np.abs(c1).max(1) > 8) >= n_out * 0.9


# --------------------------------------------------------------------------
# planted mistakes: each must be caught by one of the pins above
# --------------------------------------------------------------------------
def _absorbed_vs_explicit_gap(absorb_fn):
    case = _rand_case(60, H=8, G=2, d_c=40, d_h=24, d_r=8, lens=(50, 61))
    exp_seqs, abs_seqs = _build(case)
    o_e, l_e = O.decode_explicit(case["q"], case["qr"], case["gq"], case["gk"], case["grq"], case["wk"],
                                 exp_seqs, 1, case["scale"], case["eps"])
    qt, aq = absorb_fn(case["q"][:, 0], case["gq"], case["gk"], case["wk"], case["eps"])
    o_a, l_a = O.decode_absorbed(qt[:, None], aq[:, None], case["qr"], case["grq"], abs_seqs, case["G"], 1,
                                 case["scale"], case["eps"])
    return max(np.max(np.abs(l_a - l_e)), np.max(np.abs(o_a - o_e)))


def test_mutation_dropped_gamma_k_is_caught():
    def bad(q, gq, gk, wk, eps):
        return O.absorb_query(q, gq, np.ones_like(gk), wk, eps)
    assert _absorbed_vs_explicit_gap(O.absorb_query) < 1e-10
    assert _absorbed_vs_explicit_gap(bad) > 1e-3


def test_mutation_wrong_group_is_caught():
    def bad(q, gq, gk, wk, eps):
        return O.absorb_query(q, gq, gk, wk[::-1].copy(), eps)
    assert _absorbed_vs_explicit_gap(bad) > 1e-3


def test_mutation_eps_outside_root_is_caught(monkeypatch):
    real = O.qkmla_oracle.inv_rms
    monkeypatch.setattr(O.qkmla_oracle, "inv_rms",
                        lambda z, eps: 1.0 / (np.sqrt(np.mean(np.asarray(z) ** 2, axis=-1)) + eps))
    case = _rand_case(61, B=1, lens=(40,))
    case["eps"] = 0.3
    case["q"] *= 0.05
    exp_seqs, _ = _build(case)
    o, _ = O.decode_explicit(case["q"], case["qr"], case["gq"], case["gk"], case["grq"], case["wk"],
                             exp_seqs, 1, case["scale"], case["eps"])
    monkeypatch.setattr(O.qkmla_oracle, "inv_rms", real)
    ref = _torch_reference(case)
    assert np.max(np.abs(o - ref)) > 1e-4


@pytest.mark.parametrize("cache", ["f32", "bf16"])
@pytest.mark.parametrize("mutation", ["dropped_gamma_rk", "key_scaled_1.05", "norm_over_wrong_axis"])
def test_mutation_rope_key_is_caught(monkeypatch, cache, mutation):
    """The stored RoPE key is pinned by the torch reference built from the raw key:
    a dropped RoPE gamma, a mis-scaled key or a statistic over the wrong axis in
    the oracle's rope_key must move the explicit decode away from it."""
    real = O.qkmla_oracle.rope_key
    bad = {
        "dropped_gamma_rk": lambda r, g, eps, c, plain=False: real(r, None, eps, c, plain),
        "key_scaled_1.05": lambda r, g, eps, c, plain=False: real(r, g, eps, c, plain) * 1.05,
        "norm_over_wrong_axis": lambda r, g, eps, c, plain=False: O.cache_cast(
            (np.asarray(r, np.float64) * np.asarray(g, np.float64)
             * O.inv_rms(np.asarray(r, np.float64).T, eps)[None, :]).astype(np.float32), c),
    }[mutation]
    case = _rand_case(62, B=2, lens=(40, 57), cache=cache)
    ref = _torch_reference(case)

    def gap():
        exp_seqs, _ = _build(case)
        o, _ = O.decode_explicit(case["q"], case["qr"], case["gq"], case["gk"], case["grq"], case["wk"],
                                 exp_seqs, 1, case["scale"], case["eps"])
        return np.max(np.abs(o - ref))

    assert gap() < 1e-11
    monkeypatch.setattr(O.qkmla_oracle, "rope_key", bad)
    assert gap() > 1e-5


# --------------------------------------------------------------------------
# reduced-precision scalar cache: alpha^k stored in fp16
# --------------------------------------------------------------------------
def test_f16_alpha_is_the_rne_cast_of_fp32_alpha():
    case = _rand_case(70, B=1, lens=(90,))
    c, r = case["seqs_raw"][0]
    _, _, a32 = O.append_tokens(c, r, case["wk"], case["grk"], case["eps"], "bf16")
    _, _, a16 = O.append_tokens(c, r, case["wk"], case["grk"], case["eps"], "bf16", alpha_dtype="f16")
    ref = torch.from_numpy(a32.astype(np.float32)).to(torch.float16).to(torch.float64).numpy()
    np.testing.assert_array_equal(a16, ref)
    # fp16 keeps 11 significant bits: one RNE rounding moves a value by at most 2^-11 of it
    assert np.max(np.abs(a16 / a32 - 1)) <= 2.0 ** -11 + 1e-7


def test_f16_alpha_is_exact_when_alpha_is_a_power_of_two():
    """With W^K = I, eps = 0 and latents of constant magnitude 2^m per token,
    alpha^k = 2^-m is exact in fp16: the half-precision scalar cache changes nothing."""
    g = np.random.default_rng(71)
    d = 16
    wk = np.eye(d, dtype=np.float32)[None]                         # G = 1, d_c = d_h = 16
    L = 40
    c = np.sign(g.standard_normal((L, d))).astype(np.float32) * (2.0 ** g.integers(-3, 4, size=(L, 1))).astype(np.float32)
    r = g.standard_normal((L, 8)).astype(np.float32)
    q = g.standard_normal((1, 1, 4, d)).astype(np.float32)
    qr = g.standard_normal((1, 1, 4, 8)).astype(np.float32)
    gq = np.ones(d, np.float32)
    gk = np.ones(d, np.float32)
    outs = []
    for ad in ("f32", "f16"):
        ch, rh, ak = O.append_tokens(c, r, wk, None, 0.0, "f32", alpha_dtype=ad)
        qt, aq = O.absorb_query(q[:, 0], gq, gk, wk, 0.0)
        outs.append(O.decode_absorbed(qt[:, None], aq[:, None], qr, None, [(ch, rh, ak)], 1, 1, 0.25, 0.0))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


def test_f16_alpha_moves_logits_within_the_rounding_bound():
    """Each content logit moves by at most |content logit| 2^-11 (one fp16 RNE
    rounding of alpha^k), so lse moves by at most the largest such change."""
    case = _rand_case(72, B=1, lens=(300,), H=8, G=2)
    c, r = case["seqs_raw"][0]
    qt, aq = O.absorb_query(case["q"][:, 0], case["gq"], case["gk"], case["wk"], case["eps"])
    res, cont = [], None
    for ad in ("f32", "f16"):
        ch, rh, ak = O.append_tokens(c, r, case["wk"], case["grk"], case["eps"], "f32", alpha_dtype=ad)
        res.append(O.decode_absorbed(qt[:, None], aq[:, None], case["qr"], case["grq"], [(ch, rh, ak)], case["G"], 1,
                                     case["scale"], case["eps"]))
        if ad == "f32":
            g_of = O.group_of_head(case["H"], case["G"])
            cont = case["scale"] * np.abs(aq[0][None, :] * ak[:, g_of] * (ch @ qt[0].T))    # [L, H]
    bound = cont.max(axis=0) * 2.0 ** -11 * 1.001
    dl = np.abs(res[1][1][0, 0] - res[0][1][0, 0])
    assert np.all(dl <= bound + 1e-12)
    assert np.any(dl > 0)                                  # the rounding is visible


# --------------------------------------------------------------------------
# value up-projection
# --------------------------------------------------------------------------
@pytest.mark.parametrize("G_v", [2, 8])
def test_up_projection_equals_attention_over_materialised_values(G_v):
    """o W^V (the latent path, projected once per row) equals torch attention with
    every value v_t = c^_t W^V_{g(h)} materialised (softmax weights sum to one)."""
    case = _rand_case(80, B=2, s_q=2, H=8, G=2, lens=(45, 70), cache="bf16")
    g = np.random.default_rng(81)
    wv = O.bf16_rne(g.standard_normal((G_v, case["d_c"], 12)) / math.sqrt(case["d_c"])).astype(np.float64)
    exp_seqs, _ = _build(case)
    o, _ = O.decode_explicit(case["q"], case["qr"], case["gq"], case["gk"], case["grq"], case["wk"],
                             exp_seqs, 2, case["scale"], case["eps"])
    out = O.up_project(o, wv)
    H, G = case["H"], case["G"]
    for b in range(2):
        c_raw, r_raw = case["seqs_raw"][b]
        ch = _torch_cache(torch.from_numpy(c_raw), "bf16")
        rh = _torch_rope_key(r_raw, case["grk"], case["eps"], "bf16")
        T = ch.shape[0]
        for h in range(H):
            k = F.rms_norm(ch @ torch.from_numpy(case["wk"][h // (H // G)].astype(np.float64)), (case["d_h"],),
                           torch.from_numpy(case["gk"].astype(np.float64)), eps=case["eps"])
            qh = F.rms_norm(torch.from_numpy(case["q"][b, :, h].astype(np.float64)), (case["d_h"],),
                            torch.from_numpy(case["gq"].astype(np.float64)), eps=case["eps"])
            qrh = F.rms_norm(torch.from_numpy(case["qr"][b, :, h].astype(np.float64)), (case["d_r"],),
                             torch.from_numpy(case["grq"].astype(np.float64)), eps=case["eps"])
            V = ch @ torch.from_numpy(wv[h // (H // G_v)])                      # materialised values [T, d_v]
            mask = torch.ones(2, T, dtype=torch.bool)
            for i in range(2):
                mask[i, O.valid_length(T, 2, i):] = False
            ref = F.scaled_dot_product_attention(torch.cat([qh, qrh], -1)[None, None],
                                                 torch.cat([k, rh], -1)[None, None], V[None, None],
                                                 attn_mask=mask, scale=case["scale"])[0, 0].numpy()
            np.testing.assert_allclose(out[b, :, h], ref, rtol=1e-11, atol=1e-12)


def test_mutation_up_projection_wrong_group_is_caught():
    o = np.random.default_rng(82).standard_normal((3, 8, 16))
    wv = np.random.default_rng(83).standard_normal((4, 16, 5))
    ref = np.stack([o[:, h] @ wv[h // 2] for h in range(8)], axis=1)         # g(h) = h // (H / G_v)
    np.testing.assert_allclose(O.up_project(o, wv), ref, rtol=1e-14)
    bad = np.stack([o[:, h] @ wv[h % 4] for h in range(8)], axis=1)          # interleaved groups
    assert np.max(np.abs(O.up_project(o, wv) - bad)) > 1e-3


# --------------------------------------------------------------------------
# rotary position embedding and the query projection
# --------------------------------------------------------------------------
def test_rope_rotation_matches_complex_multiplication():
    """Interleaved pairs as complex numbers times e^{i pos theta^(-2k/d)} (torch polar)."""
    g = np.random.default_rng(90)
    x = g.standard_normal((7, 3, 16))
    pos = g.integers(0, 200000, size=(7, 3))
    got = O.rope_rotate(x, pos, 10000.0)
    xc = torch.view_as_complex(torch.from_numpy(x.reshape(7, 3, 8, 2).copy()))
    freq = torch.tensor(10000.0, dtype=torch.float64) ** (-torch.arange(0, 16, 2, dtype=torch.float64) / 16)
    rot = torch.polar(torch.ones(7, 3, 8, dtype=torch.float64), torch.from_numpy(pos).double()[..., None] * freq)
    ref = torch.view_as_real(xc * rot).reshape(7, 3, 16).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_rope_rotation_invariants():
    g = np.random.default_rng(91)
    q, k = g.standard_normal((2, 32))
    # a rotation: norms (hence the RMS statistic) are preserved
    np.testing.assert_allclose(np.linalg.norm(O.rope_rotate(q, 1234, 500.0)), np.linalg.norm(q), rtol=1e-13)
    # position 0 is the identity
    np.testing.assert_allclose(O.rope_rotate(q, 0, 500.0), q, rtol=0, atol=0)
    # relative position: <R(m) q, R(n) k> depends on m - n only
    a = O.rope_rotate(q, 700, 500.0) @ O.rope_rotate(k, 300, 500.0)
    b = O.rope_rotate(q, 1400, 500.0) @ O.rope_rotate(k, 1000, 500.0)
    np.testing.assert_allclose(a, b, rtol=1e-10)
    # d = 2: one rotation by pos (theta^0 = 1)
    v = O.rope_rotate(np.array([1.0, 0.0]), 0.5, 10000.0)
    np.testing.assert_allclose(v, [math.cos(0.5), math.sin(0.5)], rtol=1e-15)


def test_mutation_rope_half_split_pairs_are_caught():
    """The other common convention pairs x_i with x_{i+d/2}; it is a different map."""
    g = np.random.default_rng(92)
    x = g.standard_normal(16)
    d = 16
    inv = 10000.0 ** (-np.arange(0, d, 2) / d)
    ang = 77 * inv
    half = np.concatenate([x[:8] * np.cos(ang) - x[8:] * np.sin(ang), x[:8] * np.sin(ang) + x[8:] * np.cos(ang)])
    assert np.max(np.abs(O.rope_rotate(x, 77, 10000.0) - half)) > 1e-3


def test_project_query_matches_torch_linear():
    g = np.random.default_rng(93)
    x = g.standard_normal((5, 48))
    w = g.standard_normal((4, 24 + 8, 48))
    pos = g.integers(0, 5000, size=5)
    q, qr = O.project_query(x, w, 24, pos, 10000.0)
    full = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(w.reshape(-1, 48))).reshape(5, 4, 32).numpy()
    np.testing.assert_allclose(q, full[..., :24], rtol=1e-13, atol=1e-13)
    for r in range(5):
        np.testing.assert_allclose(qr[r], O.rope_rotate(full[r, :, 24:], pos[r], 10000.0), rtol=1e-13, atol=1e-13)
