"""GPU parity: every call of the CUDA path against the fp64 CPU oracle on the
same seeded inputs.

Tolerances (fixed for this method): bf16 cache with fp32 accumulation --
max-abs <= 2e-2 and relative L2 <= 5e-3 on o and lse; fp32 cache -- relative
L2 <= 1e-5 and |diff| <= 1e-5 * max(1, |ref|) element-wise.  Cache writes are
compared bit for bit where the operation is a pure cast.

Edge cases with very short sequences (a few to ~100 tokens, shorter than any
benchmark workload) keep the relative-L2 bound, and their max-abs bound is
taken relative to the output scale, 2e-2 * max(1, max|o_ref|): with few
tokens carrying the softmax mass, one outlier latent (x30) dominates o and
the bf16 rounding of q~ and P gives an absolute error proportional to it.

Plain MLA (the comparator without normalisation) is checked on inputs without
outlier tokens: its logits are unbounded, and with x30 outliers they reach
the hundreds, where any bf16 rounding of the query moves the softmax by more
than a fixed tolerance -- the instability the method removes.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import oracle.run as OR
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from qk_normed_latent_gb300 import build as B
    B.build()
    import qk_normed_latent_gb300 as Q
    return Q


def report_margin(what, max_abs, rel_l2, lim_abs, lim_rel):
    """Print a parity margin (and append it to $QKMLA_PARITY_LOG as a JSON line)."""
    print(f"PARITY {what}: max-abs {max_abs:.3e} (limit {lim_abs:.1e}), rel-L2 {rel_l2:.3e} (limit {lim_rel:.1e})")
    path = os.environ.get("QKMLA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"what": what, "max_abs": max_abs, "rel_l2": rel_l2, "lim_abs": lim_abs,
                                "lim_rel": lim_rel}) + "\n")


def check_close(got, ref, kind, what="", edge=False):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    d = np.abs(got - ref)
    rel_l2 = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    if kind == "f32":
        report_margin(what, float(np.max(d / np.maximum(1.0, np.abs(ref)))), float(rel_l2), 1e-5, 1e-5)
        assert rel_l2 <= 1e-5, f"{what}: rel-L2 {rel_l2:.3e}"
        worst = np.max(d / np.maximum(1.0, np.abs(ref)))
        assert worst <= 1e-5, f"{what}: elementwise {worst:.3e}"
    else:
        lim = 2e-2 * (max(1.0, float(np.abs(ref).max())) if edge else 1.0)
        report_margin(what, float(d.max()), float(rel_l2), lim, 5e-3)
        assert d.max() <= lim, f"{what}: max-abs {d.max():.3e} > {lim:.3e}"
        assert rel_l2 <= 5e-3, f"{what}: rel-L2 {rel_l2:.3e}"
    return float(d.max()), float(rel_l2)


def assert_status_ok(Q):
    """The library's device status word is clear; on a failed stream sync, name the CUDA error."""
    st = Q.get_device_status()
    if st == Q.ERR_CUDA:
        try:
            torch.cuda.synchronize()
            msg = "stream sync failed, context still usable"
        except Exception as e:                      # the sticky error of the context
            msg = f"{type(e).__name__}: {e}"
        raise AssertionError(f"device status QKMLA_ERR_CUDA ({msg})")
    assert st == 0, st


def _np(t):
    return t.detach().float().cpu().numpy()


# ---------------------------------------------------------------------------
# qkmla_absorb_query
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("widx", [0, 1, 2, 4])
@pytest.mark.parametrize("qt", ["f32", "bf16"])
@pytest.mark.parametrize("plain", [False, True])
def test_absorb_matches_oracle(Q, widx, qt, plain):
    w = W.WORKLOADS[widx]
    wk, gq, gk, _, _ = W.weights(w)
    q, _ = W.queries(w)
    q = q.reshape(w.rows, w.H, w.d_h)
    d = "cuda"
    dt = torch.float32 if qt == "f32" else torch.bfloat16
    qt_out = torch.empty((w.rows, w.H, w.d_c), dtype=dt, device=d)
    aq_out = torch.empty((w.rows, w.H), dtype=torch.float32, device=d)
    Q.absorb_query(torch.from_numpy(q).to(d), torch.from_numpy(gq).to(d), torch.from_numpy(gk).to(d),
                   torch.from_numpy(wk).to(d), w.eps, qt_out, aq_out, plain=plain)
    torch.cuda.synchronize()
    ref_qt, ref_aq = O.absorb_query(q, gq, gk, wk, w.eps, plain=plain)
    np.testing.assert_allclose(_np(aq_out), ref_aq, rtol=2e-6)
    g = _np(qt_out)
    # summation error of a length-d_h dot product is bounded relative to the sum
    # of |terms| (not to |result|): scale_n = sum_j |W_nj q'_j|, computed in fp64
    qa = np.abs(q.astype(np.float64)) * (1.0 if plain else np.abs(gq.astype(np.float64) * gk))
    wa = np.abs(wk.astype(np.float64))
    g_of = np.arange(w.H) // (w.H // w.G)
    scale = np.stack([qa[:, h, :] @ wa[g_of[h]].T for h in range(w.H)], axis=1)
    if qt == "f32":
        assert np.max(np.abs(g - ref_qt)) <= 1e-5 * max(1.0, np.abs(ref_qt).max())
    else:
        # one bf16 rounding (<= 2^-8 relative) on top of a GEMM accurate to 2^-15 of
        # sum|terms| (split-bf16 tensor cores keep ~2^-17; fp32 FMA ~2^-20)
        assert np.all(np.abs(g - ref_qt) <= 2.0 ** -8 * np.abs(ref_qt) + 2.0 ** -15 * scale)


# ---------------------------------------------------------------------------
# qkmla_append: layout and values
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cache", ["f32", "bf16"])
@pytest.mark.parametrize("plain", [False, True])
@pytest.mark.parametrize("widx", [1, 2])
def test_append_matches_oracle_bit_exact_layout(Q, cache, plain, widx):
    w = W.WORKLOADS[widx].with_(cache_dtype=cache)
    wk, _, _, _, grk = W.weights(w)
    grk = (1 + 0.1 * np.random.default_rng(5).standard_normal(w.d_r)).astype(np.float32)  # non-trivial gamma
    c, r = W.sequence(W.small(w, 1, (301,)), 0)
    num_slots = 1024
    rng = np.random.default_rng(7)
    slots = rng.choice(num_slots, size=301, replace=False).astype(np.int64)
    slots[::17] = -1                                          # skipped tokens
    d = "cuda"
    cdt = torch.float32 if cache == "f32" else torch.bfloat16
    kv = torch.empty((num_slots, w.d_c + w.d_r), dtype=cdt, device=d)
    ak = torch.empty((num_slots, w.G), dtype=torch.float32, device=d)
    from qk_normed_latent_gb300.pipeline import sentinel_fill
    sentinel_fill(kv)
    sentinel_fill(ak)
    kv0 = kv.clone()
    ak0 = ak.clone()
    Q.append(torch.from_numpy(c).to(d), torch.from_numpy(r).to(d), torch.from_numpy(wk).to(d),
             torch.from_numpy(grk).to(d), torch.from_numpy(slots).to(d), kv, ak, w.eps, plain=plain)
    assert_status_ok(Q)
    ch, rh, a = O.append_tokens(c, r, wk, grk, w.eps, cache, plain=plain)
    ok = slots >= 0
    kvh = kv.cpu()
    # latent: a pure cast -> bit-exact against the oracle's RNE cast
    lat = kvh[torch.from_numpy(slots[ok]), : w.d_c].float().numpy()
    np.testing.assert_array_equal(lat.astype(np.float64), ch[ok])
    # RoPE key: one rounding of an fp32 product -> within one cache ulp
    rope = kvh[torch.from_numpy(slots[ok]), w.d_c:].float().numpy()
    if cache == "bf16":
        assert np.all(np.abs(rope - rh[ok]) <= 2.0 ** -7 * np.abs(rh[ok]) + 1e-30)
    else:
        # fp32: the RMS statistic itself is an fp32 sum; a few ulps
        np.testing.assert_allclose(rope, rh[ok], rtol=2e-6, atol=1e-30)
    # alpha^k: fp32 GEMM + reduction vs fp64
    np.testing.assert_allclose(ak.cpu().numpy()[slots[ok]], a[ok], rtol=1e-5)
    # untouched slots keep their sentinel bits
    untouched = np.setdiff1d(np.arange(num_slots), slots[ok])
    iv = torch.int16 if cache == "bf16" else torch.int32
    assert torch.equal(kvh[untouched].view(iv), kv0.cpu()[untouched].view(iv))
    assert torch.equal(ak.cpu()[untouched].view(torch.int32), ak0.cpu()[untouched].view(torch.int32))


@pytest.mark.parametrize("widx", [1, 2])
def test_append_cluster_and_plain_kernels_agree(Q, widx):
    """A misaligned token buffer sends qkmla_append to its plain-load kernel.  The
    cache rows are pure casts and must match bit for bit.  The plain kernel forms
    each key element with one fp32 FMA chain over d_c; the cluster kernel adds
    per-slice chains (64 rows each) and reduces the sum of squares in another
    order, so alpha^k agrees to fp32 rounding."""
    w = W.WORKLOADS[widx]
    wk, _, _, _, grk = W.weights(w)
    c, r = W.sequence(W.small(w, 1, (77,)), 0)
    slots = torch.arange(77, dtype=torch.int64, device="cuda") * 3
    outs = []
    for shift in (0, 1):
        buf = torch.zeros(77 * w.d_c + 1, dtype=torch.float32, device="cuda")
        cn = buf[shift:shift + 77 * w.d_c].view(77, w.d_c)
        cn.copy_(torch.from_numpy(c))
        kv = torch.zeros((256, w.d_c + w.d_r), dtype=torch.bfloat16, device="cuda")
        ak = torch.zeros((256, w.G), dtype=torch.float32, device="cuda")
        Q.append(cn, torch.from_numpy(r).cuda(), torch.from_numpy(wk).cuda(), torch.from_numpy(grk).cuda(),
                 slots, kv, ak, w.eps)
        assert_status_ok(Q)
        outs.append((kv.view(torch.int16).cpu(), ak.cpu()))
    assert torch.equal(outs[0][0], outs[1][0])
    np.testing.assert_allclose(outs[0][1].numpy(), outs[1][1].numpy(), rtol=2e-6)


def test_append_out_of_range_slot_is_reported(Q):
    w = W.WORKLOADS[1]
    wk = torch.from_numpy(W.weights(w)[0]).cuda()
    kv = torch.zeros((128, w.d_c + w.d_r), dtype=torch.bfloat16, device="cuda")
    ak = torch.zeros((128, w.G), dtype=torch.float32, device="cuda")
    c = torch.randn(2, w.d_c, device="cuda")
    r = torch.randn(2, w.d_r, device="cuda")
    slots = torch.tensor([5, 128], dtype=torch.int64, device="cuda")
    Q.append(c, r, wk, None, slots, kv, ak, w.eps)
    assert Q.get_device_status() == Q.ERR_DEVICE_BOUNDS
    assert_status_ok(Q)            # cleared by the read
    assert torch.count_nonzero(kv[5]) > 0


# ---------------------------------------------------------------------------
# qkmla_decode end to end (absorb -> append -> decode) against the explicit definition
# ---------------------------------------------------------------------------
CASES = {
    "tiny_fp32": (0, None),
    "small_bf16_full": (1, None),
    "dsv3_B4_T4096": (2, dict(B=4, lens=(4096, 4096, 4096, 4096))),
    "dsv3_ragged": (2, dict(B=6, lens=(1, 63, 64, 65, 129, 3001))),
    "long_ctx_B1_T20000": (3, dict(B=1, lens=(20011,))),
    "mixed_sq2_ragged": (4, dict(B=6, lens=(2, 64, 65, 130, 777, 5000))),
    "mixed_sq2_B3": (4, dict(B=3, lens=(512, 4097, 20000))),
    "small_bf16_B3": (1, dict(B=3, lens=(1024, 1500, 8192))),
    "small_ragged": (1, dict(B=6, lens=(1, 63, 64, 65, 129, 3001))),
    # more than 128 sequences: the split plan comes from the scheduler kernel
    # instead of being computed inside the decode and combine kernels
    "small_B160_sched": (1, dict(B=160, lens=tuple(16 + (37 * i) % 600 for i in range(160)))),
    "dsv3_B136_sched": (2, dict(B=136, lens=tuple(64 + (53 * i) % 500 for i in range(136)))),
    # the same scheduler-kernel batches without outlier tokens, held to the absolute 2e-2 bound
    "small_B160_sched_clean": (1, dict(B=160, lens=tuple(16 + (37 * i) % 600 for i in range(160)),
                                       kw=dict(outlier_frac=0.0))),
    "dsv3_B136_sched_clean": (2, dict(B=136, lens=tuple(64 + (53 * i) % 500 for i in range(136)),
                                      kw=dict(outlier_frac=0.0))),
    # non-unit RoPE gammas (gamma_rope_q in decode, gamma_rope_k in append) on every decode kernel:
    # CUDA cores (fp32), the 64-row tensor-core kernel at d_c = 256 and 512, the CTA-pair kernel
    "tiny_fp32_grope": (0, dict(B=1, lens=(256,), kw=dict(rope_gamma_std=0.1))),
    "small_grope": (1, dict(B=3, lens=(1024, 1500, 8192), kw=dict(rope_gamma_std=0.1))),
    "dsv3_H64_grope": (2, dict(B=3, lens=(1000, 4096, 700), kw=dict(H=64, G=4, rope_gamma_std=0.1))),
    "dsv3_grope": (2, dict(B=4, lens=(4096, 1000, 640, 3000), kw=dict(rope_gamma_std=0.1))),
    "mixed_sq2_grope": (4, dict(B=3, lens=(600, 5000, 20000), kw=dict(rope_gamma_std=0.1))),
    # more query tokens per step (multi-token prediction, chunked prefill), causal within the step:
    # CTA-pair kernel, 64-row kernel and CUDA cores
    "dsv3_sq4": (4, dict(B=3, lens=(4, 700, 9000), kw=dict(s_q=4, n_append=4))),
    "dsv3_sq16": (4, dict(B=2, lens=(16, 3001), kw=dict(s_q=16, n_append=16))),
    "dsv3_sq16_clean": (4, dict(B=2, lens=(16, 3001), kw=dict(s_q=16, n_append=16, outlier_frac=0.0))),
    "small_sq8": (1, dict(B=3, lens=(8, 1000, 4100), kw=dict(s_q=8, n_append=8))),
    "tiny_fp32_sq8": (0, dict(B=2, lens=(9, 256), kw=dict(s_q=8, n_append=8))),
    # the 64-row kernel with 64 rows at d_c = 256 (P^T in its own stage slot): 64 heads of one
    # query token, and two query tokens of 32 heads packed into one CTA
    "small_H64": (1, dict(B=3, lens=(1024, 300, 5000), kw=dict(H=64))),
    "small_H32_sq2": (1, dict(B=3, lens=(700, 2, 4100), kw=dict(H=32, s_q=2, n_append=2))),
}
# sequences of 1-130 tokens (the larger-s_q cases include one of exactly s_q tokens, so its first
# query token sees one token)
EDGE = {"dsv3_ragged", "mixed_sq2_ragged", "small_ragged", "small_B160_sched", "dsv3_B136_sched",
        "dsv3_sq4", "dsv3_sq16", "small_sq8", "small_H32_sq2"}


def make_args_only(Q, w):
    """qkmla_decode arguments for workload w on empty (uninitialised) buffers: enough
    for the host-side planning calls, which read shapes and pointers only."""
    lens = W.seq_lens(w)
    ps, max_pages, num_slots, table = W.page_layout(w, lens)
    dt = torch.bfloat16 if w.cache_dtype == "bf16" else torch.float32
    d = "cuda"
    keep = dict(
        qt=torch.empty((w.B, w.s_q, w.H, w.d_c), dtype=dt, device=d),
        aq=torch.empty((w.B, w.s_q, w.H), dtype=torch.float32, device=d),
        qr=torch.empty((w.B, w.s_q, w.H, w.d_r), dtype=torch.float32, device=d),
        kv=torch.empty((num_slots, w.d_c + w.d_r), dtype=dt, device=d),
        ak=torch.empty((num_slots, w.G), dtype=torch.float32, device=d),
        sl=torch.from_numpy(lens.astype(np.int32)).to(d),
        pt=torch.from_numpy(table).to(d),
        o=torch.empty((w.B, w.s_q, w.H, w.d_c), dtype=torch.float32, device=d),
        lse=torch.empty((w.B, w.s_q, w.H), dtype=torch.float32, device=d))
    a = Q.make_decode_args(keep["qt"], keep["aq"], keep["qr"], None, keep["kv"], keep["ak"], keep["sl"],
                           keep["pt"], ps, max_pages, w.G, w.scale, w.eps, keep["o"], keep["lse"])
    a._keep = keep                    # the buffers live as long as the arguments
    return a


def _workload(name):
    widx, red = CASES[name]
    w = W.WORKLOADS[widx]
    if red:
        w = W.small(w, red["B"], red["lens"], **red.get("kw", {}))
    return w


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("plain", [False, True])
def test_decode_end_to_end_matches_oracle(Q, name, plain):
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = _workload(name)
    if plain:
        w = w.with_(outlier_frac=0.0)
    st = DeviceState(w, plain=plain)
    st.step()
    assert_status_ok(Q)
    o_ref, lse_ref = OR.reference(w, plain=plain)
    edge = name in EDGE
    check_close(_np(st.o), o_ref, w.cache_dtype, f"{name} o", edge)
    check_close(_np(st.lse), lse_ref, w.cache_dtype, f"{name} lse", edge)


@pytest.mark.parametrize("name", ["small_bf16_B3", "dsv3_B4_T4096", "mixed_sq2_B3", "dsv3_grope", "dsv3_H64_grope"])
def test_tensor_core_kernel_is_selected_and_agrees_with_simt(Q, name):
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = _workload(name)
    st = DeviceState(w)
    st.absorb()
    st.append_step()
    assert Q.decode_kernel_name(st.decode_args()) == "tcgen05"
    assert Q.decode_kernel_name(st.decode_args(force_simt=True)) == "simt"
    st.decode(force_simt=True)
    o_s, l_s = _np(st.o).copy(), _np(st.lse).copy()
    st.decode()
    assert_status_ok(Q)
    check_close(_np(st.o), o_s, "bf16", f"{name} tc-vs-simt o")
    check_close(_np(st.lse), l_s, "bf16", f"{name} tc-vs-simt lse")


@pytest.mark.parametrize("name,launches", [("small_bf16_B3", 2), ("dsv3_B4_T4096", 2), ("small_B160_sched", 3)])
def test_decode_launch_count(Q, name, launches):
    """Up to 128 sequences the decode and combine kernels plan the split themselves
    (two launches); larger batches add the scheduler kernel."""
    w = _workload(name)
    a = make_args_only(Q, w)
    assert Q.decode_kernel_name(a) == "tcgen05"
    assert Q.decode_launch_count(a) == launches


@pytest.mark.parametrize("name", ["dsv3_B4_T4096", "mixed_sq2_B3", "small_bf16_B3"])
def test_plain_with_outliers_rescales_agree_across_kernels(Q, name):
    """Plain MLA on x30-outlier data: unbounded logits make the running max move
    on different tiles for different rows, exercising every rescale path of the
    tensor-core kernel.  Both kernels see the same q~ and cache; they must agree
    (bf16 P vs fp32 P: relative L2 within 1e-2)."""
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = _workload(name)
    st = DeviceState(w, plain=True)
    st.absorb()
    st.append_step()
    for _ in range(3):                          # repeated launches on the same state
        st.decode()
    assert_status_ok(Q)
    o_tc, l_tc = _np(st.o).copy(), _np(st.lse).copy()
    st.decode(force_simt=True)
    o_s, l_s = _np(st.o), _np(st.lse)
    assert np.all(np.isfinite(o_tc)) and np.all(np.isfinite(l_tc))
    assert np.linalg.norm(o_tc - o_s) <= 1e-2 * np.linalg.norm(o_s)
    assert np.max(np.abs(l_tc - l_s)) <= 1e-2 * max(1.0, np.abs(l_s).max())


@pytest.mark.parametrize("splits", [1, 2, 5, 33])
@pytest.mark.parametrize("simt", [False, True])
def test_decode_split_counts_agree(Q, splits, simt):
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = _workload("dsv3_ragged")
    st = DeviceState(w)
    st.absorb()
    st.append_step()
    st.decode(num_splits=0, force_simt=simt)
    o_auto, l_auto = _np(st.o).copy(), _np(st.lse).copy()
    st.decode(num_splits=splits, force_simt=simt)
    assert_status_ok(Q)
    o_ref, lse_ref = OR.reference(w)
    check_close(_np(st.o), o_ref, "bf16", f"splits={splits} o", edge=True)
    check_close(_np(st.lse), lse_ref, "bf16", f"splits={splits} lse", edge=True)
    # different split counts change the reference maxima the bf16 P is rounded
    # against (tensor-core kernel) or only the fp32 summation order (CUDA cores)
    check_close(_np(st.o), o_auto, "bf16", f"splits={splits} vs auto o", edge=True)
    check_close(_np(st.lse), l_auto, "bf16", f"splits={splits} vs auto lse", edge=True)


@pytest.mark.parametrize("splits", [0, 2, 3])
def test_packed_query_tokens_mask_per_row(Q, splits):
    """The 64-row kernel packs two query tokens of the small shape (16 heads) into
    one CTA; a sequence of 65 tokens split at the 64-token tile boundary gives the
    first query token (length 64) no token in the second item, the second query
    token (length 65) one."""
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = W.small(W.WORKLOADS[1], 3, (65, 2, 700), s_q=2, n_append=2)
    st = DeviceState(w)
    st.step()
    st.decode(num_splits=splits)
    assert_status_ok(Q)
    o_ref, lse_ref = OR.reference(w)
    check_close(_np(st.o), o_ref, "bf16", f"packed s_q=2 splits={splits} o", edge=True)
    check_close(_np(st.lse), lse_ref, "bf16", f"packed s_q=2 splits={splits} lse", edge=True)


def test_decode_bad_page_id_is_reported_not_trapped(Q):
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = _workload("dsv3_ragged")
    st = DeviceState(w)
    st.step()
    assert_status_ok(Q)
    bad = st.page_table.clone()
    bad[5, 3] = 10 ** 6                     # outside [0, num_pages)
    st.page_table = bad
    st.args = None
    st.decode(force_simt=True)
    assert Q.get_device_status() == Q.ERR_DEVICE_BOUNDS
    st.decode()
    assert Q.get_device_status() == Q.ERR_DEVICE_BOUNDS
    # a length beyond the page table is reported too
    st.page_table = st.page_table.clone()
    st.page_table[5, 3] = 0
    st.seq_lens[1] = st.max_pages * st.page_size + 1
    st.decode()
    assert Q.get_device_status() == Q.ERR_DEVICE_BOUNDS


def test_decode_workspace_too_small_is_rejected(Q):
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = _workload("dsv3_B4_T4096")
    st = DeviceState(w)
    st.absorb()
    a = st.decode_args(num_splits=4)
    need = Q.decode_workspace_size(a)
    assert need > 0
    a.workspace_bytes = need - 1
    with pytest.raises(Q.QkmlaError) as e:
        Q.decode_raw(a)
    assert e.value.code == Q.ERR_WORKSPACE


# ---------------------------------------------------------------------------
# full-size workloads, in the bench's launch configuration: sampled sequences
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("widx,picks,heads", [
    (1, (0, 7, 15), None),
    (2, (0, 33, 63), None),
    (3, (2,), tuple(range(16, 32))),
    (4, "spread", tuple(range(0, 16)) + tuple(range(112, 128))),
])
def test_full_size_sampled_rows(Q, widx, picks, heads):
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = W.WORKLOADS[widx]
    st = DeviceState(w)
    st.step()
    assert_status_ok(Q)
    if picks == "spread":
        order = np.argsort(W.seq_lens(w))
        picks = (int(order[0]), int(order[len(order) // 2]), int(order[-1]))
    o_ref, lse_ref = OR.reference(w, seqs=picks, heads=heads)
    o = _np(st.o)[list(picks)]
    lse = _np(st.lse)[list(picks)]
    hsel = slice(None) if heads is None else list(heads)
    check_close(o[:, :, hsel], o_ref[:, :, hsel], w.cache_dtype, f"w{widx} o")
    check_close(lse[:, :, hsel], lse_ref[:, :, hsel], w.cache_dtype, f"w{widx} lse")
    # every output row is finite and lse is bounded by the normalised-logit bound
    assert np.all(np.isfinite(_np(st.o))) and np.all(np.isfinite(_np(st.lse)))


@pytest.mark.parametrize("widx", [1, 2])
def test_graph_replay_matches_direct_calls(Q, widx):
    """bench.py replays a CUDA graph of one step (absorb, append, decode call).  The
    graph holds the same kernels with the same arguments and the split plan is made
    on the device, so a replay must reproduce the direct calls bit for bit."""
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = W.WORKLOADS[widx]
    st = DeviceState(w)
    st.step()
    assert_status_ok(Q)
    o1, l1 = st.o.clone(), st.lse.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        st.step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    st.o.zero_()
    st.lse.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        st.absorb()
        st.append_step()
        Q.decode_raw(st.args)
    g.replay()
    torch.cuda.synchronize()
    assert_status_ok(Q)
    assert torch.equal(st.o, o1) and torch.equal(st.lse, l1)


# ---------------------------------------------------------------------------
# reduced-precision scalar cache: A^k_cache in fp16
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("widx", [1, 2])
def test_append_f16_alpha_is_the_rne_cast_of_the_fp32_alpha(Q, widx):
    """The fp16 A^k_cache holds the round-to-nearest-even cast of the fp32 alpha^k
    the same kernel writes to an fp32 cache (bit for bit); the latent and RoPE key
    rows do not change; untouched slots keep their sentinel bits."""
    from qk_normed_latent_gb300.pipeline import sentinel_fill
    w = W.WORKLOADS[widx]
    wk, _, _, _, grk = W.weights(w)
    c, r = W.sequence(W.small(w, 1, (203,)), 0)
    num_slots = 512
    slots = np.random.default_rng(8).choice(num_slots, size=203, replace=False).astype(np.int64)
    d = "cuda"
    outs = []
    for adt in (torch.float32, torch.float16):
        kv = torch.empty((num_slots, w.d_c + w.d_r), dtype=torch.bfloat16, device=d)
        ak = torch.empty((num_slots, w.G), dtype=adt, device=d)
        sentinel_fill(kv)
        sentinel_fill(ak)
        ak0 = ak.clone()
        Q.append(torch.from_numpy(c).to(d), torch.from_numpy(r).to(d), torch.from_numpy(wk).to(d),
                 torch.from_numpy(grk).to(d), torch.from_numpy(slots).to(d), kv, ak, w.eps)
        assert_status_ok(Q)
        outs.append((kv.cpu(), ak.cpu(), ak0.cpu()))
    (kv32, ak32, _), (kv16, ak16, ak16_0) = outs
    assert torch.equal(kv32.view(torch.int16), kv16.view(torch.int16))
    sl = torch.from_numpy(slots)
    assert torch.equal(ak16[sl].view(torch.int16), ak32[sl].to(torch.float16).view(torch.int16))
    untouched = torch.from_numpy(np.setdiff1d(np.arange(num_slots), slots))
    assert torch.equal(ak16[untouched].view(torch.int16), ak16_0[untouched].view(torch.int16))
    # and the oracle's fp16 alpha^k: within one fp16 rounding of the fp32 difference
    _, _, a_ref = O.append_tokens(c, r, wk, grk, w.eps, "bf16", alpha_dtype="f16")
    got = ak16[sl].float().numpy().astype(np.float64)
    assert np.all(np.abs(got - a_ref) <= 2.0 ** -10 * np.abs(a_ref))


ALPHA_CASES = {
    # CUDA cores (fp32 latent cache), 64-row tensor-core kernel (d_c = 256 and 512), CTA-pair kernel
    "tiny_fp32_af16": (0, dict(B=1, lens=(256,))),
    "small_af16": (1, dict(B=3, lens=(1024, 1500, 8192))),
    "dsv3_H64_af16": (2, dict(B=3, lens=(1000, 4096, 700), kw=dict(H=64, G=4))),
    "dsv3_af16": (2, dict(B=4, lens=(4096, 1000, 640, 3000))),
    "mixed_sq2_af16": (4, dict(B=3, lens=(600, 5000, 20000))),
}


@pytest.mark.parametrize("name", list(ALPHA_CASES))
def test_decode_f16_alpha_matches_oracle(Q, name):
    """fp16 alpha^k against the explicit definition (the cache dtype's tolerance)
    and against the absorbed form evaluated on the oracle's own fp16 scalar cache
    (fp32 latent cache: 1e-5, as the fp32 path; bf16: the bf16 tolerance)."""
    from qk_normed_latent_gb300.pipeline import DeviceState
    widx, red = ALPHA_CASES[name]
    w = W.small(W.WORKLOADS[widx], red["B"], red["lens"], alpha_dtype="f16", **red.get("kw", {}))
    st = DeviceState(w)
    assert st.ak.dtype == torch.float16
    st.step()
    assert_status_ok(Q)
    o_ref, lse_ref = OR.reference(w)
    kind_explicit = "bf16"        # fp16 alpha^k is a 2^-11 approximation of the explicit statistic
    check_close(_np(st.o), o_ref, kind_explicit, f"{name} o vs explicit")
    check_close(_np(st.lse), lse_ref, kind_explicit, f"{name} lse vs explicit")
    # the fp16 code of each alpha^k is decided from the kernel's fp32 value and from
    # the oracle's (fp64 -> fp32); they can fall on either side of a rounding tie,
    # so a code may differ by one fp16 step -- any other difference is an error
    lens = W.seq_lens(w)
    ps_, mp_, _, table = W.page_layout(w, lens)
    ak_gpu = st.ak.float().cpu().numpy().astype(np.float64)
    ties = 0
    for b in range(w.B):
        a_ref = OR.sequence_cache(w, b)[2]
        a_got = ak_gpu[W.slots_of(table, ps_, b, np.arange(int(lens[b])))]
        diff = a_got != a_ref
        ties += int(diff.sum())
        assert np.all(np.abs(a_got[diff] - a_ref[diff]) <= 2.0 ** -10 * np.abs(a_ref[diff]))
    o_abs, lse_abs = OR.reference_absorbed(w)
    kind_abs = w.cache_dtype if ties == 0 else "bf16"
    check_close(_np(st.o), o_abs, kind_abs, f"{name} o vs absorbed f16-alpha ({ties} tie codes)")
    check_close(_np(st.lse), lse_abs, kind_abs, f"{name} lse vs absorbed f16-alpha ({ties} tie codes)")
