"""The steps ahead of the decode path against the oracle: the query projection
with its RoPE rotation (qkmla_project_query), the RoPE-rotating append
(qkmla_append_rope), and the whole chain x -> project -> absorb -> append ->
decode against the explicit definition."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

from test_gpu_parity import assert_status_ok, check_close

pytestmark = pytest.mark.gpu
THETA = 10000.0


@pytest.fixture(scope="module")
def Q():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from qk_normed_latent_gb300 import build as B
    B.build()
    import qk_normed_latent_gb300 as Q
    return Q


@pytest.mark.parametrize("rows,d_x,H,d_h,d_r", [
    (256, 1536, 128, 128, 64),    # two query tokens x 128 sequences, DeepSeek-V3 shape
    (5, 256, 16, 64, 32),         # the small model, a ragged row tile
    (130, 512, 8, 128, 0),        # no RoPE block
    (7, 128, 4, 80, 16),          # d_h not a multiple of 32: the threads store their rows
])
def test_project_query_matches_oracle(Q, rows, d_x, H, d_h, d_r):
    g = np.random.default_rng(rows + d_x)
    x = O.bf16_rne(g.standard_normal((rows, d_x)))                       # the stored operands
    wq = O.bf16_rne(g.standard_normal((H, d_h + d_r, d_x)) / np.sqrt(d_x))
    pos = g.integers(0, 1 << 18, size=rows).astype(np.int32)
    pos[:3] = [0, 1, (1 << 18) - 1]
    d = "cuda"
    q = torch.empty((rows, H, d_h), dtype=torch.float32, device=d)
    qr = torch.empty((rows, H, d_r), dtype=torch.float32, device=d) if d_r else None
    Q.project_query(torch.from_numpy(x).to(d).to(torch.bfloat16), torch.from_numpy(wq).to(d).to(torch.bfloat16),
                    torch.from_numpy(pos).to(d), THETA, q, qr)
    assert_status_ok(Q)
    q_ref, qr_ref = O.project_query(x, wq, d_h, pos, THETA)
    # fp32 accumulation of exact bf16 products: 2^-16 of sum |terms|
    terms = np.einsum("rk,hjk->rhj", np.abs(x), np.abs(wq))
    got = q.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - q_ref) <= 2.0 ** -16 * terms[..., :d_h] + 1e-30)
    if d_r:
        # + the rotation with fp32 cos/sin of an exactly reduced angle: 2^-20 of the pair's norm
        tp = terms[..., d_h:]
        pair_terms = np.repeat(tp[..., 0::2] + tp[..., 1::2], 2, axis=-1)
        pair_norm = np.repeat(np.hypot(qr_ref[..., 0::2], qr_ref[..., 1::2]), 2, axis=-1)
        gotr = qr.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(gotr - qr_ref) <= 2.0 ** -16 * pair_terms + 2.0 ** -20 * pair_norm + 1e-30)


@pytest.mark.parametrize("widx", [1, 2])
@pytest.mark.parametrize("shift", [0, 1])          # 1: a misaligned token buffer takes the plain-load kernel
def test_append_rope_matches_oracle(Q, widx, shift):
    w = W.WORKLOADS[widx]
    wk, _, _, _, grk = W.weights(w)
    grk = (1 + 0.1 * np.random.default_rng(5).standard_normal(w.d_r)).astype(np.float32)
    c, r = W.sequence(W.small(w, 1, (301,)), 0)
    pos = np.random.default_rng(6).integers(0, 1 << 18, size=301).astype(np.int32)
    num_slots = 1024
    slots = np.random.default_rng(7).choice(num_slots, size=301, replace=False).astype(np.int64)
    d = "cuda"
    kv = torch.zeros((num_slots, w.d_c + w.d_r), dtype=torch.bfloat16, device=d)
    ak = torch.zeros((num_slots, w.G), dtype=torch.float32, device=d)
    buf = torch.zeros(301 * w.d_c + 1, dtype=torch.float32, device=d)
    cn = buf[shift:shift + 301 * w.d_c].view(301, w.d_c)
    cn.copy_(torch.from_numpy(c))
    Q.append_rope(cn, torch.from_numpy(r).to(d), torch.from_numpy(pos).to(d), THETA, torch.from_numpy(wk).to(d),
                  torch.from_numpy(grk).to(d), torch.from_numpy(slots).to(d), kv, ak, w.eps)
    assert_status_ok(Q)
    ch, rh, a = O.append_tokens(c, O.rope_rotate(r, pos, THETA), wk, grk, w.eps, "bf16")
    kvh = kv.cpu()
    sl = torch.from_numpy(slots)
    np.testing.assert_array_equal(kvh[sl, :w.d_c].float().numpy().astype(np.float64), ch)
    rope = kvh[sl, w.d_c:].float().numpy().astype(np.float64)
    # one bf16 step of the larger of the two values, plus the fp32 rotation's error,
    # which is relative to the pair's norm (a rotated element can cancel to ~0)
    pair = np.repeat(np.hypot(rh[:, 0::2], rh[:, 1::2]), 2, axis=1)
    err = np.abs(rope - rh)
    lim = 2.0 ** -7 * np.maximum(np.abs(rope), np.abs(rh)) + 2.0 ** -18 * pair
    assert np.all(err <= lim + 1e-30), (float(np.max(err - lim)), int(np.sum(err > lim)))
    np.testing.assert_allclose(ak.cpu().numpy()[slots], a, rtol=1e-5)


@pytest.mark.parametrize("widx,lens,d_x", [(1, (1024, 1500, 8192), 256), (4, (600, 5000, 20000), 1536)])
def test_decode_from_layer_input_matches_oracle(Q, widx, lens, d_x):
    """x -> qkmla_project_query -> qkmla_absorb_query; cache by qkmla_append_rope at
    the tokens' positions; qkmla_decode -- against the explicit definition on the
    oracle's projection and rotation of the same inputs."""
    w = W.small(W.WORKLOADS[widx], len(lens), lens, rope_gamma_std=0.1)
    lens_a = W.seq_lens(w)
    ps, max_pages, num_slots, table = W.page_layout(w, lens_a)
    wk, gq, gk, grq, grk = W.weights(w)
    x, wq = W.query_inputs(w, d_x)
    x_b, wq_b = O.bf16_rne(x), O.bf16_rne(wq)
    d = "cuda"
    kv = torch.zeros((num_slots, w.d_c + w.d_r), dtype=torch.bfloat16, device=d)
    ak = torch.zeros((num_slots, w.G), dtype=torch.float32, device=d)
    wk_d, grk_d = torch.from_numpy(wk).to(d), torch.from_numpy(grk).to(d)
    seqs = []
    for b in range(w.B):
        c, r = W.sequence(w, b)
        L = c.shape[0]
        pos = np.arange(L, dtype=np.int32)
        slots = W.slots_of(table, ps, b, pos)
        Q.append_rope(torch.from_numpy(c).to(d), torch.from_numpy(r).to(d), torch.from_numpy(pos).to(d), THETA, wk_d,
                      grk_d, torch.from_numpy(slots).to(d), kv, ak, w.eps)
        seqs.append((O.cache_cast(c, "bf16"), O.rope_key(O.rope_rotate(r, pos, THETA), grk, w.eps, "bf16")))
    rows = w.B * w.s_q
    qpos = np.array([int(lens_a[b]) - w.s_q + i for b in range(w.B) for i in range(w.s_q)], dtype=np.int32)
    q = torch.empty((rows, w.H, w.d_h), dtype=torch.float32, device=d)
    qr = torch.empty((w.B, w.s_q, w.H, w.d_r), dtype=torch.float32, device=d)
    Q.project_query(torch.from_numpy(x.reshape(rows, d_x)).to(d).to(torch.bfloat16),
                    torch.from_numpy(wq).to(d).to(torch.bfloat16), torch.from_numpy(qpos).to(d), THETA, q,
                    qr.view(rows, w.H, w.d_r))
    qt = torch.empty((w.B, w.s_q, w.H, w.d_c), dtype=torch.bfloat16, device=d)
    aq = torch.empty((w.B, w.s_q, w.H), dtype=torch.float32, device=d)
    Q.absorb_query(q, torch.from_numpy(gq).to(d), torch.from_numpy(gk).to(d), wk_d, w.eps, qt.view(rows, w.H, w.d_c),
                   aq.view(rows, w.H))
    o = torch.empty((w.B, w.s_q, w.H, w.d_c), dtype=torch.float32, device=d)
    lse = torch.empty((w.B, w.s_q, w.H), dtype=torch.float32, device=d)
    Q.decode(qt, aq, qr, torch.from_numpy(grq).to(d), kv, ak, torch.from_numpy(lens_a.astype(np.int32)).to(d),
             torch.from_numpy(table).to(d), ps, max_pages, w.G, w.scale, w.eps, o, lse)
    assert_status_ok(Q)
    q_o, qr_o = O.project_query(x_b.reshape(rows, d_x), wq_b, w.d_h, qpos, THETA)
    o_ref, lse_ref = O.decode_explicit(q_o.reshape(w.B, w.s_q, w.H, w.d_h), qr_o.reshape(w.B, w.s_q, w.H, w.d_r),
                                       gq, gk, grq, wk, seqs, w.s_q, w.scale, w.eps)
    check_close(o.cpu().numpy(), o_ref, "bf16", f"w{widx} from x o")
    check_close(lse.cpu().numpy(), lse_ref, "bf16", f"w{widx} from x lse")
