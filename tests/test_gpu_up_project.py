"""qkmla_up_project against the oracle: the value up-projection of the latent
decode output, alone (random o, fp32 and bf16) and end to end after decode."""
import numpy as np
import pytest
import torch

import oracle as O
import oracle.run as OR
import workloads as W

from test_gpu_parity import assert_status_ok, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from qk_normed_latent_gb300 import build as B
    B.build()
    import qk_normed_latent_gb300 as Q
    return Q


@pytest.mark.parametrize("rows,H,G_v,d_c,d_v", [
    (5, 16, 4, 256, 64),          # the small model's heads, a ragged last tile
    (256, 128, 8, 512, 128),      # two query tokens x 128 sequences, DeepSeek-V3 shape
    (3, 8, 8, 128, 192),          # one matrix per head
    (70, 16, 2, 64, 256),
    (3, 192, 1, 128, 64),         # 192 heads a group: two head blocks, the threads store their rows
])
@pytest.mark.parametrize("o_dt", ["f32", "bf16"])
@pytest.mark.parametrize("out_dt", ["f32", "bf16"])
def test_up_project_matches_oracle(Q, rows, H, G_v, d_c, d_v, o_dt, out_dt):
    g = np.random.default_rng(rows * 7 + d_v)
    o = g.standard_normal((rows, H, d_c)).astype(np.float32)
    wv = (g.standard_normal((G_v, d_c, d_v)) / np.sqrt(d_c)).astype(np.float32)
    wv_b = O.bf16_rne(wv)                                    # the stored weights
    o_in = O.bf16_rne(o) if o_dt == "bf16" else o            # the stored output
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}
    o_d = torch.from_numpy(o).to("cuda").to(tdt[o_dt])
    w_d = torch.from_numpy(wv).to("cuda").to(torch.bfloat16)
    out = torch.empty((rows, H, d_v), dtype=tdt[out_dt], device="cuda")
    Q.up_project(o_d, w_d, out)
    assert_status_ok(Q)
    ref = O.up_project(o_in, wv_b)
    # fp32 accumulation of exact bf16 products (bf16 o), or of the hi/lo split of an
    # fp32 o (each part exact, the split leaves <= 2^-17 |o|): 2^-14 of sum |terms|
    scale = O.up_project(np.abs(o_in), np.abs(wv_b))
    got = out.float().cpu().numpy().astype(np.float64)
    lim = 2.0 ** -14 * scale + (2.0 ** -8 * np.abs(ref) if out_dt == "bf16" else 0.0)
    assert np.all(np.abs(got - ref) <= lim + 1e-30), float(np.max(np.abs(got - ref) - lim))


@pytest.mark.parametrize("widx,B,lens", [(1, 3, (1024, 1500, 8192)), (4, 3, (600, 5000, 20000))])
def test_decode_then_up_project_matches_oracle(Q, widx, B, lens):
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = W.small(W.WORKLOADS[widx], B, lens)
    st = DeviceState(w)
    st.step()
    assert_status_ok(Q)
    wv = W.value_weights(w)
    out = torch.empty((w.B, w.s_q, w.H, wv.shape[2]), dtype=torch.float32, device="cuda")
    Q.up_project(st.o, torch.from_numpy(wv).cuda().to(torch.bfloat16), out)
    assert_status_ok(Q)
    o_ref, _ = OR.reference(w)
    ref = O.up_project(o_ref, O.bf16_rne(wv))
    check_close(out.cpu().numpy(), ref, "bf16", f"w{widx} up-projected values")


def test_up_project_rejects_bad_shapes(Q):
    o = torch.zeros((2, 16, 100), device="cuda")                 # d_c % 64 != 0
    w = torch.zeros((4, 100, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((2, 16, 64), device="cuda")
    with pytest.raises(Q.QkmlaError) as e:
        Q.up_project(o, w, out)
    assert e.value.code == Q.ERR_UNSUPPORTED
    o = torch.zeros((2, 15, 128), device="cuda")                 # H % G_v != 0
    w = torch.zeros((4, 128, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((2, 15, 64), device="cuda")
    with pytest.raises(Q.QkmlaError) as e:
        Q.up_project(o, w, out)
    assert e.value.code == Q.ERR_INVALID
