"""Failure path of the bounded waits, made on purpose without faulting the GPU.

QKMLA_FLAG_TEST_STALL makes the 64-row tensor-core decode kernel's loader stop
before its second tile and shortens every wait to 1 ms.  The consumers' waits
for that tile then run out: the kernel records QKMLA_ERR_TIMEOUT in the status
word and unwinds with nothing in flight (every tile it issued was consumed, no
matrix multiply is pending), so the context stays usable and the next, normal
call must match the oracle.
"""
import numpy as np
import pytest
import torch

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


def _np(t):
    return t.detach().float().cpu().numpy()


def test_expired_wait_reports_timeout_and_context_survives(Q):
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = W.small(W.WORKLOADS[1], 2, (1024, 3000))
    st = DeviceState(w)
    st.absorb()
    st.append_step()
    assert_status_ok(Q)
    a = st.decode_args()
    assert Q.decode_kernel_name(a) == "tcgen05"
    a.flags |= Q.FLAG_TEST_STALL
    Q.decode_raw(a)
    assert Q.get_device_status() == Q.ERR_TIMEOUT
    assert_status_ok(Q)                    # the read cleared the word; the stream still syncs
    st.decode()
    assert_status_ok(Q)
    o_ref, lse_ref = OR.reference(w)
    check_close(_np(st.o), o_ref, "bf16", "after timeout o")
    check_close(_np(st.lse), lse_ref, "bf16", "after timeout lse")


def test_stall_flag_is_refused_by_other_kernels(Q):
    """The hook lives in the 64-row kernel only: the CTA-pair and CUDA-core paths
    reject it before launching anything."""
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = W.small(W.WORKLOADS[2], 2, (128, 200))
    st = DeviceState(w)
    a = st.decode_args()
    a.flags |= Q.FLAG_TEST_STALL
    with pytest.raises(Q.QkmlaError) as e:
        Q.decode_raw(a)
    assert e.value.code == Q.ERR_UNSUPPORTED
    a = st.decode_args(force_simt=True)
    a.flags |= Q.FLAG_TEST_STALL
    with pytest.raises(Q.QkmlaError) as e:
        Q.decode_raw(a)
    assert e.value.code == Q.ERR_UNSUPPORTED
    assert_status_ok(Q)
