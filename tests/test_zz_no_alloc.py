"""qkmla_decode_noalloc: the decode entry point for callers that cannot
allocate device memory when they decode (an allocator-free serving runtime,
a plugin whose host owns every allocation).  It keeps its split-KV scratch in
a fixed per-device array inside the library instead of a caller workspace.

Checked here through the C ABI: two calls in a row give the same outputs as
qkmla_decode with a caller workspace (within the bf16 parity tolerance), and
arguments whose scratch would exceed the array are rejected.  This file is
collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

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


def _close(a, b):
    d = np.abs(a - b)
    assert d.max() <= 2e-2
    assert np.linalg.norm(a - b) <= 5e-3 * max(np.linalg.norm(b), 1e-30)


def _dirty_scratch(Q):
    """A no-alloc call of another shape first, so the shared array holds stale
    scheduler entries and partials when the checked calls run."""
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = W.small(W.WORKLOADS[1], 5, (700, 64, 9000, 3000, 131))
    st = DeviceState(w)
    st.absorb()
    st.append_step()
    a = st.decode_args(num_splits=7)
    rc = Q.lib().qkmla_decode_noalloc(ctypes.byref(a), Q._stream(None))
    assert rc == Q.OK, Q.status_string(rc)
    assert Q.get_device_status() == 0


@pytest.mark.parametrize("name,widx,lens,splits", [
    ("dsv3_B4", 2, (4096, 1000, 20000, 64), 0),
    ("small_B3", 1, (1024, 5000, 8192), 0),
    # more than 128 sequences: the scheduler kernel's items and split lists live in the array too
    ("small_B160_sched", 1, tuple(16 + (37 * i) % 600 for i in range(160)), 0),
    # the CUDA-core kernel's split partials (fp32 latent cache)
    ("tiny_fp32_split", 0, (256, 77), 4),
])
def test_noalloc_matches_workspace_entry_point_twice(Q, name, widx, lens, splits):
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = W.small(W.WORKLOADS[widx], len(lens), lens)
    st = DeviceState(w)
    st.absorb()
    st.append_step()
    st.decode(num_splits=splits)                  # existing entry point, torch workspace
    assert Q.get_device_status() == 0
    o_ref = st.o.float().cpu().numpy().copy()
    l_ref = st.lse.cpu().numpy().copy()
    assert Q.decode_workspace_size(st.args) > 0   # this case does use scratch
    _dirty_scratch(Q)
    for _ in range(2):
        st.o.fill_(float("nan"))
        st.lse.fill_(float("nan"))
        a = st.decode_args(num_splits=splits)
        a.workspace, a.workspace_bytes = None, 0  # ignored by the no-alloc entry point
        rc = Q.lib().qkmla_decode_noalloc(ctypes.byref(a), Q._stream(None))
        assert rc == Q.OK, Q.status_string(rc)
        assert Q.get_device_status() == 0
        _close(st.o.float().cpu().numpy(), o_ref)
        _close(st.lse.cpu().numpy(), l_ref)


def test_noalloc_rejects_scratch_beyond_its_limit(Q):
    from qk_normed_latent_gb300.pipeline import DeviceState
    w = W.small(W.WORKLOADS[2], 4, (64, 64, 64, 64))
    st = DeviceState(w)
    a = st.decode_args(num_splits=256)
    assert Q.decode_workspace_size(a) > Q.lib().qkmla_decode_noalloc_max_workspace()
    assert Q.lib().qkmla_decode_noalloc(ctypes.byref(a), Q._stream(None)) == Q.ERR_WORKSPACE
