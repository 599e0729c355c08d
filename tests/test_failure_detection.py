"""Failure detection on the GPU without a GPU fault.

Every pipelined kernel of libgdn waits on mbarriers through one bounded wait.
When a wait runs out, the kernel records GDN_ERR_TIMEOUT in a device error
word and returns normally. This test makes such a wait run out: a diagnostic
kernel waits on an mbarrier that nothing completes. It checks that the host
reads the status and that the context is still usable afterwards. Nothing
faults, traps or hangs: the wait gives up after 2 s.
"""
import time

import numpy as np
import pytest
import torch

from gated_deltanet_linear_02_gb300 import inputs as I
from oracle import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from gated_deltanet_linear_02_gb300 import build, ops
    build.build()
    return ops


def test_bounded_wait_reports_timeout_and_context_survives(ops):
    assert ops.device_error() == ops.GDN_OK              # nothing pending
    t0 = time.time()
    ops.selftest_wait_timeout()
    assert ops.device_error() == ops.GDN_ERR_TIMEOUT     # synchronises, reads, clears
    waited = time.time() - t0
    assert 1.5 < waited < 30.0, f"the bounded wait took {waited:.1f} s"
    assert ops.device_error() == ops.GDN_OK              # the word was cleared

    # the same query under its specified name and arguments (the workspace is not read)
    ops.selftest_wait_timeout()
    assert ops.lib().gdn_get_device_error(None, None) == ops.GDN_ERR_TIMEOUT
    assert ops.lib().gdn_get_device_error(None, None) == ops.GDN_OK

    # the context still runs the library's kernels correctly
    a = I.attn_inputs(31, 2, 200, [200, 50])
    d = a.to("cuda")
    out = torch.empty(2, 16, 256, device="cuda")
    ops.attn_decode(d.q, d.k_cache, d.v_cache, d.ctx_len, d.z, out)
    assert ops.device_error() == ops.GDN_OK
    ref = oracle.attn_decode(a.q, a.k_cache, a.v_cache, a.ctx_len.numpy(), a.z)
    assert np.abs(out.cpu().double().numpy() - ref).max() / np.abs(ref).max() < 3e-3
