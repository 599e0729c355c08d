"""gdn_prefill_static: prefill for callers that cannot allocate device memory.

Some callers of this library may not allocate device memory at the point where
they run a prefill. Examples are a plugin inside a framework that owns every
allocation, and a serving loop that forbids allocation after start-up. They
cannot pass a workspace. gdn_prefill_static runs the same kernels with the
library's fixed 64 MiB device scratch instead.

These tests call it through the C ABI and check that it gives the same results
as gdn_prefill with a caller-provided workspace, within the parity tolerances
of the other tests, on two calls in a row. The second call runs on the first
call's leftover scratch contents. The tests also check that a prompt too long
for one window of the scratch runs in several windows, that a request the
scratch cannot hold is refused with a clear error after the argument checks,
and that a call allocates nothing.

The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_02_gb300 import inputs as I
from tests import gdn_testlib as tl

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ops():
    from gated_deltanet_linear_02_gb300 import build, ops
    build.build()
    return ops


def _case(seed, lengths, act):
    lp = I.layer_params(seed).to(DEV)
    st = I.streams(seed, int(sum(lengths)), act).to(DEV)
    conv0, S0 = I.initial_states(seed, len(lengths), act)
    return lp, st, I.cu_seqlens(lengths).to(DEV), conv0.to(DEV), S0.to(DEV)


def _outputs(T, N, act):
    return (torch.full((T, I.D_INNER), float("nan"), device=DEV),
            torch.full((N, I.KCONV - 1, I.C_CONV), float("nan"), dtype=act, device=DEV),
            torch.full((N, I.HV, I.DV, I.DK), float("nan"), device=DEV))


def _run(ops, fn, lp, st, cu, conv0, S0, chunk):
    T, N = st.qkv.shape[0], cu.shape[0] - 1
    out, cs, S = _outputs(T, N, st.qkv.dtype)
    fn(lp, st.qkv, st.z, st.alpha, st.beta, cu, out, conv_state_in=conv0, conv_state_out=cs, ssm_state_in=S0,
       ssm_state_out=S, chunk_size=chunk)
    assert ops.device_error() == ops.GDN_OK
    return out, cs, S


def _compare(ref, got, act):
    tol_o = tl.TOL_F32 if act == torch.float32 else tl.TOL_BF16_OUT
    tol_s = tl.TOL_F32 if act == torch.float32 else tl.TOL_BF16_STATE
    assert tl.max_rel(got[0], ref[0]) < tol_o
    assert tl.max_rel(got[2], ref[2]) < tol_s
    np.testing.assert_array_equal(got[1].float().cpu().numpy(), ref[1].float().cpu().numpy())


@pytest.mark.parametrize("act,chunk", [(torch.bfloat16, 0), (torch.float32, 1)])
def test_static_matches_workspace_entry_two_calls(ops, act, chunk):
    # two calls in a row with different sizes: the second runs on the first's leftover scratch
    for seed, lengths in ((4101, [300, 77]), (4102, [129, 5, 0, 64])):
        lp, st, cu, conv0, S0 = _case(seed, lengths, act)
        ref = _run(ops, ops.prefill, lp, st, cu, conv0, S0, chunk)
        got = _run(ops, ops.prefill_static, lp, st, cu, conv0, S0, chunk)
        torch.cuda.synchronize()
        _compare(ref, got, act)


def test_static_allocates_nothing(ops):
    lp, st, cu, conv0, S0 = _case(4103, [200, 3], torch.bfloat16)
    _run(ops, ops.prefill_static, lp, st, cu, conv0, S0, 0)     # set-up (first call on this device)
    torch.cuda.synchronize()
    out, cs, S = _outputs(st.qkv.shape[0], 2, torch.bfloat16)
    torch_before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    ops.prefill_static(lp, st.qkv, st.z, st.alpha, st.beta, cu, out, conv_state_in=conv0, conv_state_out=cs,
                       ssm_state_in=S0, ssm_state_out=S)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == torch_before
    assert free_after == free_before
    assert torch.isfinite(out).all()


def test_static_long_prompt_runs_in_windows(ops):
    # One bf16 sequence of 4096 tokens does not fit the 64 MiB scratch in one
    # window; the chunked form runs it as several windows with the state
    # carried, and gives what gdn_prefill gives with a full-size workspace.
    full = ops.prefill_workspace_size(1, 4096, torch.bfloat16, 0)
    assert full > ops.static_scratch_bytes()
    lp, st, cu, conv0, S0 = _case(4104, [4096], torch.bfloat16)
    ref = _run(ops, ops.prefill, lp, st, cu, conv0, S0, 0)
    got = _run(ops, ops.prefill_static, lp, st, cu, conv0, S0, 0)
    torch.cuda.synchronize()
    _compare(ref, got, torch.bfloat16)


def test_static_refuses_oversized_request(ops):
    # the exact scan keeps all of its tokens in scratch: 4096 fp32 tokens need
    # about 200 MB, more than the static scratch holds
    need = ops.prefill_workspace_size(1, 4096, torch.float32, 1)
    assert need > ops.static_scratch_bytes()
    lp, st, cu, conv0, S0 = _case(4105, [4096], torch.float32)
    out, cs, S = _outputs(4096, 1, torch.float32)
    with pytest.raises(ops.GdnError) as err:
        ops.prefill_static(lp, st.qkv, st.z, st.alpha, st.beta, cu, out, ssm_state_out=S, chunk_size=1)
    assert err.value.status == ops.GDN_ERR_WORKSPACE
    assert str(need) in str(err.value)
    torch.cuda.synchronize()
    assert torch.isnan(out).all()           # nothing was launched


def test_static_checks_arguments_before_scratch_size(ops):
    # A request that would not fit AND has a null tensor pointer reports the
    # invalid argument, as gdn_prefill does, not the scratch size.
    import ctypes
    lp, st, cu, conv0, S0 = _case(4106, [4096], torch.float32)
    out, cs, S = _outputs(4096, 1, torch.float32)
    cp = ops.make_params(lp)
    rc = ops.lib().gdn_prefill_static(ctypes.byref(cp), None, st.z.data_ptr(), st.alpha.data_ptr(),
                                      st.beta.data_ptr(), cu.data_ptr(), 1, 4096, None, None, None,
                                      S.data_ptr(), out.data_ptr(), ops.GDN_F32, ops.GDN_F32, 1, None)
    assert rc == ops.GDN_ERR_INVALID_ARG
