"""gdn_in_proj_conv (the input projections with the conv, SiLU and q/k L2 norms
in the GEMM's epilogue) and gdn_prefill_xhat (the chunked prefill from those
activations), against the fp64 oracle: oracle.in_proj, then the conv and the
norms per token from the oracle's single steps, and end to end oracle.in_proj
followed by oracle.gdn_sequence per sequence.

Tolerances.
- x^ is stored in fp16 (relative rounding 2^-11). SiLU uses the hardware tanh
  (absolute error about 2.5e-4 |u|). The projection accumulates in fp32 over
  K = 2048. Against max |x^| per head group that is below 1.5e-3; the bound is 2e-3.
- z, alpha, beta and conv_state_out are the projection rounded to bf16, so
  within 2^-8 relative of the largest value, plus 1e-5 for the accumulation.
- End to end, the mixer's output carries its own 3e-3 (bf16 activations). It
  also carries the bf16 rounding of z, which the oracle in fp64 does not have:
  2^-9 relative on z, times at most about 1.1 through silu near the largest
  outputs. The bound is 3e-3 + 2^-8. The state carries 1e-3.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_02_gb300 import inputs as I
from oracle import oracle
from tests import gdn_testlib as tl

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL_XHAT = 2e-3
TOL_PROJ = 2.0 ** -8 + 1e-5


@pytest.fixture(scope="module")
def ops():
    from gated_deltanet_linear_02_gb300 import build, ops
    build.build()
    return ops


@pytest.fixture(scope="module")
def weights():
    ws = I.in_proj_weights(I.seed_of(9, 30))
    return ws, torch.cat(ws, dim=0)


def hidden(M, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(M, I.N_EMBD, generator=g).to(torch.bfloat16)


def run_conv(ops, lp, h, w_in, lengths, cs_in):
    M, N = h.shape[0], len(lengths)
    xhat = torch.full((M, I.C_CONV), float("nan"), dtype=torch.float16, device=DEV)
    z = torch.empty(M, I.D_INNER, dtype=torch.bfloat16, device=DEV)
    al = torch.empty(M, I.HV, dtype=torch.bfloat16, device=DEV)
    be = torch.empty(M, I.HV, dtype=torch.bfloat16, device=DEV)
    cs_out = torch.full((N, I.KCONV - 1, I.C_CONV), float("nan"), dtype=torch.bfloat16, device=DEV)
    cu = I.cu_seqlens(lengths).to(DEV)
    ops.in_proj_conv(lp.to(DEV), h.to(DEV), w_in.to(DEV), cu, xhat, z, al, be,
                     conv_state_in=None if cs_in is None else cs_in.to(DEV), conv_state_out=cs_out)
    torch.cuda.synchronize()
    assert ops.device_error() == ops.GDN_OK
    return xhat.cpu(), z.cpu(), al.cpu(), be.cpu(), cs_out.cpu()


def oracle_xhat(lp, qkv, lengths, cs_in):
    """conv + SiLU per token from the oracle's conv step, then the q/k L2 norms."""
    conv_w = tl.f64(lp.conv_w)
    out = np.empty_like(qkv)
    cs_out = []
    a = 0
    for n, L in enumerate(lengths):
        st = np.zeros((I.KCONV - 1, I.C_CONV)) if cs_in is None else tl.f64(cs_in[n])
        for t in range(a, a + L):
            out[t], st = oracle.conv_token(qkv[t], conv_w, st)
            for hd in range(2 * I.HK):          # q heads, then k heads
                sl = slice(hd * I.DK, (hd + 1) * I.DK)
                out[t, sl] = oracle.l2norm(out[t, sl], lp.l2_eps)
        cs_out.append(st)
        a += L
    return out, np.stack(cs_out)


@pytest.mark.parametrize("lengths,with_state", [([300], True), ([130, 2, 0, 260, 1], True), ([126, 125], False)])
def test_in_proj_conv_matches_oracle(ops, weights, lengths, with_state):
    # several 125-row tiles with sequence starts inside them and at their edges,
    # a sequence shorter than the conv window, an empty one, with and without
    # conv_state_in
    (wq, wg, wa, wb), w_in = weights
    M = sum(lengths)
    seed = I.seed_of(9, 31) + M
    lp = I.layer_params(seed)
    h = hidden(M, seed)
    cs_in = I.initial_states(seed, len(lengths), torch.bfloat16)[0] if with_state else None
    xhat, z, al, be, cs_out = run_conv(ops, lp, h, w_in, lengths, cs_in)
    qkv, z_ref, a_ref, b_ref = oracle.in_proj(h, wq, wg, wa, wb)
    x_ref, cs_ref = oracle_xhat(lp, qkv, lengths, cs_in)
    e_q = tl.max_rel(xhat[:, :2048], x_ref[:, :2048])
    e_k = tl.max_rel(xhat[:, 2048:4096], x_ref[:, 2048:4096])
    e_v = tl.max_rel(xhat[:, 4096:], x_ref[:, 4096:])
    print(f"in_proj_conv {lengths}: q {e_q:.2e} k {e_k:.2e} v {e_v:.2e}")
    assert max(e_q, e_k, e_v) < TOL_XHAT
    assert tl.max_rel(z, z_ref) < TOL_PROJ
    assert tl.max_rel(al, a_ref) < TOL_PROJ
    assert tl.max_rel(be, b_ref) < TOL_PROJ
    assert tl.max_rel(cs_out, cs_ref) < TOL_PROJ


def test_in_proj_conv_rejects_overlapping_states(ops, weights):
    import ctypes
    _, w_in = weights
    lp = I.layer_params(I.seed_of(9, 32))
    cp = ops.make_params(lp.to(DEV))
    cs = torch.zeros(2, I.KCONV - 1, I.C_CONV, dtype=torch.bfloat16, device=DEV)
    h = hidden(8, 1).to(DEV)
    cu = I.cu_seqlens([4, 4]).to(DEV)
    xhat = torch.empty(8, I.C_CONV, dtype=torch.float16, device=DEV)
    z = torch.empty(8, I.D_INNER, dtype=torch.bfloat16, device=DEV)
    ab = torch.empty(8, I.HV, dtype=torch.bfloat16, device=DEV)
    rc = ops.lib().gdn_in_proj_conv(ctypes.byref(cp), h.data_ptr(), w_in.to(DEV).data_ptr(), cu.data_ptr(), 2, 8,
                                    cs.data_ptr(), cs.data_ptr(), xhat.data_ptr(), z.data_ptr(), ab.data_ptr(),
                                    ab.data_ptr(), None)
    assert rc == ops.GDN_ERR_INVALID_ARG


@pytest.mark.parametrize("lengths", [[200, 77], [700]])
def test_fused_projection_and_prefill_end_to_end(ops, weights, lengths):
    # h -> gdn_in_proj_conv -> gdn_prefill_xhat, against oracle.in_proj and
    # oracle.gdn_sequence per sequence from the same states
    (wq, wg, wa, wb), w_in = weights
    M, N = sum(lengths), len(lengths)
    seed = I.seed_of(9, 33) + M
    lp = I.layer_params(seed)
    h = hidden(M, seed)
    cs_in, S_in = I.initial_states(seed, N, torch.bfloat16)
    xhat, z, al, be, cs_out = (t.to(DEV) for t in run_conv(ops, lp, h, w_in, lengths, cs_in))
    out = torch.full((M, I.D_INNER), float("nan"), device=DEV)
    S_out = torch.full((N, I.HV, I.DV, I.DK), float("nan"), device=DEV)
    ops.prefill_xhat(lp.to(DEV), xhat, z, al, be, I.cu_seqlens(lengths).to(DEV), out, ssm_state_in=S_in.to(DEV),
                     ssm_state_out=S_out)
    torch.cuda.synchronize()
    assert ops.device_error() == ops.GDN_OK
    qkv, z_ref, a_ref, b_ref = oracle.in_proj(h, wq, wg, wa, wb)
    P = tl.oparams(lp)
    a = 0
    for n, L in enumerate(lengths):
        o_ref, cs_ref, S_ref = oracle.gdn_sequence(P, qkv[a:a + L], z_ref[a:a + L], a_ref[a:a + L], b_ref[a:a + L],
                                                   tl.f64(cs_in[n]), tl.to_page(tl.f64(S_in[n])))
        e_o = tl.max_rel(out[a:a + L].cpu(), o_ref)
        e_S = tl.max_rel(S_out[n].cpu(), tl.to_lib(S_ref))
        print(f"fused in_proj + prefill seq {n} (T={L}): out {e_o:.2e} state {e_S:.2e}")
        assert e_o < tl.TOL_BF16_OUT + tl.BF16_ROUND
        assert e_S < tl.TOL_BF16_STATE
        assert tl.max_rel(cs_out[n].cpu(), cs_ref) < TOL_PROJ
        a += L
