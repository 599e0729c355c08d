"""gdn_gated_out_proj -- the gated RMSNorm . silu(z) formed inside the ssm_out
GEMM -- against the fp64 oracle: oracle.gated_rmsnorm per (row, head), then
oracle.out_proj, on the same inputs.

Tolerance. The GEMM's A operand is the gated row rounded to bf16 (relative
error at most 2^-9 per element, independent across elements), and silu uses
the hardware tanh (absolute error about 2.5e-4 |z|). An output is a sum of
4096 such products with random signs, so its error is about 2^-9 / sqrt(3)
= 1.1e-3 of the sum's own scale; the largest error over all outputs against
the largest output stays near that ratio. 4e-3 bounds it with margin, and a
wrong head, a missing factor of the norm or a transposed operand gives
errors of order 1. fp32 accumulation adds about 1e-5.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_02_gb300 import inputs as I
from oracle import oracle
from tests import gdn_testlib as tl

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL_GATED = 4e-3


@pytest.fixture(scope="module")
def ops():
    from gated_deltanet_linear_02_gb300 import build, ops
    build.build()
    return ops


@pytest.fixture(scope="module")
def weight():
    return I.out_proj_weight(I.seed_of(9, 7))


def oracle_gated(y, z, norm_w, eps):
    """The gated output of section "Output path", per (row, head), in fp64."""
    y64, z64 = tl.f64(y), tl.f64(z)
    M = y64.shape[0]
    out = np.empty_like(y64)
    for m in range(M):
        for h in range(I.HV):
            sl = slice(h * I.DV, (h + 1) * I.DV)
            out[m, sl] = oracle.gated_rmsnorm(y64[m, sl], z64[m, sl], norm_w, eps)
    return out


def inputs(M, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    # y at the scale the mixer gives (|y| ~ 0.1 .. 1, heads of different scale)
    y = (torch.randn(M, I.D_INNER, generator=g) * (0.05 + torch.rand(M, I.HV, 1, generator=g)).repeat_interleave(
        I.DV, dim=2).reshape(M, I.D_INNER))
    z = torch.randn(M, I.D_INNER, generator=g) * 2.0
    return y.to(dtype), z.to(dtype)


def run(ops, y, z, norm_w, eps, w, out_dtype):
    out = torch.full((y.shape[0], I.N_EMBD), float("nan"), dtype=out_dtype, device=DEV)
    ops.gated_out_proj(norm_w.to(DEV), eps, y.to(DEV), z.to(DEV), w.to(DEV), out)
    torch.cuda.synchronize()
    assert ops.device_error() == ops.GDN_OK
    return out.cpu()


@pytest.mark.parametrize("M,act", [(1, torch.bfloat16), (100, torch.bfloat16), (256, torch.bfloat16),
                                   (300, torch.float32), (1000, torch.bfloat16), (2500, torch.bfloat16)])
def test_gated_out_proj_matches_oracle(ops, weight, M, act):
    # one row; a ragged single tile; the decode batch (split K over a cluster);
    # fp32 y and z; several tile rows; wide tiles (2500 rows: 512-column tiles)
    lp = I.layer_params(I.seed_of(9, 8))
    y, z = inputs(M, 7000 + M, act)
    got = run(ops, y, z, lp.norm_w, lp.norm_eps, weight, torch.float32)
    ref = oracle.out_proj(oracle_gated(y, z, lp.norm_w, lp.norm_eps), weight)
    e = tl.max_rel(got, ref)
    print(f"gated_out_proj M={M} {act}: {e:.2e}")
    assert e < TOL_GATED


def test_gated_out_proj_bf16_output_large(ops, weight):
    # 4096 rows, bf16 output: the prefill length, a rounding of 2^-8 on top.
    # Sampled rows (every 37th) against the oracle keep the check fast.
    M = 4096
    lp = I.layer_params(I.seed_of(9, 9))
    y, z = inputs(M, 7777, torch.bfloat16)
    got = run(ops, y, z, lp.norm_w, lp.norm_eps, weight, torch.bfloat16)
    rows = np.arange(0, M, 37)
    ref = oracle.out_proj(oracle_gated(y[rows], z[rows], lp.norm_w, lp.norm_eps), weight)
    e = tl.max_rel(got[rows], ref)
    print(f"gated_out_proj M=4096 bf16 out: {e:.2e}")
    assert e < TOL_GATED + tl.BF16_ROUND
    assert torch.isfinite(got.float()).all()


def test_gated_out_proj_zero_rows_and_scale(ops, weight):
    # A row of zeros gives 0 (the eps keeps the norm finite); a head scaled by
    # 1000 gives the same output as unscaled up to eps (the norm divides the
    # scale out), which a missing or misplaced norm factor would break.
    lp = I.layer_params(I.seed_of(9, 10))
    y, z = inputs(130, 7100, torch.float32)
    y[5] = 0.0
    y2 = y.clone()
    y2[:, 3 * I.DV:4 * I.DV] *= 1000.0
    a = run(ops, y, z, lp.norm_w, lp.norm_eps, weight, torch.float32)
    b = run(ops, y2, z, lp.norm_w, lp.norm_eps, weight, torch.float32)
    assert torch.count_nonzero(a[5]) == 0
    assert tl.max_rel(b, a) < TOL_GATED


def test_gated_out_proj_argument_checks(ops, weight):
    import ctypes
    lp = I.layer_params(I.seed_of(9, 11))
    y, z = inputs(8, 7200, torch.bfloat16)
    out = torch.empty(8, I.N_EMBD, device=DEV)
    L = ops.lib()
    args = [lp.norm_w.to(DEV).data_ptr(), ctypes.c_float(1e-6), y.to(DEV).data_ptr(), z.to(DEV).data_ptr(),
            weight.to(DEV).data_ptr(), out.data_ptr(), 8, ops.GDN_BF16, ops.GDN_F32, None]
    bad = list(args)
    bad[2] = None
    assert L.gdn_gated_out_proj(*bad) == ops.GDN_ERR_INVALID_ARG
    bad = list(args)
    bad[6] = -1
    assert L.gdn_gated_out_proj(*bad) == ops.GDN_ERR_INVALID_ARG
    bad = list(args)
    bad[7] = 7
    assert L.gdn_gated_out_proj(*bad) == ops.GDN_ERR_INVALID_ARG
    bad = list(args)
    bad[6] = 0
    assert L.gdn_gated_out_proj(*bad) == ops.GDN_OK          # M == 0: nothing to do


# ---------------------------------------------------------------------------
# The mixer with the norm left out (params.norm_w == NULL) writes y itself,
# and the fused projection applies the norm: together they must give the
# oracle's whole path, ssm_out . gated.

def _no_norm(lp):
    import dataclasses
    return dataclasses.replace(lp, norm_w=None)


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
def test_decode_step_without_norm_writes_y(ops, act):
    seed = I.seed_of(9, 20)
    lp = I.layer_params(seed)
    B = 6
    conv0, S0 = I.initial_states(seed, B, act)
    st = I.streams(seed, B, act)
    conv, S = conv0.to(DEV), S0.to(DEV)
    out = torch.empty(B, I.D_INNER, device=DEV)
    ops.decode_step(_no_norm(lp.to(DEV)), st.qkv.to(DEV), st.z.to(DEV), st.alpha.to(DEV), st.beta.to(DEV),
                    conv, S, out)
    torch.cuda.synchronize()
    assert ops.device_error() == ops.GDN_OK
    for b in range(B):
        ref = tl.oracle_y_sequence(lp, st.qkv[b:b + 1], st.alpha[b:b + 1], st.beta[b:b + 1], conv0[b], S0[b])
        e = tl.max_rel(out[b:b + 1].cpu(), ref)
        assert e < (tl.TOL_F32 if act == torch.float32 else tl.TOL_BF16_OUT), (b, e)


@pytest.mark.parametrize("act,chunk", [(torch.bfloat16, 64), (torch.float32, 1)])
def test_prefill_without_norm_writes_y(ops, act, chunk):
    # ragged lengths over several chunks; the chunked form and the exact scan
    seed = I.seed_of(9, 21)
    lp = I.layer_params(seed)
    lengths = [150, 7]
    conv0, S0 = I.initial_states(seed, len(lengths), act)
    st = I.streams(seed, sum(lengths), act)
    out = torch.empty(sum(lengths), I.D_INNER, device=DEV)
    ops.prefill(_no_norm(lp.to(DEV)), st.qkv.to(DEV), st.z.to(DEV), st.alpha.to(DEV), st.beta.to(DEV),
                I.cu_seqlens(lengths).to(DEV), out, conv_state_in=conv0.to(DEV), ssm_state_in=S0.to(DEV),
                chunk_size=chunk)
    torch.cuda.synchronize()
    assert ops.device_error() == ops.GDN_OK
    a = 0
    for n, L in enumerate(lengths):
        ref = tl.oracle_y_sequence(lp, st.qkv[a:a + L], st.alpha[a:a + L], st.beta[a:a + L], conv0[n], S0[n])
        e = tl.max_rel(out[a:a + L].cpu(), ref)
        print(f"prefill y chunk={chunk} seq {n}: {e:.2e}")
        assert e < (tl.TOL_F32 if act == torch.float32 else tl.TOL_BF16_OUT), (n, e)
        a += L


def test_decode_multi_without_norm_writes_y(ops):
    seed = I.seed_of(9, 22)
    lp = I.layer_params(seed)
    B, T = 4, 3
    conv0, S0 = I.initial_states(seed, B, torch.float32)
    st = I.streams(seed, T, torch.float32, lead=(B,))
    out = torch.empty(B, T, I.D_INNER, device=DEV)
    ops.decode_multi(_no_norm(lp.to(DEV)), st.qkv.to(DEV), st.z.to(DEV), st.alpha.to(DEV), st.beta.to(DEV),
                     conv0.to(DEV), S0.to(DEV), out)
    torch.cuda.synchronize()
    assert ops.device_error() == ops.GDN_OK
    for b in range(B):
        ref = tl.oracle_y_sequence(lp, st.qkv[b], st.alpha[b], st.beta[b], conv0[b], S0[b])
        assert tl.max_rel(out[b].cpu(), ref) < tl.TOL_F32


def test_fused_decode_step_end_to_end(ops, weight):
    # decode without the norm (bf16 y) then the fused projection, against the
    # oracle's gated output of the same token projected by the oracle. The bf16
    # rounding of y adds at most 2^-9 per element on top of the operand rounding.
    seed = I.seed_of(9, 23)
    lp = I.layer_params(seed)
    B = 64
    conv0, S0 = I.initial_states(seed, B, torch.bfloat16)
    st = I.streams(seed, B, torch.bfloat16)
    y = torch.empty(B, I.D_INNER, dtype=torch.bfloat16, device=DEV)
    ops.decode_step(_no_norm(lp.to(DEV)), st.qkv.to(DEV), st.z.to(DEV), st.alpha.to(DEV), st.beta.to(DEV),
                    conv0.to(DEV), S0.to(DEV), y)
    out = run(ops, y, st.z, lp.norm_w, lp.norm_eps, weight, torch.float32)
    P = tl.oparams(lp)
    gated = np.stack([oracle.gdn_sequence(P, st.qkv[b:b + 1], st.z[b:b + 1], st.alpha[b:b + 1], st.beta[b:b + 1],
                                          tl.f64(conv0[b]), tl.to_page(tl.f64(S0[b])))[0][0] for b in range(B)])
    e = tl.max_rel(out, oracle.out_proj(gated, weight))
    print(f"fused decode step: {e:.2e}")
    assert e < TOL_GATED + tl.BF16_ROUND


def test_fused_prefill_end_to_end(ops, weight):
    # the chunked prefill without the norm, then the fused projection, against
    # the oracle's sequence output projected by the oracle
    seed = I.seed_of(9, 24)
    lp = I.layer_params(seed)
    T = 200
    conv0, S0 = I.initial_states(seed, 1, torch.bfloat16)
    st = I.streams(seed, T, torch.bfloat16)
    y = torch.empty(T, I.D_INNER, dtype=torch.bfloat16, device=DEV)
    ops.prefill(_no_norm(lp.to(DEV)), st.qkv.to(DEV), st.z.to(DEV), st.alpha.to(DEV), st.beta.to(DEV),
                I.cu_seqlens([T]).to(DEV), y, conv_state_in=conv0.to(DEV), ssm_state_in=S0.to(DEV))
    out = run(ops, y, st.z, lp.norm_w, lp.norm_eps, weight, torch.float32)
    gated = oracle.gdn_sequence(tl.oparams(lp), st.qkv, st.z, st.alpha, st.beta, tl.f64(conv0[0]),
                                tl.to_page(tl.f64(S0[0])))[0]
    e = tl.max_rel(out, oracle.out_proj(gated, weight))
    print(f"fused prefill: {e:.2e}")
    assert e < TOL_GATED + tl.BF16_ROUND + tl.TOL_BF16_OUT
