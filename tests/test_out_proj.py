"""The ssm_out projection (gdn_out_proj, tcgen05 GEMM) against the fp64
oracle's matrix product on the same bf16 inputs."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_02_gb300 import inputs as I
from oracle import oracle
from tests import gdn_testlib as tl

pytestmark = pytest.mark.gpu

DEV = "cuda"
# fp32 accumulation of exact bf16 products over K = 4096: relative error of
# order sqrt(4096) * 2^-24, far below this bound.
TOL = 1e-5


@pytest.fixture(scope="module")
def ops():
    from gated_deltanet_linear_02_gb300 import build, ops
    build.build()
    return ops


@pytest.fixture(scope="module")
def weight():
    return I.out_proj_weight(I.seed_of(9))


def run(ops, x, w, out_dtype):
    y = torch.empty(x.shape[0], I.N_EMBD, dtype=out_dtype, device=DEV)
    ops.out_proj(x.to(DEV), w.to(DEV), y)
    torch.cuda.synchronize()
    assert ops.device_error() == ops.GDN_OK
    return y.cpu()


def rows(M, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(M, I.D_INNER, generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("M", [1, 100, 128, 129, 256, 300, 1000])
def test_out_proj_matches_oracle(ops, weight, M):
    # one tile row, partial tiles, exact multiples and several tile rows
    x = rows(M, 900 + M)
    y = run(ops, x, weight, torch.float32)
    ref = oracle.out_proj(x, weight)
    e = tl.max_rel(y, ref)
    print(f"out_proj M={M}: {e:.2e}")
    assert e < TOL


def test_out_proj_prefill_size_bf16_output(ops, weight):
    # T = 4096 rows (the prefill length), bf16 output: rounding of 2^-8 on top
    x = rows(4096, 4096)
    y = run(ops, x, weight, torch.bfloat16)
    ref = oracle.out_proj(x, weight)
    e = tl.max_rel(y, ref)
    print(f"out_proj M=4096 bf16 out: {e:.2e}")
    assert e < TOL + tl.BF16_ROUND


def test_out_proj_of_the_mixer_output(ops, weight):
    # the projection of a real gated output (gdn_prefill, bf16 out) against the
    # oracle's projection of the same rows
    seed = I.seed_of(9, 1)
    lp = I.layer_params(seed)
    st = I.streams(seed, 200, torch.bfloat16)
    conv0, S0 = I.initial_states(seed, 1, torch.bfloat16)
    cu = I.cu_seqlens([200])
    out = torch.empty(200, I.D_INNER, dtype=torch.bfloat16, device=DEV)
    ops.prefill(lp.to(DEV), st.qkv.to(DEV), st.z.to(DEV), st.alpha.to(DEV), st.beta.to(DEV),
                cu.to(DEV), out, conv_state_in=conv0.to(DEV), ssm_state_in=S0.to(DEV))
    y = run(ops, out, weight, torch.float32)
    ref = oracle.out_proj(out.cpu(), weight)
    assert tl.max_rel(y, ref) < TOL
