"""The input projections (gdn_in_proj, one tcgen05 GEMM over the stacked
weight) against the fp64 oracle's four separate products."""
import pytest
import torch

from gated_deltanet_linear_02_gb300 import inputs as I
from oracle import oracle
from tests import gdn_testlib as tl

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = 1e-5          # fp32 accumulation of exact bf16 products over K = 2048


@pytest.fixture(scope="module")
def ops():
    from gated_deltanet_linear_02_gb300 import build, ops
    build.build()
    return ops


@pytest.fixture(scope="module")
def weights():
    return I.in_proj_weights(I.seed_of(9, 2))


def run(ops, h, weights, act):
    M = h.shape[0]
    w_in = torch.cat(weights, dim=0).to(DEV)
    outs = [torch.empty(M, n, dtype=act, device=DEV) for n in (I.C_CONV, I.D_INNER, I.HV, I.HV)]
    ops.in_proj(h.to(DEV), w_in, *outs)
    torch.cuda.synchronize()
    assert ops.device_error() == ops.GDN_OK
    return [o.cpu() for o in outs]


@pytest.mark.parametrize("M,act", [(1, torch.float32), (130, torch.float32), (1000, torch.bfloat16),
                                   (4096, torch.bfloat16)])
def test_in_proj_matches_oracle(ops, weights, M, act):
    g = torch.Generator().manual_seed(700 + M)
    h = torch.randn(M, I.N_EMBD, generator=g).to(torch.bfloat16)
    got = run(ops, h, weights, act)
    ref = oracle.in_proj(h, *weights)
    tol = TOL + (tl.BF16_ROUND if act == torch.bfloat16 else 0.0)
    for name, a, b in zip(("qkv", "z", "alpha", "beta"), got, ref):
        e = tl.max_rel(a, b)
        print(f"in_proj M={M} {name}: {e:.2e}")
        assert e < tol
