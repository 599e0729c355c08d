"""Decode parity: the fused gdn_decode_step (and gdn_conv_step) against the
fp64 oracle on the same seeded inputs. Each decode step is one token of a
sequence, so B sequences over `steps` steps equal B oracle sequences of
length `steps`."""
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


def run_decode(ops, lp, st, conv0, S0, out_dtype, steps):
    """Runs `steps` decode steps on the GPU. Returns (outs [steps, B, 4096],
    conv, S) as CPU tensors; the inputs stay untouched."""
    lpd = lp.to(DEV)
    cp = ops.make_params(lpd)
    conv = conv0.to(DEV).clone()
    S = S0.to(DEV).clone()
    s = st.to(DEV)
    B = conv.shape[0]
    outs = torch.empty(steps, B, I.D_INNER, dtype=out_dtype, device=DEV)
    for t in range(steps):
        ops.decode_step(None, s.qkv[t], s.z[t], s.alpha[t], s.beta[t], conv, S, outs[t], cparams=cp)
    torch.cuda.synchronize()
    return outs.cpu(), conv.cpu(), S.cpu()


def oracle_decode(lp, st, conv0, S0, seqs=None):
    """The oracle over each sequence's `steps` tokens. st fields are [steps, B, ...]."""
    B = conv0.shape[0]
    seqs = list(range(B)) if seqs is None else list(seqs)
    P = tl.oparams(lp)
    qkv, z, al, be = (tl.f64(x) for x in (st.qkv, st.z, st.alpha, st.beta))
    c0, s0 = tl.f64(conv0), tl.to_page(tl.f64(S0))

    def one(b):
        from oracle import oracle
        return oracle.gdn_sequence(P, qkv[:, b], z[:, b], al[:, b], be[:, b], c0[b], s0[b])

    res = list(tl.pool().map(one, seqs))
    out = np.stack([r[0] for r in res], axis=1)          # [steps, len(seqs), 4096]
    return out, np.stack([r[1] for r in res]), tl.to_lib(np.stack([r[2] for r in res]))


def case(seed, B, steps, act, zero=False):
    lp = I.layer_params(seed)
    st = I.streams(seed, B, act, lead=(steps,))
    conv0, S0 = I.initial_states(seed, B, act, zero=zero)
    return lp, st, conv0, S0


def test_decode_fp32_T64_zero_state(ops):
    """64 single-token steps, fp32 activations, zero initial states, B=1 (the
    T=64 fp32 workload run through the decode entry point). Tolerance 1e-4."""
    lp, st, conv0, S0 = case(I.seed_of(0), 1, 64, torch.float32, zero=True)
    outs, conv, S = run_decode(ops, lp, st, conv0, S0, torch.float32, 64)
    ro, rc, rS = oracle_decode(lp, st, conv0, S0)
    e_out, e_S = tl.max_rel(outs, ro), tl.max_rel(S, rS)
    print(f"fp32 decode: out {e_out:.2e} (elem {tl.elem_rel(outs, ro):.2e}), state {e_S:.2e}")
    assert e_out < tl.TOL_F32 and e_S < tl.TOL_F32
    np.testing.assert_array_equal(tl.f64(conv), rc)


def test_decode_B64_128_steps_bf16(ops):
    """The batched-decode workload: B=64 sequences, 128 steps, bf16
    activations, fp32 state, random initial states. fp32 output for parity."""
    lp, st, conv0, S0 = case(I.seed_of(1), 64, 128, torch.bfloat16)
    outs, conv, S = run_decode(ops, lp, st, conv0, S0, torch.float32, 128)
    ro, rc, rS = oracle_decode(lp, st, conv0, S0)
    e_out, e_S = tl.max_rel(outs, ro), tl.max_rel(S, rS)
    print(f"bf16 decode B=64x128: out {e_out:.2e} (elem {tl.elem_rel(outs, ro):.2e}), state {e_S:.2e}")
    assert e_out < tl.TOL_BF16_OUT and e_S < tl.TOL_BF16_STATE
    np.testing.assert_array_equal(tl.f64(conv), rc)      # raw inputs: bit-exact


@pytest.mark.parametrize("act,out_dt", [(torch.float32, torch.bfloat16), (torch.bfloat16, torch.bfloat16),
                                        (torch.bfloat16, torch.float32)])
@pytest.mark.parametrize("B", [1, 3])
def test_decode_small_batches_and_dtypes(ops, act, out_dt, B):
    lp, st, conv0, S0 = case(777 + B, B, 5, act)
    outs, conv, S = run_decode(ops, lp, st, conv0, S0, out_dt, 5)
    ro, rc, rS = oracle_decode(lp, st, conv0, S0)
    tol_out = (tl.TOL_F32 if act == torch.float32 else tl.TOL_BF16_OUT) + \
        (tl.BF16_ROUND if out_dt == torch.bfloat16 else 0.0)
    tol_S = tl.TOL_F32 if act == torch.float32 else tl.TOL_BF16_STATE
    assert tl.max_rel(outs, ro) < tol_out
    assert tl.max_rel(S, rS) < tol_S
    np.testing.assert_array_equal(tl.f64(conv), rc)


def test_decode_GQA_pairs_share_conv_state(ops):
    """V-heads vh and vh+16 read the same q/k conv_state channels; after a step
    the shared rows must hold the shifted inputs exactly once (no double shift,
    no stale read). 8 steps with random conv_state make a wrong order visible."""
    lp, st, conv0, S0 = case(4242, 2, 8, torch.bfloat16)
    outs, conv, S = run_decode(ops, lp, st, conv0, S0, torch.float32, 8)
    ro, rc, rS = oracle_decode(lp, st, conv0, S0)
    np.testing.assert_array_equal(tl.f64(conv), rc)
    assert tl.max_rel(outs, ro) < tl.TOL_BF16_OUT


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
def test_conv_step(ops, act):
    from oracle import oracle
    B = 5
    lp = I.layer_params(55)
    st = I.streams(55, B, act)
    conv0, _ = I.initial_states(55, B, act)
    x = st.qkv.to(DEV)
    out = torch.empty_like(x)
    cs = conv0.to(DEV).clone()
    ops.conv_step(lp.conv_w.to(DEV), x, out, cs)
    torch.cuda.synchronize()
    for b in range(B):
        xh, nst = oracle.conv_token(tl.f64(st.qkv[b]), tl.f64(lp.conv_w), tl.f64(conv0[b]))
        tol = tl.TOL_F32 if act == torch.float32 else tl.BF16_ROUND
        assert tl.max_rel(out[b].cpu(), xh) < tol
        np.testing.assert_array_equal(tl.f64(cs[b].cpu()), nst)


def test_decode_30_layers_B256(ops):
    """Decode at scale: the 30 GDN layers of the 40-layer stack, each with its own
    seeded parameters and states, B=256, 32 steps, launched as the benchmark
    launches it (one gdn_decode_step per layer per step, bf16 activations).
    Sampled parity: every sequence of layers 0 and 29, eight seeded sequences of
    every other layer."""
    L, B, steps = 30, 256, 32
    gen = torch.Generator().manual_seed(3)
    checks = []
    for layer in range(L):
        seed = I.seed_of(3, layer)
        lp = I.layer_params(seed)
        lpd = lp.to(DEV)
        cp = ops.make_params(lpd)
        st = I.streams(seed, B, torch.bfloat16, device=DEV, lead=(steps,))
        conv, S = I.initial_states(seed, B, torch.bfloat16, device=DEV)
        seqs = list(range(B)) if layer in (0, L - 1) else sorted(torch.randperm(B, generator=gen)[:8].tolist())
        idx = torch.tensor(seqs, device=DEV)
        snap = (conv[idx].cpu(), S[idx].cpu())
        outs = torch.empty(steps, B, I.D_INNER, dtype=torch.float32, device=DEV)
        for t in range(steps):
            ops.decode_step(None, st.qkv[t], st.z[t], st.alpha[t], st.beta[t], conv, S, outs[t], cparams=cp)
        sub = I.Streams(st.qkv[:, idx].cpu(), st.z[:, idx].cpu(), st.alpha[:, idx].cpu(), st.beta[:, idx].cpu())
        checks.append((layer, lp, sub, snap, outs[:, idx].cpu(), conv[idx].cpu(), S[idx].cpu()))
        del st, conv, S, outs
    torch.cuda.synchronize()
    worst_o = worst_s = 0.0
    for layer, lp, sub, (c0, s0), o, c, s in checks:
        ro, rc, rS = oracle_decode(lp, sub, c0, s0)
        worst_o = max(worst_o, tl.max_rel(o, ro))
        worst_s = max(worst_s, tl.max_rel(s, rS))
        np.testing.assert_array_equal(tl.f64(c), rc)
    print(f"30-layer decode: worst out {worst_o:.2e}, worst state {worst_s:.2e}")
    assert worst_o < tl.TOL_BF16_OUT and worst_s < tl.TOL_BF16_STATE
