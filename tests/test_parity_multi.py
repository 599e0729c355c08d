"""Multi-token decode parity: gdn_decode_multi (T consecutive tokens for each of
B sequences, one sweep over the states) against the fp64 oracle run over the
same T tokens of every sequence, and against T successive gdn_decode_step
calls on the GPU."""
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


def case(seed, B, T, act):
    lp = I.layer_params(seed)
    st = I.streams(seed, T, act, lead=(B,))           # [B][T][...]
    conv0, S0 = I.initial_states(seed, B, act)
    return lp, st, conv0, S0


def run_multi(ops, lp, st, conv0, S0, out_dtype):
    cp = ops.make_params(lp.to(DEV))
    conv = conv0.to(DEV).clone()
    S = S0.to(DEV).clone()
    s = st.to(DEV)
    B, T = s.qkv.shape[0], s.qkv.shape[1]
    out = torch.empty(B, T, I.D_INNER, dtype=out_dtype, device=DEV)
    ops.decode_multi(None, s.qkv, s.z, s.alpha, s.beta, conv, S, out, cparams=cp)
    torch.cuda.synchronize()
    assert ops.device_error() == ops.GDN_OK
    return out.cpu(), conv.cpu(), S.cpu()


def oracle_multi(lp, st, conv0, S0):
    """The oracle over each sequence's T tokens. st fields are [B, T, ...]."""
    B = conv0.shape[0]
    P = tl.oparams(lp)
    qkv, z, al, be = (tl.f64(x) for x in (st.qkv, st.z, st.alpha, st.beta))
    c0, s0 = tl.f64(conv0), tl.to_page(tl.f64(S0))

    def one(b):
        from oracle import oracle
        return oracle.gdn_sequence(P, qkv[b], z[b], al[b], be[b], c0[b], s0[b])

    res = list(tl.pool().map(one, range(B)))
    return (np.stack([r[0] for r in res]), np.stack([r[1] for r in res]),
            tl.to_lib(np.stack([r[2] for r in res])))


def check(out, conv, S, ref, act, label):
    ro, rc, rS = ref
    e_o, e_S = tl.max_rel(out, ro), tl.max_rel(S, rS)
    tol_o, tol_S = (tl.TOL_F32, tl.TOL_F32) if act == torch.float32 else (tl.TOL_BF16_OUT, tl.TOL_BF16_STATE)
    print(f"{label}: out {e_o:.2e} (elem {tl.elem_rel(out, ro):.2e}) state {e_S:.2e} (tol {tol_o:.1e}/{tol_S:.1e})")
    assert e_o < tol_o and e_S < tol_S
    # conv_state holds raw inputs: it must match exactly
    assert tl.max_rel(conv, rc) == 0.0


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_multi_matches_oracle(ops, act, T):
    lp, st, conv0, S0 = case(I.seed_of(7, T), 6, T, act)
    out, conv, S = run_multi(ops, lp, st, conv0, S0, torch.float32)
    check(out, conv, S, oracle_multi(lp, st, conv0, S0), act, f"decode_multi T={T} {act}")


def test_multi_many_items_per_cta(ops):
    # B=40 gives 640 items: every persistent CTA takes several, so the state
    # slots wrap around the ring and the next item's inputs are prefetched.
    lp, st, conv0, S0 = case(I.seed_of(7, 40), 40, 4, torch.bfloat16)
    out, conv, S = run_multi(ops, lp, st, conv0, S0, torch.float32)
    check(out, conv, S, oracle_multi(lp, st, conv0, S0), torch.bfloat16, "decode_multi B=40 T=4")


def test_multi_bf16_output(ops):
    lp, st, conv0, S0 = case(I.seed_of(7, 3), 8, 3, torch.bfloat16)
    out, conv, S = run_multi(ops, lp, st, conv0, S0, torch.bfloat16)
    ro, _, _ = oracle_multi(lp, st, conv0, S0)
    e = tl.max_rel(out, ro)
    print(f"decode_multi bf16 out: {e:.2e}")
    assert e < tl.TOL_BF16_OUT + tl.BF16_ROUND


@pytest.mark.parametrize("T", [2, 6])
def test_multi_equals_successive_decode_steps(ops, T):
    # The same tokens through T gdn_decode_step calls: only rounding order may differ.
    lp, st, conv0, S0 = case(I.seed_of(7, 100 + T), 12, T, torch.bfloat16)
    out_m, conv_m, S_m = run_multi(ops, lp, st, conv0, S0, torch.float32)
    cp = ops.make_params(lp.to(DEV))
    conv = conv0.to(DEV).clone()
    S = S0.to(DEV).clone()
    s = st.to(DEV)
    outs = torch.empty(12, T, I.D_INNER, dtype=torch.float32, device=DEV)
    for t in range(T):
        o = torch.empty(12, I.D_INNER, dtype=torch.float32, device=DEV)
        ops.decode_step(None, s.qkv[:, t].contiguous(), s.z[:, t].contiguous(), s.alpha[:, t].contiguous(),
                        s.beta[:, t].contiguous(), conv, S, o, cparams=cp)
        outs[:, t] = o
    torch.cuda.synchronize()
    e_o, e_S = tl.max_rel(out_m, outs.cpu()), tl.max_rel(S_m, S.cpu())
    print(f"decode_multi vs {T} decode steps: out {e_o:.2e} state {e_S:.2e}")
    assert e_o < 1e-5 and e_S < 1e-5
    assert torch.equal(conv_m, conv.cpu())


def test_multi_empty_batch_is_noop(ops):
    lp = I.layer_params(I.seed_of(7, 0))
    cp = ops.make_params(lp.to(DEV))
    x = torch.zeros(0, 2, I.C_CONV, dtype=torch.bfloat16, device=DEV)
    ops.decode_multi(None, x, torch.zeros(0, 2, I.D_INNER, dtype=torch.bfloat16, device=DEV),
                     torch.zeros(0, 2, I.HV, dtype=torch.bfloat16, device=DEV),
                     torch.zeros(0, 2, I.HV, dtype=torch.bfloat16, device=DEV),
                     torch.zeros(0, 3, I.C_CONV, dtype=torch.bfloat16, device=DEV),
                     torch.zeros(0, I.HV, I.DV, I.DK, dtype=torch.float32, device=DEV),
                     torch.zeros(0, 2, I.D_INNER, dtype=torch.float32, device=DEV), cparams=cp)
    torch.cuda.synchronize()


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [3, 8])
def test_multi_strong_decays(ops, act, T):
    # Large alpha gives g = -exp(A_log) softplus(alpha + dt_bias) from about -7
    # down to below -100, where exp(g) is 0 in fp32: the kernel's running decay
    # product crosses its renormalisation threshold after one or two tokens, or
    # meets a decay of exactly 0. Heads vh % 3 == 2 and every third token keep
    # the ordinary gates, so strong and weak decays alternate within a state.
    lp, st, conv0, S0 = case(I.seed_of(7, 200 + T), 5, T, act)
    al = st.alpha.float().clone()
    vh = torch.arange(I.HV)
    for t in range(T):
        if t % 3 == 2:
            continue
        al[:, t, vh % 3 == 0] = 8.0
        al[:, t, vh % 3 == 1] = 30.0
    st.alpha = al.to(act)
    out, conv, S = run_multi(ops, lp, st, conv0, S0, torch.float32)
    check(out, conv, S, oracle_multi(lp, st, conv0, S0), act, f"decode_multi strong decays T={T} {act}")


def test_multi_bench_launch_B256_T4_sampled(ops):
    # The benchmarked launch: B=256 sequences, T=4 tokens each, bf16 in and out
    # (27 items per persistent CTA). Every output and state is checked finite;
    # eight seeded sequences against the oracle.
    B, T = 256, 4
    lp, st, conv0, S0 = case(I.seed_of(3, 100), B, T, torch.bfloat16)
    out, conv, S = run_multi(ops, lp, st, conv0, S0, torch.bfloat16)
    assert torch.isfinite(out.float()).all() and torch.isfinite(S).all()
    seqs = sorted(set(int(x) for x in np.random.default_rng(41).choice(B, 8, replace=False)) | {0, B - 1})
    sel = torch.tensor(seqs)
    sub = I.Streams(st.qkv[sel], st.z[sel], st.alpha[sel], st.beta[sel])
    ref = oracle_multi(lp, sub, conv0[sel], S0[sel])
    ro, rc, rS = ref
    e_o, e_S = tl.max_rel(out[sel].float(), ro), tl.max_rel(S[sel], rS)
    print(f"decode_multi B=256 T=4 sampled {seqs}: out {e_o:.2e} state {e_S:.2e}")
    assert e_o < tl.TOL_BF16_OUT + tl.BF16_ROUND and e_S < tl.TOL_BF16_STATE
    assert tl.max_rel(conv[sel], rc) == 0.0


def test_multi_bitwise_repeatable(ops):
    # The slot ring, the last-warp refills and the bulk state stores change
    # which warp issues which copy from run to run, but no sum: two runs from
    # the same inputs agree bit for bit (40 sequences: several items per CTA).
    lp, st, conv0, S0 = case(I.seed_of(7, 300), 40, 5, torch.bfloat16)
    runs = [run_multi(ops, lp, st, conv0, S0, torch.bfloat16) for _ in range(2)]
    for a, b in zip(runs[0], runs[1]):
        assert torch.equal(a, b)
