"""Prefill parity: gdn_prefill (packed varlen, state in/out) against the fp64
oracle on the same seeded inputs, for the exact scan (chunk_size 1) and the
library's default choice for each activation dtype."""
import math

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


def gpu_prefill(ops, lp, st, lengths, conv0, S0, out_dtype, chunk, pass_states=True, alias=False, ws_tokens=None):
    cu = I.cu_seqlens(lengths).to(DEV)
    N, T = len(lengths), int(sum(lengths))
    s = st.to(DEV)
    out = torch.full((T, I.D_INNER), float("nan"), dtype=out_dtype, device=DEV)
    cin = conv0.to(DEV).clone() if (pass_states and conv0 is not None) else None
    sin = S0.to(DEV).clone() if (pass_states and S0 is not None) else None
    if alias:
        cout, sout = cin, sin
    else:
        cout = torch.full((N, I.KCONV - 1, I.C_CONV), float("nan"), dtype=st.qkv.dtype, device=DEV)
        sout = torch.full((N, I.HV, I.DV, I.DK), float("nan"), dtype=torch.float32, device=DEV)
    ws = None
    if ws_tokens is not None:   # a workspace sized for windows of ws_tokens tokens
        ws = torch.empty(ops.prefill_workspace_size(N, ws_tokens, st.qkv.dtype, chunk), dtype=torch.uint8, device=DEV)
    ws = ops.prefill(lp.to(DEV), s.qkv, s.z, s.alpha, s.beta, cu, out, conv_state_in=cin, conv_state_out=cout,
                     ssm_state_in=sin, ssm_state_out=sout, chunk_size=chunk, workspace=ws)
    assert ops.device_error() == ops.GDN_OK
    return out.cpu(), cout.cpu(), sout.cpu()


def tol_for(act, out_dt):
    t_out = tl.TOL_F32 if act == torch.float32 else tl.TOL_BF16_OUT
    t_S = tl.TOL_F32 if act == torch.float32 else tl.TOL_BF16_STATE
    if out_dt == torch.bfloat16:
        t_out += tl.BF16_ROUND
    return t_out, t_S


def check(name, got, ref, act, out_dt, heads=None):
    (o, c, S), (ro, rc, rS) = got, ref
    if heads is not None:
        cols = np.concatenate([np.arange(h * 128, (h + 1) * 128) for h in heads])
        o, ro = tl.f64(o)[:, cols], ro[:, cols]
        S, rS = tl.f64(S)[:, heads], rS[:, heads]
    t_out, t_S = tol_for(act, out_dt)
    e_o, e_S = tl.max_rel(o, ro), tl.max_rel(S, rS)
    print(f"{name}: out {e_o:.2e} (elem {tl.elem_rel(o, ro):.2e}) state {e_S:.2e} (tol {t_out:.1e}/{t_S:.1e})")
    assert e_o < t_out, f"{name}: output error {e_o:.3e} >= {t_out:.1e}"
    assert e_S < t_S, f"{name}: state error {e_S:.3e} >= {t_S:.1e}"
    np.testing.assert_array_equal(tl.f64(c), rc)


def varlen_case(seed, lengths, act, zero=False):
    lp = I.layer_params(seed)
    st = I.streams(seed, int(sum(lengths)), act)
    conv0, S0 = I.initial_states(seed, len(lengths), act, zero=zero)
    return lp, st, conv0, S0


def oracle_varlen(lp, st, lengths, conv0, S0, heads=None):
    cu = I.cu_seqlens(lengths).tolist()
    if heads is None:
        return tl.oracle_sequences(lp, st.qkv, st.z, st.alpha, st.beta, cu, conv0, S0)
    ro = np.zeros((int(sum(lengths)), I.D_INNER))
    rS = tl.f64(S0).copy()
    rc = None
    for h in heads:
        o, rc, s = tl.oracle_sequences(lp, st.qkv, st.z, st.alpha, st.beta, cu, conv0, S0, heads=(h, h + 1))
        ro[:, h * 128:(h + 1) * 128] = o[:, h * 128:(h + 1) * 128]
        rS[:, h] = s[:, h]
    return ro, rc, rS


def test_prefill_T64_fp32(ops):
    """The T=64 fp32 workload: batch 1, zero initial states (passed as NULL),
    exact scan. Tolerance 1e-4."""
    lp, st, conv0, S0 = varlen_case(I.seed_of(0), [64], torch.float32, zero=True)
    got = gpu_prefill(ops, lp, st, [64], conv0, S0, torch.float32, chunk=0, pass_states=False)
    ref = oracle_varlen(lp, st, [64], conv0, S0)
    check("prefill T64 fp32", got, ref, torch.float32, torch.float32)


def test_prefill_T64_fp32_matches_decode_steps(ops):
    """Prefill over 64 tokens and 64 decode steps reach the same result (the
    prefill -> decode continuity of the page's batched-prefill check)."""
    lp, st, conv0, S0 = varlen_case(I.seed_of(0), [64], torch.float32, zero=True)
    o1, c1, S1 = gpu_prefill(ops, lp, st, [64], conv0, S0, torch.float32, chunk=1)
    lpd = lp.to(DEV)
    cp = ops.make_params(lpd)
    conv, S = conv0.to(DEV).clone(), S0.to(DEV).clone()
    outs = torch.empty(64, I.D_INNER, device=DEV)
    s = st.to(DEV)
    for t in range(64):
        ops.decode_step(None, s.qkv[t:t + 1], s.z[t:t + 1], s.alpha[t:t + 1], s.beta[t:t + 1], conv, S,
                        outs[t:t + 1], cparams=cp)
    torch.cuda.synchronize()
    assert tl.max_rel(outs.cpu(), o1) < 2e-6
    assert tl.max_rel(S.cpu(), S1) < 2e-6
    np.testing.assert_array_equal(conv.cpu().numpy(), c1.numpy())


def test_prefill_T4096_bf16(ops):
    """The T=4096 bf16 workload: batch 1, zero initial state, library-chosen
    chunking, fp32 output for parity; returns the output and the final state."""
    lp, st, conv0, S0 = varlen_case(I.seed_of(2), [4096], torch.bfloat16, zero=True)
    got = gpu_prefill(ops, lp, st, [4096], conv0, S0, torch.float32, chunk=0)
    ref = tl.oracle_sequence_split_heads(lp, st.qkv, st.z, st.alpha, st.beta, conv0[0], S0[0], groups=16)
    ref = (ref[0], ref[1][None], ref[2][None])
    check("prefill T4096 bf16", got, ref, torch.bfloat16, torch.float32)


def test_prefill_varlen_8_sequences(ops):
    """The varlen workload: 8 packed sequences, log-uniform lengths in
    [256, 32768], random initial states, one layer, bf16. Sampled parity on
    four V-heads (two K-head pairs) over every token of every sequence."""
    lengths = I.varlen_lengths(I.seed_of(4))
    lp, st, conv0, S0 = varlen_case(I.seed_of(4), lengths, torch.bfloat16)
    got = gpu_prefill(ops, lp, st, lengths, conv0, S0, torch.float32, chunk=0)
    heads = [0, 16, 7, 31]
    ref = oracle_varlen(lp, st, lengths, conv0, S0, heads=heads)
    print("lengths", lengths)
    check("varlen 8 seq", got, ref, torch.bfloat16, torch.float32, heads=heads)


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("chunk", [0, 1])
def test_prefill_ragged_and_empty(ops, act, chunk):
    """Ragged tails, sequences shorter than the conv window, and empty
    sequences (their states pass through unchanged), with random states."""
    lengths = [1, 0, 2, 3, 67, 0, 130, 64, 5]
    lp, st, conv0, S0 = varlen_case(900, lengths, act)
    got = gpu_prefill(ops, lp, st, lengths, conv0, S0, torch.float32, chunk=chunk)
    ref = oracle_varlen(lp, st, lengths, conv0, S0)
    check(f"ragged {act} chunk={chunk}", got, ref, act, torch.float32)


@pytest.mark.parametrize("out_dt", [torch.bfloat16])
def test_prefill_bf16_output(ops, out_dt):
    lengths = [100, 37]
    lp, st, conv0, S0 = varlen_case(901, lengths, torch.bfloat16)
    got = gpu_prefill(ops, lp, st, lengths, conv0, S0, out_dt, chunk=0)
    ref = oracle_varlen(lp, st, lengths, conv0, S0)
    check("bf16 out", got, ref, torch.bfloat16, out_dt)


def test_prefill_states_alias_in_place(ops):
    """conv_state_out / ssm_state_out may alias the inputs."""
    lengths = [70, 2, 129]
    lp, st, conv0, S0 = varlen_case(902, lengths, torch.bfloat16)
    got = gpu_prefill(ops, lp, st, lengths, conv0, S0, torch.float32, chunk=0, alias=True)
    ref = oracle_varlen(lp, st, lengths, conv0, S0)
    check("aliased states", got, ref, torch.bfloat16, torch.float32)


def test_prefill_fragment_continuity(ops):
    """prefill(T1) then prefill(T2) with the states carried equals one
    prefill(T1+T2): a prompt processed in fragments gives the same output."""
    L = 200
    lp, st, conv0, S0 = varlen_case(903, [L], torch.bfloat16)
    full = gpu_prefill(ops, lp, st, [L], conv0, S0, torch.float32, chunk=0)
    cut = 77
    a = I.Streams(st.qkv[:cut], st.z[:cut], st.alpha[:cut], st.beta[:cut])
    b = I.Streams(st.qkv[cut:], st.z[cut:], st.alpha[cut:], st.beta[cut:])
    ga = gpu_prefill(ops, lp, a, [cut], conv0, S0, torch.float32, chunk=0)
    gb = gpu_prefill(ops, lp, b, [L - cut], ga[1], ga[2], torch.float32, chunk=0)
    out = torch.cat([ga[0], gb[0]])
    assert tl.max_rel(out, full[0]) < tl.TOL_BF16_OUT
    assert tl.max_rel(gb[2], full[2]) < tl.TOL_BF16_STATE
    np.testing.assert_array_equal(gb[1].float().numpy(), full[1].float().numpy())
    ref = oracle_varlen(lp, st, [L], conv0, S0)
    check("fragments vs oracle", (out, gb[1], gb[2]), ref, torch.bfloat16, torch.float32)


def test_prefill_no_tokens_passes_states_through(ops):
    lengths = [0, 0]
    lp = I.layer_params(904)
    conv0, S0 = I.initial_states(904, 2, torch.bfloat16)
    st = I.streams(904, 0, torch.bfloat16)
    cu = I.cu_seqlens(lengths).to(DEV)
    cout = torch.empty(2, 3, I.C_CONV, dtype=torch.bfloat16, device=DEV)
    sout = torch.empty(2, I.HV, I.DV, I.DK, device=DEV)
    out = torch.empty(0, I.D_INNER, device=DEV)
    s = st.to(DEV)
    # zero-size tensors have no storage; the library accepts NULL streams when T_total == 0
    ops.lib()  # loaded
    from gated_deltanet_linear_02_gb300.ops import prefill
    prefill(lp.to(DEV), s.qkv, s.z, s.alpha, s.beta, cu, out, conv0.to(DEV), cout, S0.to(DEV), sout)
    torch.cuda.synchronize()
    assert torch.equal(cout.cpu(), conv0)
    assert torch.equal(sout.cpu(), S0)


def test_prefill_bitwise_repeatable(ops):
    # Two chunked calls on the same inputs (two sequences, 17 chunks, a ragged
    # tail) agree bit for bit: every sum has a fixed order.
    lengths = [700, 353]
    lp, st, conv0, S0 = varlen_case(I.seed_of(2, 77), lengths, torch.bfloat16)
    a = gpu_prefill(ops, lp, st, lengths, conv0, S0, torch.bfloat16, 64)
    b = gpu_prefill(ops, lp, st, lengths, conv0, S0, torch.bfloat16, 64)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("ws_tokens,alias", [(64, False), (128, True), (192, False)])
def test_prefill_windows_small_workspace(ops, ws_tokens, alias):
    """The chunked form given a workspace for windows of 64, 128 or 192 tokens:
    the packed tokens run as many windows, sequences cross window edges with
    their state carried between windows, and the result still matches the
    oracle (also with the states updated in place)."""
    lengths = [300, 77, 1, 0, 200, 64, 130]
    lp, st, conv0, S0 = varlen_case(905, lengths, torch.bfloat16)
    got = gpu_prefill(ops, lp, st, lengths, conv0, S0, torch.float32, chunk=64, alias=alias, ws_tokens=ws_tokens)
    ref = oracle_varlen(lp, st, lengths, conv0, S0)
    check(f"windows of {ws_tokens}", got, ref, torch.bfloat16, torch.float32)



def test_prefill_split_form_matches_oracle():
    """GDN_PREFILL_SPLIT=1 runs prep and the chains as two kernels instead of
    one cooperative kernel. The many-fragment, windowed and ragged cases above
    must hold in that form too (run in a child process, which reads the switch
    at its first prefill)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, GDN_PREFILL_SPLIT="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_parity_prefill.py", "-k",
                        "ragged_and_empty or windows_small_workspace or fragment_continuity or T4096"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=1200)
    print(r.stdout[-2000:])
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " 9 passed" in r.stdout or "9 passed" in r.stdout
