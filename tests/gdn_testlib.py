"""Shared helpers of the parity tests: run the oracle on the same seeded inputs
as the CUDA path, convert state layouts, and measure errors.

Errors follow the stated tolerance: per tensor, max|gpu - ref| / max|ref|
("max relative error"). The tests print an elementwise diagnostic beside it.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from oracle import oracle

# Tolerances: 1e-4 for fp32 inputs; 3e-3 on outputs and 1e-3 on the final
# state for bf16 inputs with fp32 state. A bf16 *output* also carries its own
# rounding, up to 2^-8 relative, on top of the 3e-3.
TOL_F32 = 1e-4
TOL_BF16_OUT = 3e-3
TOL_BF16_STATE = 1e-3
BF16_ROUND = 2.0 ** -8

_pool = None


def pool() -> ThreadPoolExecutor:
    """Threads for independent oracle calls (the C calls release the GIL)."""
    global _pool
    if _pool is None:
        _pool = ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1))
    return _pool


def oparams(lp) -> oracle.Params:
    return oracle.Params.of(lp.conv_w, lp.A_log, lp.dt_bias, lp.norm_w, lp.l2_eps, lp.norm_eps)


def f64(t) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def to_page(S_lib: np.ndarray) -> np.ndarray:
    """Library state [..][32][j][i] -> the page's S[..][32][i][j]."""
    return np.ascontiguousarray(np.swapaxes(S_lib, -1, -2))


def to_lib(S_page: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(np.swapaxes(S_page, -1, -2))


def max_rel(gpu, ref) -> float:
    gpu, ref = f64(gpu), f64(ref)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if gpu.size == 0:
        return 0.0
    assert np.all(np.isfinite(gpu)), "non-finite values in the GPU result"
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(gpu - ref)) / (den if den > 0 else 1.0))


def elem_rel(gpu, ref, floor=1e-3) -> float:
    """Elementwise diagnostic: max |gpu-ref| / max(|ref|, floor * max|ref|)."""
    gpu, ref = f64(gpu), f64(ref)
    if gpu.size == 0:
        return 0.0
    den = np.maximum(np.abs(ref), floor * np.max(np.abs(ref)) + 1e-300)
    return float(np.max(np.abs(gpu - ref) / den))


def oracle_sequences(lp, qkv, z, alpha, beta, cu, conv0, S0_lib, heads=None):
    """Run the oracle over packed sequences with the library's state layout.
    qkv, ... are [T, ...] tensors; cu a list; conv0 [N, 3, 8192]; S0_lib
    [N, 32, j, i] (any array-like). Returns (out [T,4096], conv [N,3,8192],
    S [N,32,j,i]) as float64 numpy."""
    P = oparams(lp)
    S0 = to_page(f64(S0_lib))
    out, cs, S = oracle.gdn_varlen(P, qkv, z, alpha, beta, cu, conv0, S0, heads=heads, pool=pool())
    return out, cs, to_lib(S)


def oracle_sequence_split_heads(lp, qkv, z, alpha, beta, conv0, S0_lib, groups=8, heads=None):
    """One sequence, with the V-heads split across threads (each thread repeats
    the cheap conv). Returns (out, conv_state, S) like oracle_sequences."""
    P = oparams(lp)
    S0 = to_page(f64(S0_lib))
    qkv, z, alpha, beta = map(f64, (qkv, z, alpha, beta))
    conv0 = f64(conv0)
    hv = list(range(32)) if heads is None else list(heads)
    chunks = [hv[i::groups] for i in range(groups) if hv[i::groups]]

    def one(hs):
        res = []
        for h in hs:
            res.append((h, oracle.gdn_sequence(P, qkv, z, alpha, beta, conv0, S0, heads=(h, h + 1))))
        return res

    out = np.zeros((qkv.shape[0], 4096))
    S = S0.copy()
    cs = None
    for part in pool().map(one, chunks):
        for h, (o, c, s) in part:
            out[:, h * 128:(h + 1) * 128] = o[:, h * 128:(h + 1) * 128]
            S[h] = s[h]
            cs = c
    return out, cs, to_lib(S)


def oracle_y_sequence(lp, qkv, alpha, beta, conv_state, S_lib):
    """The mixer's raw output y = scale S^T q^ of every token and V-head of
    one sequence (the gated norm left out), composed from the oracle's single
    steps: conv + SiLU per token, the L2 norms, the gates, then the per-token
    recurrence of each head over the sequence. S_lib is the library layout
    [32][j][i]. Returns y [T][4096] in fp64."""
    qkv, alpha, beta = f64(qkv), f64(alpha), f64(beta)
    T = qkv.shape[0]
    conv_w = f64(lp.conv_w)
    st = f64(conv_state).copy()
    xh = np.empty((T, qkv.shape[1]))
    for t in range(T):
        xh[t], st = oracle.conv_token(qkv[t], conv_w, st)
    HV, HK, D = 32, 16, 128
    S_page = to_page(f64(S_lib))
    y = np.zeros((T, HV * D))
    A_log, dt_bias = f64(lp.A_log), f64(lp.dt_bias)
    for vh in range(HV):
        kh = vh % HK
        q = np.stack([oracle.l2norm(xh[t, kh * D:(kh + 1) * D], lp.l2_eps) for t in range(T)])
        k = np.stack([oracle.l2norm(xh[t, 2048 + kh * D:2048 + (kh + 1) * D], lp.l2_eps) for t in range(T)])
        v = xh[:, 4096 + vh * D:4096 + (vh + 1) * D]
        gb = [oracle.gates(A_log[vh], dt_bias[vh], alpha[t, vh], beta[t, vh]) for t in range(T)]
        g = np.array([x[0] for x in gb])
        b = np.array([x[1] for x in gb])
        y[:, vh * D:(vh + 1) * D], _ = oracle.delta_rule_scan(q, k, v, g, b, S_page[vh], 1.0 / np.sqrt(D))
    return y
