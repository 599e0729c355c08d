"""ctypes front end of the fp64 CPU oracle (``gdn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg use this module; the product path never does.

The oracle follows "qwen35moe -- Forward-Pass Design (Pantheon port)",
section "SSM block -- Gated-Delta-Net". Arrays cross the boundary as
contiguous float64 numpy arrays. The state convention is the page's:
``S[vh][i][j]`` with ``i`` the key index. The CUDA library keeps the
transpose ``[vh][j][i]``, and callers convert explicitly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_gdn.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` with gcc into ``oracle/_build``. Plain -O2, no
    fast-math (the oracle must keep IEEE fp64 semantics), portable flags only."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Dims(ctypes.Structure):
    _fields_ = [("Hv", ctypes.c_int), ("Hk", ctypes.c_int), ("dk", ctypes.c_int),
                ("dv", ctypes.c_int), ("Kc", ctypes.c_int)]

    @property
    def C(self) -> int:
        return 2 * self.Hk * self.dk + self.Hv * self.dv


PAGE_DIMS = (32, 16, 128, 128, 4)   # Hv, Hk, dk, dv, conv K ("Config (mini)" table)

_D = ctypes.POINTER(ctypes.c_double)


def _lib_handle():
    global _lib
    if _lib is None:
        # GDN_ORACLE_LIB points the oracle at another build of gdn_oracle.c; the
        # mutation test uses it to check that the pins catch planted mistakes.
        lib = ctypes.CDLL(os.environ.get("GDN_ORACLE_LIB") or build())
        lib.oracle_gdn_sequence.restype = ctypes.c_int
        lib.oracle_gdn_sequence.argtypes = [ctypes.POINTER(Dims), ctypes.c_int] + [_D] * 8 + \
            [ctypes.c_double, ctypes.c_double, _D, _D, _D]
        lib.oracle_gdn_sequence_heads.restype = ctypes.c_int
        lib.oracle_gdn_sequence_heads.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int] + [_D] * 8 + \
            [ctypes.c_double, ctypes.c_double, _D, _D, _D]
        lib.oracle_delta_rule_chunked.restype = ctypes.c_int
        lib.oracle_delta_rule_chunked.argtypes = [ctypes.c_int] * 4 + [_D] * 5 + [ctypes.c_double, _D, _D]
        lib.oracle_delta_rule_scan.restype = ctypes.c_int
        lib.oracle_delta_rule_scan.argtypes = [ctypes.c_int] * 3 + [_D] * 5 + [ctypes.c_double, _D, _D]
        lib.oracle_delta_rule_token.restype = None
        lib.oracle_delta_rule_token.argtypes = [ctypes.c_int, ctypes.c_int, _D, _D, _D, _D,
                                                ctypes.c_double, ctypes.c_double, ctypes.c_double, _D]
        lib.oracle_conv_token.restype = None
        lib.oracle_conv_token.argtypes = [ctypes.c_int, ctypes.c_int, _D, _D, _D, _D]
        lib.oracle_l2norm.restype = None
        lib.oracle_l2norm.argtypes = [ctypes.c_int, _D, ctypes.c_double, _D]
        lib.oracle_gates.restype = None
        lib.oracle_gates.argtypes = [ctypes.c_double] * 4 + [_D, _D]
        lib.oracle_softplus.restype = ctypes.c_double
        lib.oracle_softplus.argtypes = [ctypes.c_double]
        lib.oracle_gated_rmsnorm.restype = None
        lib.oracle_gated_rmsnorm.argtypes = [ctypes.c_int, _D, _D, _D, ctypes.c_double, _D]
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    """Contiguous float64 copy-or-view of anything array-like (torch tensors are
    converted exactly: bf16 and fp32 values are representable in fp64)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_D)


# ---------------------------------------------------------------- single steps

def conv_token(x, w, state):
    """One token of the causal conv1d + SiLU; returns (xhat, new_state)."""
    x, w, st = _f64(x), _f64(w), _f64(state).copy()
    C, Kc = w.shape
    out = np.empty(C)
    _lib_handle().oracle_conv_token(C, Kc, _p(x), _p(w), _p(st), _p(out))
    return out, st


def l2norm(x, eps=1e-6):
    x = _f64(x)
    out = np.empty_like(x)
    _lib_handle().oracle_l2norm(x.size, _p(x), eps, _p(out))
    return out


def gates(A_log, dt_bias, alpha, beta):
    """Returns (g, b): g = -exp(A_log) softplus(alpha + dt_bias), b = sigmoid(beta)."""
    g, b = ctypes.c_double(), ctypes.c_double()
    _lib_handle().oracle_gates(float(A_log), float(dt_bias), float(alpha), float(beta),
                               ctypes.byref(g), ctypes.byref(b))
    return g.value, b.value


def softplus(x):
    return _lib_handle().oracle_softplus(float(x))


def delta_rule_token(S, k, v, q, g, b, scale):
    """One recurrence step on S[i][j]; returns (S_new, y)."""
    S = _f64(S).copy()
    k, v, q = _f64(k), _f64(v), _f64(q)
    dk, dv = S.shape
    y = np.empty(dv)
    _lib_handle().oracle_delta_rule_token(dk, dv, _p(S), _p(k), _p(v), _p(q), float(g), float(b),
                                          float(scale), _p(y))
    return S, y


def gated_rmsnorm(y, z, w, eps=1e-6):
    y, z, w = _f64(y), _f64(z), _f64(w)
    out = np.empty_like(y)
    _lib_handle().oracle_gated_rmsnorm(y.size, _p(y), _p(z), _p(w), eps, _p(out))
    return out


def delta_rule_scan(q, k, v, g, b, S0, scale):
    """Per-token recurrence over pre-normalised q, k (T x dk), v (T x dv), gates g, b (T)."""
    q, k, v, g, b = map(_f64, (q, k, v, g, b))
    S = _f64(S0).copy()
    T, dk = k.shape
    dv = v.shape[1]
    y = np.zeros((T, dv))
    rc = _lib_handle().oracle_delta_rule_scan(dk, dv, T, _p(q), _p(k), _p(v), _p(g), _p(b),
                                              float(scale), _p(S), _p(y))
    assert rc == 0
    return y, S


def delta_rule_chunked(q, k, v, g, b, S0, scale, chunk):
    """The WY/UT chunked form of the same recurrence (see gdn_oracle.c)."""
    q, k, v, g, b = map(_f64, (q, k, v, g, b))
    S = _f64(S0).copy()
    T, dk = k.shape
    dv = v.shape[1]
    y = np.zeros((T, dv))
    rc = _lib_handle().oracle_delta_rule_chunked(dk, dv, T, int(chunk), _p(q), _p(k), _p(v), _p(g),
                                                 _p(b), float(scale), _p(S), _p(y))
    assert rc == 0
    return y, S


# --------------------------------------------------------------- whole mixer

def in_proj(h, w_qkv, w_gate, w_alpha, w_beta):
    """The four input projections of section "SSM block -- Gated-Delta-Net",
    each from the normed hidden states h [M][n_embd]: attn_qkv -> qkv,
    attn_gate -> z, ssm_alpha -> alpha, ssm_beta -> beta. Each weight holds one
    row per output feature. Returns (qkv, z, alpha, beta) in fp64."""
    h = _f64(h)
    return tuple(h @ _f64(w).T for w in (w_qkv, w_gate, w_alpha, w_beta))


def out_proj(x, w):
    """The projection after the mixer, section "Output path": cur = ssm_out .
    gated, 4096 -> n_embd. With x [M][K] (the gated output rows) and w [N][K]
    (ssm_out.weight, one row per output feature):
    y[m][n] = sum_k x[m][k] w[n][k]. fp64 over exact copies of the inputs;
    the library matrix product is the step."""
    x, w = _f64(x), _f64(w)
    assert x.ndim == 2 and w.ndim == 2 and x.shape[1] == w.shape[1]
    return x @ w.T


ATTN_Q_HEADS, ATTN_KV_HEADS, ATTN_HEAD_DIM = 16, 2, 256   # "Config (mini)" / "Full-attention block"


def attn_decode(q, k_cache, v_cache, ctx_len, z):
    """Decode attention of the full-attention layers, steps 5-6 of section
    "Full-attention block": every query head h of sequence b attends over the
    first ctx_len[b] cached positions of KV head h // (16 / 2) (GQA: 8 query
    heads share one KV head), with scale 1/sqrt(head_dim); then the output gate
    cur = attn_out * sigmoid(z). q and z are [B][16][256] (q after its RMSNorm
    and RoPE), the caches [B][2][Lmax][256] (keys after theirs). An empty
    context gives a zero output. fp64 over exact copies of the inputs; the
    dot products are library matrix products."""
    q, kc, vc, z = _f64(q), _f64(k_cache), _f64(v_cache), _f64(z)
    B, Hq, D = q.shape
    Hkv = kc.shape[1]
    group = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(ctx_len[b])
        if L <= 0:
            continue
        for h in range(Hq):
            g = h // group
            K, V = kc[b, g, :L], vc[b, g, :L]
            s = (K @ q[b, h]) / np.sqrt(D)          # scores of the L positions
            p = np.exp(s - s.max())
            p /= p.sum()                             # softmax
            o = p @ V
            out[b, h] = o / (1.0 + np.exp(-z[b, h]))   # o * sigmoid(z)
    return out


@dataclass
class Params:
    """One layer's parameters as fp64 arrays (the page's tensor roles:
    ssm_conv1d.weight, ssm_a via A_log, ssm_dt.bias, ssm_norm.weight)."""
    conv_w: np.ndarray   # [C][Kc]
    A_log: np.ndarray    # [Hv]
    dt_bias: np.ndarray  # [Hv]
    norm_w: np.ndarray   # [dv]
    l2_eps: float = 1e-6
    norm_eps: float = 1e-6

    @staticmethod
    def of(conv_w, A_log, dt_bias, norm_w, l2_eps=1e-6, norm_eps=1e-6) -> "Params":
        return Params(_f64(conv_w), _f64(A_log), _f64(dt_bias), _f64(norm_w), l2_eps, norm_eps)


def gdn_sequence(params: Params, qkv, z, alpha, beta, conv_state, S, dims=PAGE_DIMS,
                 heads: tuple[int, int] | None = None):
    """Run the whole mixer over one sequence.

    qkv [T][C], z [T][Hv*dv], alpha/beta [T][Hv]; conv_state [Kc-1][C];
    S [Hv][dk][dv] (page layout). Returns (out [T][Hv*dv], conv_state, S).
    With ``heads=(vh0, vh1)`` only those V-heads are computed (the others'
    outputs are left at 0 and their states unchanged)."""
    d = Dims(*dims)
    qkv, z, alpha, beta = map(_f64, (qkv, z, alpha, beta))
    cs = _f64(conv_state).copy()
    S = _f64(S).copy()
    T = qkv.shape[0]
    assert qkv.shape == (T, d.C) and z.shape == (T, d.Hv * d.dv)
    assert alpha.shape == (T, d.Hv) and beta.shape == (T, d.Hv)
    assert cs.shape == (d.Kc - 1, d.C) and S.shape == (d.Hv, d.dk, d.dv)
    out = np.zeros((T, d.Hv * d.dv))
    p = params
    args = (_p(qkv), _p(z), _p(alpha), _p(beta), _p(p.conv_w), _p(p.A_log), _p(p.dt_bias),
            _p(p.norm_w), float(p.l2_eps), float(p.norm_eps), _p(cs), _p(S), _p(out))
    if heads is None:
        rc = _lib_handle().oracle_gdn_sequence(ctypes.byref(d), T, *args)
    else:
        rc = _lib_handle().oracle_gdn_sequence_heads(ctypes.byref(d), T, int(heads[0]),
                                                     int(heads[1]), *args)
    assert rc == 0, "oracle rejected its arguments"
    return out, cs, S


def gdn_varlen(params: Params, qkv, z, alpha, beta, cu_seqlens, conv_state, S,
               dims=PAGE_DIMS, heads=None, pool=None):
    """Packed sequences: runs gdn_sequence on each [cu[n], cu[n+1]) slice with
    that sequence's own states. conv_state [N][Kc-1][C], S [N][Hv][dk][dv].
    ``pool`` (a concurrent.futures executor) runs sequences in parallel: the
    C calls release the GIL."""
    cu = [int(x) for x in cu_seqlens]
    N = len(cu) - 1
    qkv, z, alpha, beta = map(_f64, (qkv, z, alpha, beta))
    cs, S = _f64(conv_state), _f64(S)

    def one(n):
        a, b = cu[n], cu[n + 1]
        return gdn_sequence(params, qkv[a:b], z[a:b], alpha[a:b], beta[a:b], cs[n], S[n], dims, heads)

    res = list(pool.map(one, range(N))) if pool is not None else [one(n) for n in range(N)]
    out = np.concatenate([r[0] for r in res], axis=0) if N else np.zeros((0, z.shape[1]))
    return out, np.stack([r[1] for r in res]), np.stack([r[2] for r in res])
