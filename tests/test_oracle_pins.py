"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

The oracle restates "qwen35moe -- Forward-Pass Design (Pantheon port)", section
"SSM block -- Gated-Delta-Net". The page prints no worked numeric example for
the mixer. So the checks below use:
- the values the page does print (its dims table);
- closed forms of special cases;
- invariants;
- library routines for the textbook pieces (SiLU, softplus, norms);
- a brute-force product form on tiny heads.

Each is chosen so that a plausible slip fails at least one check: a dropped
term, a wrong sign or index, a transposed operand, a wrong conv tap order, a
doubled scale, or the wrong GQA pairing.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import expit

HERE = os.path.dirname(os.path.abspath(__file__))
rng = np.random.default_rng


def _unit(x):
    return x / np.linalg.norm(x)


# --------------------------------------------------------------- page values

def test_page_dims_fixture(orc):
    """The SSM dims and per-layer state sizes printed in the page's "Config" table
    and its "Dual state" section."""
    vals = {}
    with open(os.path.join(HERE, "golden", "qwen35moe_ssm_dims.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    Hv, Hk, dk, dv, Kc = orc.PAGE_DIMS
    assert (Hv, Hk, dk, Kc) == (vals["ssm_time_step_rank"], vals["ssm_group_count"],
                                vals["ssm_state_size"], vals["ssm_conv_kernel"])
    assert Hv * dv == vals["ssm_inner_size"]
    assert orc.Dims(*orc.PAGE_DIMS).C == vals["conv_dim"]
    assert (Kc - 1) * vals["conv_dim"] == vals["conv_state_f32_per_layer"]
    assert dk * Hv * dv == vals["ssm_state_f32_per_layer"]
    assert vals["conv_state_f32_per_layer"] + vals["ssm_state_f32_per_layer"] == \
        vals["state_f32_per_ssm_layer"]
    n_attn = sum(1 for i in range(vals["n_layer"]) if (i + 1) % vals["full_attention_interval"] == 0)
    assert vals["n_layer"] - n_attn == vals["ssm_layers"]
    from gated_deltanet_linear_02_gb300 import inputs
    assert (inputs.HV, inputs.HK, inputs.DK, inputs.DV, inputs.KCONV) == (Hv, Hk, dk, dv, Kc)
    assert inputs.C_CONV == vals["conv_dim"] and inputs.D_INNER == vals["ssm_inner_size"]


# --------------------------------------------------------------------- gates

def test_gates_closed_form(orc):
    # A_log = ln 16 and alpha + dt_bias = 0 give g = -16 softplus(0) = -16 ln 2.
    g, b = orc.gates(math.log(16.0), 0.7, -0.7, 0.0)
    assert g == pytest.approx(-16.0 * math.log(2.0), rel=1e-14)
    assert b == 0.5


def test_gates_library_and_ranges(orc):
    r = rng(1)
    for _ in range(200):
        A, dt, al, be = r.uniform(0, math.log(16)), r.uniform(-1, 1), r.normal(0, 3), r.normal(0, 3)
        g, b = orc.gates(A, dt, al, be)
        # softplus against numpy's logaddexp(0, x); sigmoid against scipy's expit
        assert g == pytest.approx(-math.exp(A) * np.logaddexp(0.0, al + dt), rel=1e-12)
        assert b == pytest.approx(expit(be), rel=1e-12)
        assert g <= 0.0 and 0.0 < math.exp(g) <= 1.0 and 0.0 < b < 1.0
    # linear tail of softplus above 20, and continuity across the switch
    assert orc.softplus(30.0) == pytest.approx(30.0, rel=1e-15)
    assert orc.softplus(20.0) == pytest.approx(np.logaddexp(0.0, 20.0), rel=1e-15)
    assert orc.softplus(-30.0) == pytest.approx(math.exp(-30.0), rel=1e-12)


# ---------------------------------------------------------------------- conv

def test_conv_identity_tap_is_silu(orc):
    # weight e_3: the conv output is the current input, so the token output is SiLU(x_t)
    r = rng(2)
    C = 24
    w = np.zeros((C, 4)); w[:, 3] = 1.0
    state = r.normal(size=(3, C))
    x = r.normal(size=C)
    xhat, st = orc.conv_token(x, w, state)
    np.testing.assert_allclose(xhat, x * expit(x), rtol=1e-14)
    np.testing.assert_array_equal(st, np.stack([state[1], state[2], x]))


def test_conv_impulse_tap_order_and_shift(orc):
    # a unit impulse at t=0 walks from tap 3 (the current token) down to tap 0
    r = rng(3)
    C = 5
    w = r.normal(size=(C, 4))
    st = np.zeros((3, C))
    outs = []
    for t in range(6):
        x = np.zeros(C)
        if t == 0:
            x[2] = 1.0
        xhat, st = orc.conv_token(x, w, st)
        outs.append(xhat[2])
    expect = [w[2, 3 - t] * expit(w[2, 3 - t]) for t in range(4)] + [0.0, 0.0]
    np.testing.assert_allclose(outs, expect, rtol=1e-14, atol=0)


def test_conv_state_prefix(orc):
    # zero inputs after a nonzero state: taps 0..2 meet the state rows oldest-first
    r = rng(4)
    C = 3
    w = r.normal(size=(C, 4))
    s = r.normal(size=(3, C))
    st = s.copy()
    got = []
    for _ in range(4):
        xhat, st = orc.conv_token(np.zeros(C), w, st)
        got.append(xhat)
    u = [w[:, 0] * s[0] + w[:, 1] * s[1] + w[:, 2] * s[2], w[:, 0] * s[1] + w[:, 1] * s[2],
         w[:, 0] * s[2], np.zeros(C)]
    for t in range(4):
        np.testing.assert_allclose(got[t], u[t] * expit(u[t]), rtol=1e-13, atol=1e-300)


# --------------------------------------------------------------------- norms

def test_l2norm(orc):
    r = rng(5)
    x = r.normal(size=128) * 3.0
    y = orc.l2norm(x, eps=0.0)
    np.testing.assert_allclose(y, x / np.linalg.norm(x), rtol=1e-14)
    assert np.linalg.norm(orc.l2norm(x, eps=1e-6)) == pytest.approx(1.0, abs=1e-7)
    np.testing.assert_array_equal(orc.l2norm(np.zeros(16), eps=1e-6), np.zeros(16))


def test_gated_rmsnorm_invariants(orc):
    r = rng(6)
    y, z = r.normal(size=128), r.normal(size=128)
    w1 = np.ones(128)
    o = orc.gated_rmsnorm(y, z, w1, eps=0.0)
    base = o / (z * expit(z))                      # undo the silu gate
    assert np.sqrt(np.mean(base ** 2)) == pytest.approx(1.0, rel=1e-13)   # RMS = 1
    np.testing.assert_allclose(orc.gated_rmsnorm(7.5 * y, z, w1, eps=0.0), o, rtol=1e-13)  # scale-free
    np.testing.assert_array_equal(orc.gated_rmsnorm(y, np.zeros(128), w1), np.zeros(128))  # silu(0)=0
    w = 1.0 + 0.1 * r.normal(size=128)
    np.testing.assert_allclose(orc.gated_rmsnorm(y, z, w, eps=0.0), o * w, rtol=1e-13)   # w, not 1+w
    # the gate is silu(z), not sigmoid(z): silu(z)/sigmoid(z) = z
    np.testing.assert_allclose(o / expit(z) / base, z, rtol=1e-12)


# ---------------------------------------------------------------- delta rule

def test_beta_zero_is_pure_decay(orc):
    # beta = 0: no write, S_T = exp(sum g) S_0 and y_t = scale exp(G_t) S_0^T q_t
    r = rng(7)
    dk, dv, T = 16, 12, 9
    S0 = r.normal(size=(dk, dv))
    q = np.stack([_unit(r.normal(size=dk)) for _ in range(T)])
    k = np.stack([_unit(r.normal(size=dk)) for _ in range(T)])
    v = r.normal(size=(T, dv))
    g = -r.uniform(0, 2, size=T)
    y, S = orc.delta_rule_scan(q, k, v, g, np.zeros(T), S0, scale=0.25)
    G = np.cumsum(g)
    np.testing.assert_allclose(S, math.exp(G[-1]) * S0, rtol=1e-13)
    for t in range(T):
        np.testing.assert_allclose(y[t], 0.25 * math.exp(G[t]) * (S0.T @ q[t]), rtol=1e-12, atol=1e-14)


def test_retrieval_after_write(orc):
    # g = 0, beta = 1: the write makes the state return v_t under k_t exactly
    r = rng(8)
    dk, dv = 8, 6
    S = r.normal(size=(dk, dv))
    k = _unit(r.normal(size=dk))
    v = r.normal(size=dv)
    S1, y = orc.delta_rule_token(S, k, v, k, g=0.0, b=1.0, scale=1.0)
    np.testing.assert_allclose(S1.T @ k, v, rtol=1e-12, atol=1e-13)
    # read-after-write: querying with q = k returns v too (scale 1)
    np.testing.assert_allclose(y, v, rtol=1e-12, atol=1e-13)


def test_orthonormal_keys_store_outer_products(orc):
    r = rng(9)
    dk, dv, T = 16, 5, 10
    Qm, _ = np.linalg.qr(r.normal(size=(dk, dk)))
    k = Qm[:, :T].T                     # T orthonormal keys
    v = r.normal(size=(T, dv))
    y, S = orc.delta_rule_scan(k, k, v, np.zeros(T), np.ones(T), np.zeros((dk, dv)), scale=1.0)
    np.testing.assert_allclose(S, k.T @ v, rtol=1e-12, atol=1e-13)   # S_T = sum k_t v_t^T
    np.testing.assert_allclose(S.T @ k.T, v.T, rtol=1e-12, atol=1e-13)  # every key retrieves its value


def test_first_token_closed_form(orc):
    # from S_0 = 0: S_1 = b k v^T (decay acts on zero), y = scale b (k.q) v
    r = rng(10)
    dk, dv = 8, 4
    k, q = _unit(r.normal(size=dk)), _unit(r.normal(size=dk))
    v = r.normal(size=dv)
    S1, y = orc.delta_rule_token(np.zeros((dk, dv)), k, v, q, g=-0.3, b=0.6, scale=0.125)
    np.testing.assert_allclose(S1, 0.6 * np.outer(k, v), rtol=1e-14)
    np.testing.assert_allclose(y, 0.125 * 0.6 * (k @ q) * v, rtol=1e-13)


@pytest.mark.parametrize("dk,dv,T", [(2, 2, 1), (3, 2, 3), (4, 3, 4), (2, 4, 4)])
def test_product_form_brute_force(orc, dk, dv, T):
    # S_T = P_T..P_1 S_0 + sum_t P_T..P_{t+1} b_t k_t v_t^T with P_t = a_t (I - b_t k_t k_t^T),
    # latest step leftmost; y_t = scale S_t^T q_t
    r = rng(100 + dk * 10 + T)
    S0 = r.normal(size=(dk, dv))
    q = np.stack([_unit(r.normal(size=dk)) for _ in range(T)])
    k = np.stack([_unit(r.normal(size=dk)) for _ in range(T)])
    v = r.normal(size=(T, dv))
    g = -r.uniform(0, 1.5, size=T)
    b = r.uniform(0.05, 0.95, size=T)
    y, S = orc.delta_rule_scan(q, k, v, g, b, S0, scale=0.5)
    P = [math.exp(g[t]) * (np.eye(dk) - b[t] * np.outer(k[t], k[t])) for t in range(T)]
    for t in range(T):
        prod = np.eye(dk)
        for s in range(t + 1):          # prod = P_t ... P_0 (latest left)
            prod = P[s] @ prod
        St = prod @ S0
        for s in range(t + 1):
            tail = np.eye(dk)
            for u in range(s + 1, t + 1):
                tail = P[u] @ tail
            St = St + tail @ (b[s] * np.outer(k[s], v[s]))
        np.testing.assert_allclose(y[t], 0.5 * St.T @ q[t], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(S, St, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("T,chunk", [(13, 4), (13, 1), (64, 64), (70, 64), (5, 64), (128, 16)])
def test_chunked_form_matches_scan(orc, T, chunk):
    """The WY/UT chunked re-association equals the token scan in fp64, including
    partial last chunks and strong decay (cumulative log-decay far below -700)."""
    r = rng(200 + T + chunk)
    dk, dv = 16, 8
    q = np.stack([_unit(r.normal(size=dk)) for _ in range(T)])
    k = np.stack([_unit(r.normal(size=dk)) for _ in range(T)])
    v = r.normal(size=(T, dv))
    g = -r.uniform(0, 3, size=T)
    g[T // 2:] -= 40.0                    # very strong decay: exp(G) underflows inside chunks
    b = r.uniform(0, 1, size=T)
    S0 = r.normal(size=(dk, dv)) * 0.5
    y1, S1 = orc.delta_rule_scan(q, k, v, g, b, S0, scale=0.25)
    y2, S2 = orc.delta_rule_chunked(q, k, v, g, b, S0, scale=0.25, chunk=chunk)
    np.testing.assert_allclose(y2, y1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(S2, S1, rtol=1e-10, atol=1e-12)
    assert np.all(np.isfinite(y2)) and np.all(np.isfinite(S2))


# ------------------------------------------------------------- whole mixer

SMALL = (4, 2, 8, 6, 4)   # Hv, Hk, dk, dv, Kc


def _small_case(seed, T, dims=SMALL, state=True):
    Hv, Hk, dk, dv, Kc = dims
    C = 2 * Hk * dk + Hv * dv
    r = rng(seed)
    from oracle.oracle import Params
    p = Params.of(r.normal(size=(C, Kc)) * 0.5, r.uniform(0, math.log(16), Hv),
                  r.uniform(-1, 1, Hv), 1 + 0.1 * r.normal(size=dv))
    x = dict(qkv=r.normal(size=(T, C)), z=r.normal(size=(T, Hv * dv)),
             alpha=r.normal(size=(T, Hv)), beta=r.normal(size=(T, Hv)))
    cs = r.normal(size=(Kc - 1, C)) if state else np.zeros((Kc - 1, C))
    S = r.normal(size=(Hv, dk, dv)) * 0.1 if state else np.zeros((Hv, dk, dv))
    return p, x, cs, S


def test_layer_first_token_closed_form(orc):
    """T=1 from zero states reduces the whole mixer to a closed form.

    The conv keeps only tap 3, and the state write is S_1 = b k v^T, so
    y = scale b (k.q) v. The norm eps is set large so that the 1/sqrt(dk)
    scale shows in the output. A doubled scale, a wrong split offset, a wrong
    GQA pairing or a wrong gate would each fail this check."""
    Hv, Hk, dk, dv, Kc = SMALL
    p, x, cs, S = _small_case(11, 1, state=False)
    p.norm_eps = 0.5
    out, cs1, S1 = orc.gdn_sequence(p, x["qkv"], x["z"], x["alpha"], x["beta"], cs, S, dims=SMALL)
    u = p.conv_w[:, Kc - 1] * x["qkv"][0]
    xh = u * expit(u)
    for vh in range(Hv):
        kh = vh % Hk
        q = xh[kh * dk:(kh + 1) * dk]
        k = xh[Hk * dk + kh * dk: Hk * dk + (kh + 1) * dk]
        v = xh[2 * Hk * dk + vh * dv: 2 * Hk * dk + (vh + 1) * dv]
        qn, kn = q / np.sqrt(q @ q + p.l2_eps), k / np.sqrt(k @ k + p.l2_eps)
        b = expit(x["beta"][0, vh])
        y = b * (kn @ qn) * v / math.sqrt(dk)
        zz = x["z"][0, vh * dv:(vh + 1) * dv]
        o = y / np.sqrt(np.mean(y * y) + p.norm_eps) * p.norm_w * zz * expit(zz)
        np.testing.assert_allclose(out[0, vh * dv:(vh + 1) * dv], o, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(S1[vh], b * np.outer(kn, v), rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(cs1[-1], x["qkv"][0])


def test_gqa_interleaved_pairing(orc):
    """V-head vh reads K-head vh % Hk (the watch-list item on the interleaved
    ggml_repeat): perturbing K-head kh's q|k channels changes exactly V-heads
    {kh, kh + Hk}. The blocked pairing would change {2kh, 2kh+1} instead."""
    Hv, Hk, dk, dv, Kc = dims = (8, 4, 4, 3, 4)
    p, x, cs, S = _small_case(12, 3, dims=dims)
    base, _, _ = orc.gdn_sequence(p, x["qkv"], x["z"], x["alpha"], x["beta"], cs, S, dims=dims)
    for kh in range(Hk):
        qkv = x["qkv"].copy()
        qkv[:, kh * dk:(kh + 1) * dk] += 0.5                          # q channels of K-head kh
        qkv[:, Hk * dk + kh * dk: Hk * dk + (kh + 1) * dk] -= 0.5      # k channels of K-head kh
        out, _, _ = orc.gdn_sequence(p, qkv, x["z"], x["alpha"], x["beta"], cs, S, dims=dims)
        changed = {vh for vh in range(Hv)
                   if not np.allclose(out[:, vh * dv:(vh + 1) * dv], base[:, vh * dv:(vh + 1) * dv],
                                      rtol=0, atol=1e-14)}
        assert changed == {kh, kh + Hk}


def test_layer_split_continuity(orc):
    """Processing T1 then T2 tokens with the states carried equals one pass over
    T1+T2 (fragmented prefill, and prefill followed by single-token decode)."""
    p, x, cs, S = _small_case(13, 11)
    full = orc.gdn_sequence(p, x["qkv"], x["z"], x["alpha"], x["beta"], cs, S, dims=SMALL)
    for cut in (1, 2, 5, 10):
        a = orc.gdn_sequence(p, *(x[n][:cut] for n in ("qkv", "z", "alpha", "beta")), cs, S, dims=SMALL)
        b = orc.gdn_sequence(p, *(x[n][cut:] for n in ("qkv", "z", "alpha", "beta")), a[1], a[2],
                             dims=SMALL)
        np.testing.assert_array_equal(np.concatenate([a[0], b[0]]), full[0])
        np.testing.assert_array_equal(b[1], full[1])
        np.testing.assert_array_equal(b[2], full[2])


def test_layer_heads_subset(orc):
    """The per-head restriction used for sampled parity equals the full call on
    those heads and leaves the conv state identical."""
    p, x, cs, S = _small_case(14, 6)
    full = orc.gdn_sequence(p, x["qkv"], x["z"], x["alpha"], x["beta"], cs, S, dims=SMALL)
    part = orc.gdn_sequence(p, x["qkv"], x["z"], x["alpha"], x["beta"], cs, S, dims=SMALL, heads=(1, 3))
    dv = SMALL[3]
    np.testing.assert_array_equal(part[0][:, dv:3 * dv], full[0][:, dv:3 * dv])
    np.testing.assert_array_equal(part[2][1:3], full[2][1:3])
    np.testing.assert_array_equal(part[2][0], S[0])
    np.testing.assert_array_equal(part[1], full[1])


def test_layer_matches_chunked_form_composition(orc):
    """The whole mixer at page dims, one head, against the chunked form. The
    per-token conv, norms and gates come from the single-step routines, and
    the recurrence comes from the chunked re-association with C=64."""
    from oracle.oracle import Params
    Hv, Hk, dk, dv, Kc = orc.PAGE_DIMS
    C = 2 * Hk * dk + Hv * dv
    r = rng(15)
    T = 70
    p = Params.of(r.normal(size=(C, Kc)) * 0.25, r.uniform(0, math.log(16), Hv),
                  r.uniform(-1, 1, Hv), 1 + 0.1 * r.normal(size=dv))
    qkv, z = r.normal(size=(T, C)), r.normal(size=(T, Hv * dv))
    al, be = r.normal(size=(T, Hv)), r.normal(size=(T, Hv))
    cs, S = r.normal(size=(Kc - 1, C)), r.normal(size=(Hv, dk, dv)) * 0.02
    vh = 21
    out, _, Sf = orc.gdn_sequence(p, qkv, z, al, be, cs, S, heads=(vh, vh + 1))
    kh = vh % Hk
    st = cs.copy()
    qs, ks, vs, gs, bs = [], [], [], [], []
    for t in range(T):
        xh, st = orc.conv_token(qkv[t], p.conv_w, st)
        qs.append(orc.l2norm(xh[kh * dk:(kh + 1) * dk]))
        ks.append(orc.l2norm(xh[Hk * dk + kh * dk:Hk * dk + (kh + 1) * dk]))
        vs.append(xh[2 * Hk * dk + vh * dv:2 * Hk * dk + (vh + 1) * dv])
        g, b = orc.gates(p.A_log[vh], p.dt_bias[vh], al[t, vh], be[t, vh])
        gs.append(g); bs.append(b)
    y, S2 = orc.delta_rule_chunked(np.array(qs), np.array(ks), np.array(vs), np.array(gs),
                                   np.array(bs), S[vh], 1 / math.sqrt(dk), 64)
    o = np.stack([orc.gated_rmsnorm(y[t], z[t, vh * dv:(vh + 1) * dv], p.norm_w) for t in range(T)])
    np.testing.assert_allclose(out[:, vh * dv:(vh + 1) * dv], o, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(Sf[vh], S2, rtol=1e-10, atol=1e-13)


# ---------------------------------------------------------------- out_proj

def test_out_proj_identity_block(orc):
    """w = [I | 0] (n_embd x 4096) selects the first n_embd columns of x:
    pins the orientation y = x w^T (one weight row per output feature)."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((5, 4096))
    w = np.zeros((2048, 4096))
    w[:, :2048] = np.eye(2048)
    np.testing.assert_array_equal(orc.out_proj(x, w), x[:, :2048])


def test_out_proj_brute_force(orc):
    """Each output is the plain sum over k, written out as a loop on a slice."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((3, 64))
    w = rng.standard_normal((5, 64))
    y = orc.out_proj(x, w)
    for m in range(3):
        for n in range(5):
            ref = 0.0
            for k in range(64):
                ref += x[m, k] * w[n, k]
            assert abs(y[m, n] - ref) <= 1e-12 * (1 + abs(ref))


def test_out_proj_rows_independent_and_linear(orc):
    """Row m of y depends on row m of x only, linearly."""
    rng = np.random.default_rng(13)
    x = rng.standard_normal((4, 256))
    w = rng.standard_normal((16, 256))
    y = orc.out_proj(x, w)
    y2 = orc.out_proj(2.0 * x[2:3], w)
    np.testing.assert_allclose(y2[0], 2.0 * y[2], rtol=1e-12, atol=1e-12)


def test_in_proj_streams_and_order(orc):
    """Each stream comes from its own weight, in the page's order; the first
    n_embd rows of an identity-block attn_qkv weight copy h into qkv."""
    rng = np.random.default_rng(14)
    h = rng.standard_normal((3, 2048))
    w_qkv = np.zeros((8192, 2048))
    w_qkv[:2048] = np.eye(2048)
    w_gate = np.zeros((4096, 2048))
    w_gate[5, 7] = 2.0                      # z[:, 5] = 2 h[:, 7]
    w_alpha = np.zeros((32, 2048))
    w_alpha[0, 0] = 1.0
    w_beta = np.zeros((32, 2048))
    w_beta[31, 2047] = -1.0
    qkv, z, al, be = orc.in_proj(h, w_qkv, w_gate, w_alpha, w_beta)
    assert qkv.shape == (3, 8192) and z.shape == (3, 4096) and al.shape == (3, 32) and be.shape == (3, 32)
    np.testing.assert_array_equal(qkv[:, :2048], h)
    assert not qkv[:, 2048:].any()
    np.testing.assert_array_equal(z[:, 5], 2.0 * h[:, 7])
    np.testing.assert_array_equal(al[:, 0], h[:, 0])
    np.testing.assert_array_equal(be[:, 31], -h[:, 2047])

