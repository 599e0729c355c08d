"""Pins of the oracle's decode attention (steps 5-6 of section "Full-attention
block" of "qwen35moe -- Forward-Pass Design (Pantheon port)") to facts that do
not come from the oracle itself: closed forms of special contexts, invariants,
and the library attention routine on random inputs.

A plausible slip fails at least one check: a doubled or missing 1/sqrt(256)
scale (two-key weights), the blocked vs. interleaved GQA pairing (distinct KV
heads), a missing or wrong gate (z = 0 halves the output exactly), positions
past the context read (NaN past ctx_len), or a transposed score product.
"""
import math

import numpy as np
import pytest
from scipy.special import expit

B_, HQ, HKV, D = 3, 16, 2, 256


def _inputs(seed, B=B_, L=8):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, HQ, D))
    k = r.standard_normal((B, HKV, L, D))
    v = r.standard_normal((B, HKV, L, D))
    z = r.standard_normal((B, HQ, D))
    return q, k, v, z


def test_attn_single_position_closed_form(orc):
    """One cached position: the softmax weight is 1, so out = v_0 * sigmoid(z)
    for every query head of the group, whatever q and k are."""
    q, k, v, z = _inputs(1, L=4)
    out = orc.attn_decode(q, k, v, np.array([1, 1, 1]), z)
    for b in range(B_):
        for h in range(HQ):
            np.testing.assert_allclose(out[b, h], v[b, h // 8, 0] * expit(z[b, h]), rtol=1e-13, atol=1e-15)


def test_attn_scale_two_keys(orc):
    """Two keys whose scores differ by ln 3 after the 1/sqrt(256) = 1/16 scale:
    q . (k1 - k2) = 16 ln 3 gives weights 3/4 and 1/4 exactly."""
    q = np.zeros((1, HQ, D))
    q[0, :, 5] = 1.0
    k = np.zeros((1, HKV, 2, D))
    k[0, :, 0, 5] = 16.0 * math.log(3.0)
    r = np.random.default_rng(2)
    v = r.standard_normal((1, HKV, 2, D))
    z = r.standard_normal((1, HQ, D))
    out = orc.attn_decode(q, k, v, np.array([2]), z)
    for h in range(HQ):
        g = h // 8
        ref = (0.75 * v[0, g, 0] + 0.25 * v[0, g, 1]) * expit(z[0, h])
        np.testing.assert_allclose(out[0, h], ref, rtol=1e-12, atol=1e-14)


def test_attn_equal_keys_average_values(orc):
    """All keys equal: every weight is 1/L, the output is the mean value row."""
    q, k, v, z = _inputs(3, L=7)
    k[:] = k[:, :, :1]
    out = orc.attn_decode(q, k, v, np.array([7, 3, 5]), z)
    for b, L in enumerate((7, 3, 5)):
        for h in range(HQ):
            ref = v[b, h // 8, :L].mean(axis=0) * expit(z[b, h])
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-14)


def test_attn_gqa_blocked_grouping_and_gate(orc):
    """KV head g holds the constant value row c_g, so any softmax gives c_g; with
    z = 0 the gate is exactly 1/2. Query heads 0..7 must read KV head 0 and 8..15
    KV head 1 (eight query heads share one KV head)."""
    q, k, v, _ = _inputs(4, L=6)
    c = np.random.default_rng(40).standard_normal((HKV, D))
    for g in range(HKV):
        v[:, g] = c[g]
    out = orc.attn_decode(q, k, v, np.array([6, 2, 4]), np.zeros((B_, HQ, D)))
    for h in range(HQ):
        np.testing.assert_allclose(out[:, h], np.broadcast_to(0.5 * c[h // 8], (B_, D)), rtol=1e-12, atol=1e-14)
    assert not np.allclose(c[0], c[1])


def test_attn_invariances(orc):
    """Permuting the cached positions (keys with their values) leaves the output
    unchanged, and so does adding one vector u to every key of a KV head (all
    scores move by q . u / 16)."""
    q, k, v, z = _inputs(5, L=9)
    ctx = np.array([9, 9, 9])
    base = orc.attn_decode(q, k, v, ctx, z)
    perm = np.random.default_rng(50).permutation(9)
    np.testing.assert_allclose(orc.attn_decode(q, k[:, :, perm], v[:, :, perm], ctx, z), base, rtol=1e-11,
                               atol=1e-13)
    u = np.random.default_rng(51).standard_normal((B_, HKV, 1, D))
    np.testing.assert_allclose(orc.attn_decode(q, k + u, v, ctx, z), base, rtol=1e-10, atol=1e-12)


def test_attn_context_length_and_empty(orc):
    """Positions at or past ctx_len are never read (NaN there changes nothing),
    and an empty context gives a zero output."""
    q, k, v, z = _inputs(6, L=10)
    ctx = np.array([4, 0, 10])
    base = orc.attn_decode(q, k, v, ctx, z)
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 4:] = np.nan
    v2[0, :, 4:] = np.nan
    k2[1] = np.nan
    v2[1] = np.nan
    np.testing.assert_array_equal(orc.attn_decode(q, k2, v2, ctx, z), base)
    assert not base[1].any()


def test_attn_matches_library_attention(orc):
    """Random inputs with ragged context lengths against torch's
    scaled_dot_product_attention in fp64 (its default scale is 1/sqrt(256)),
    with each KV head repeated for its eight query heads."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    q, k, v, z = _inputs(7, L=33)
    ctx = [33, 1, 17]
    out = orc.attn_decode(q, k, v, np.array(ctx), z)
    for b, L in enumerate(ctx):
        qt = torch.from_numpy(q[b]).unsqueeze(1)                            # [16, 1, D]
        kt = torch.from_numpy(k[b, :, :L]).repeat_interleave(HQ // HKV, 0)   # [16, L, D]
        vt = torch.from_numpy(v[b, :, :L]).repeat_interleave(HQ // HKV, 0)
        o = F.scaled_dot_product_attention(qt, kt, vt)[:, 0].numpy()
        np.testing.assert_allclose(out[b], o * expit(z[b]), rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------ planted mistakes

def _mutant(kind):
    """The oracle's attention with one plausible mistake planted (CPU only)."""
    def attn(q, kc, vc, ctx_len, z):
        B, Hq, Dd = q.shape
        out = np.zeros((B, Hq, Dd))
        for b in range(B):
            L = int(ctx_len[b]) + (1 if kind == "reads_past_ctx" else 0)
            if L <= 0:
                continue
            for h in range(Hq):
                g = h % 2 if kind == "interleaved_gqa" else h // 8
                s = kc[b, g, :L] @ q[b, h] / (np.sqrt(Dd) if kind != "scale_sqrt_half" else np.sqrt(Dd / 2))
                if kind == "no_scale":
                    s = kc[b, g, :L] @ q[b, h]
                p = np.exp(s - s.max())
                p /= p.sum()
                o = p @ vc[b, g, :L]
                gate = 1.0 if kind == "no_gate" else 1.0 / (1.0 + np.exp(-z[b, h]))
                out[b, h] = o * gate
        return out
    return type("Mutant", (), {"attn_decode": staticmethod(attn)})


PINS = [test_attn_single_position_closed_form, test_attn_scale_two_keys, test_attn_equal_keys_average_values,
        test_attn_gqa_blocked_grouping_and_gate, test_attn_invariances, test_attn_context_length_and_empty,
        test_attn_matches_library_attention]


@pytest.mark.parametrize("kind", ["interleaved_gqa", "no_scale", "scale_sqrt_half", "no_gate", "reads_past_ctx"])
def test_attn_pins_catch_planted_mistakes(kind):
    m = _mutant(kind)
    failed = 0
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(m)
        except (AssertionError, IndexError, ValueError):
            failed += 1
    assert failed > 0, f"no pin caught the planted mistake {kind!r}"
