"""Decode attention of the full-attention layers (gdn_attn_decode, tcgen05)
against the fp64 oracle on the same seeded bf16 inputs.

Tolerance, from the arithmetic. Scores are exact bf16 products summed in fp32
(relative error ~1e-6), and q is scaled by 1/16 exactly. The softmax weights
enter the value product rounded to bf16, each with a relative error
|delta_p| <= 2^-9, and the sum that normalises them is taken over the same
rounded weights. So per output element d
    |o' - o| = |sum_p w_p delta_p (v_p[d] - o[d])| / (1 + sum_p w_p delta_p)
             <= 2^-9 / (1 - 2^-9) * max_p |v_p[d] - o[d]|,
times the gate sigmoid(z) <= 1. On top: fp32 accumulation over up to 4096
positions (slack 1e-4 * max|v|) and, for a bf16 output, its own rounding to
nearest: at most half a unit in the last place, 2^-8 relative. The test checks
every element against that bound.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

from gated_deltanet_linear_02_gb300 import inputs as I
from oracle import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def ops():
    from gated_deltanet_linear_02_gb300 import build, ops
    build.build()
    return ops


def bound(inp, seqs, ref, out_dtype):
    """Per-element error bound for sequences `seqs` (see the module docstring)."""
    q = inp.q.cpu().double().numpy()
    z = inp.z.cpu().double().numpy()
    tol = np.zeros((len(seqs), 16, 256))
    for i, b in enumerate(seqs):
        L = int(min(max(int(inp.ctx_len[b]), 0), inp.k_cache.shape[2]))
        if L == 0:
            continue
        for g in range(2):
            V = inp.v_cache[b, g, :L].cpu().double().numpy()
            for hl in range(8):
                h = 8 * g + hl
                o = ref[i, h] / expit(z[b, h])                    # the ungated output
                spread = np.abs(V - o[None, :]).max(axis=0)
                tol[i, h] = expit(z[b, h]) * (2.0 ** -9 / (1 - 2.0 ** -9) * spread + 1e-4 * np.abs(V).max())
    if out_dtype == torch.bfloat16:
        tol += 2.0 ** -8 * (np.abs(ref) + tol)
    del q
    return tol


def check(ops, inp, seqs=None, out_dtype=torch.float32, label=""):
    B = inp.q.shape[0]
    d = inp.to(DEV) if not inp.q.is_cuda else inp
    out = torch.full((B, 16, 256), float("nan"), dtype=out_dtype, device=DEV)
    ops.attn_decode(d.q, d.k_cache, d.v_cache, d.ctx_len, d.z, out)
    torch.cuda.synchronize()
    assert ops.device_error() == ops.GDN_OK
    seqs = list(range(B)) if seqs is None else list(seqs)
    sel = torch.tensor(seqs)
    cpu = lambda t: t[sel.to(t.device)].cpu()
    ref = oracle.attn_decode(cpu(inp.q), cpu(inp.k_cache), cpu(inp.v_cache), cpu(inp.ctx_len).numpy(), cpu(inp.z))
    got = out[sel.to(DEV)].cpu().double().numpy()
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    tol = bound(inp, seqs, ref, out_dtype)
    err = np.abs(got - ref)
    ratio = (err / np.maximum(tol, 1e-30)).max()
    rel = err.max() / max(np.abs(ref).max(), 1e-30)
    print(f"attn {label}: max|d|/max|ref| = {rel:.2e}, worst element at {ratio:.2f} of its bound")
    assert (err <= tol).all(), f"{label}: {int((err > tol).sum())} elements outside the bound (worst {ratio:.2f}x)"
    return out


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_attn_ragged_small(ops, out_dtype):
    # one full cache, a single position, one position past a tile, a partial first tile
    inp = I.attn_inputs(I.seed_of(20), 4, 300, [300, 1, 129, 77])
    check(ops, inp, out_dtype=out_dtype, label=f"ragged {out_dtype}")


def test_attn_degenerate_lengths(ops):
    # ctx_len 0 gives zeros; values past Lmax or below 0 clamp to [0, Lmax]
    inp = I.attn_inputs(I.seed_of(21), 4, 200, [0, 200, 200, 0])
    inp.ctx_len = torch.tensor([0, 500, 200, -3], dtype=torch.int32)
    out = check(ops, inp, label="degenerate")
    assert not out[0].any() and not out[3].any()


def test_attn_one_tile_blocks(ops):
    # a small batch over a long context: 1-tile blocks, 40 of them per KV head
    inp = I.attn_inputs(I.seed_of(22), 2, 5000, [5000, 2049])
    check(ops, inp, label="B=2 L=5000")


def test_attn_two_tile_blocks_sampled(ops):
    # B = 16 at 16K: 2-tile blocks; sequences sampled for the oracle
    lens = [16384, 16000, 1, 8191, 8193, 300, 16384, 129, 256, 255, 257, 1024, 1023, 1025, 4000, 9999]
    inp = I.attn_inputs(I.seed_of(23), 16, 16384, lens, device=DEV)
    check(ops, inp, seqs=[0, 1, 3, 4, 7, 10, 13], label="B=16 L=16384")


def test_attn_decode_batch_full_size_sampled(ops):
    # the benchmarked step: B = 256 sequences at 4K context, 8-tile blocks;
    # sampled sequences against the oracle, the others only checked finite
    inp = I.attn_inputs(I.seed_of(24), 256, 4096, device=DEV)
    out = check(ops, inp, seqs=[0, 1, 77, 128, 255], label="B=256 L=4096")
    assert torch.isfinite(out).all()


def test_attn_deterministic(ops):
    inp = I.attn_inputs(I.seed_of(25), 3, 1000, [1000, 513, 640]).to(DEV)
    outs = []
    for _ in range(2):
        out = torch.empty(3, 16, 256, device=DEV)
        ops.attn_decode(inp.q, inp.k_cache, inp.v_cache, inp.ctx_len, inp.z, out)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("Lmax,lens", [(1, [1, 0]), (129, [129, 128]), (128, [128, 127])])
def test_attn_tile_edges(ops, Lmax, lens):
    # a one-row cache, a context one position past a tile, and an exact tile
    inp = I.attn_inputs(I.seed_of(26), len(lens), Lmax, lens)
    check(ops, inp, label=f"Lmax={Lmax}")


def test_attn_single_sequence_long_context(ops):
    # one sequence at a 128K-token context: 1-tile blocks, 1024 of them per KV
    # head, merged by the combine kernel 8 blocks at a time
    inp = I.attn_inputs(I.seed_of(27), 1, 131072, [131072 - 77], device=DEV)
    check(ops, inp, label="B=1 L=128K")
