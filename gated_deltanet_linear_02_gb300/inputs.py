"""Seeded synthetic inputs for the Gated-DeltaNet mixer workloads.

This module draws random numbers and nothing else: it holds none of the
mixer's arithmetic, and both the CUDA path and the CPU oracle take their
inputs from here.

The shapes are those of the SSM layers in "qwen35moe -- Forward-Pass Design
(Pantheon port)", section "Config (mini)":
- 32 V-heads and 16 K-heads, both of dimension 128;
- a conv of width 4 over 8192 channels, laid out q(16x128) | k(16x128) |
  v(32x128).

The pages fix no input distribution, and no checkpoint is available, so the
values are synthetic:
- qkv, z, alpha and beta ~ N(0, 1);
- conv weights ~ N(0, 0.25), where 0.25 is the standard deviation;
- A_log ~ U(0, ln 16);
- dt_bias ~ U(-1, 1);
- norm weight = 1 + N(0, 0.1);
- initial SSM state ~ N(0, 0.02);
- initial conv_state ~ N(0, 1).

Activations are drawn in fp32 and rounded once to the activation dtype, so
both sides see the same bits. Each (workload, layer) pair has its own seed.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

HV, HK, DK, DV, KCONV = 32, 16, 128, 128, 4
C_CONV = 2 * HK * DK + HV * DV      # 8192
D_INNER = HV * DV                    # 4096


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


@dataclass
class LayerParams:
    conv_w: torch.Tensor    # [8192, 4] fp32, tap 3 multiplies the current token
    A_log: torch.Tensor     # [32] fp32
    dt_bias: torch.Tensor   # [32] fp32
    norm_w: torch.Tensor    # [128] fp32
    norm_eps: float = 1e-6
    l2_eps: float = 1e-6

    def to(self, device) -> "LayerParams":
        return LayerParams(self.conv_w.to(device), self.A_log.to(device), self.dt_bias.to(device),
                           self.norm_w.to(device), self.norm_eps, self.l2_eps)


def layer_params(seed: int, device="cpu") -> LayerParams:
    g = _gen(seed, device)
    conv_w = torch.randn(C_CONV, KCONV, generator=g, device=device) * 0.25
    A_log = torch.rand(HV, generator=g, device=device) * math.log(16.0)
    dt_bias = torch.rand(HV, generator=g, device=device) * 2.0 - 1.0
    norm_w = 1.0 + 0.1 * torch.randn(DV, generator=g, device=device)
    return LayerParams(conv_w.contiguous(), A_log, dt_bias, norm_w)


@dataclass
class Streams:
    qkv: torch.Tensor     # [T, 8192]
    z: torch.Tensor       # [T, 4096]
    alpha: torch.Tensor   # [T, 32]
    beta: torch.Tensor    # [T, 32]

    def to(self, device) -> "Streams":
        return Streams(self.qkv.to(device), self.z.to(device), self.alpha.to(device),
                       self.beta.to(device))

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.qkv, self.z, self.alpha, self.beta))


def streams(seed: int, T: int, act_dtype=torch.bfloat16, device="cpu", lead=()) -> Streams:
    """Projected streams for T tokens (``lead`` prepends extra leading dims,
    e.g. (steps,) for a decode run: shapes become [*lead, T, ...])."""
    g = _gen(seed + 500_000, device)
    shp = tuple(lead) + (T,)
    qkv = torch.randn(*shp, C_CONV, generator=g, device=device).to(act_dtype)
    z = torch.randn(*shp, D_INNER, generator=g, device=device).to(act_dtype)
    alpha = torch.randn(*shp, HV, generator=g, device=device).to(act_dtype)
    beta = torch.randn(*shp, HV, generator=g, device=device).to(act_dtype)
    return Streams(qkv, z, alpha, beta)


def initial_states(seed: int, N: int, act_dtype=torch.bfloat16, device="cpu", zero=False):
    """(conv_state [N, 3, 8192] act dtype, ssm_state [N, 32, 128(j), 128(i)] fp32).
    The SSM state is stored value-index-major (the transpose of the page's
    S[i][j]); random draws are i.i.d. so the layout does not change the law."""
    if zero:
        return (torch.zeros(N, KCONV - 1, C_CONV, dtype=act_dtype, device=device),
                torch.zeros(N, HV, DV, DK, dtype=torch.float32, device=device))
    g = _gen(seed + 900_000, device)
    conv = torch.randn(N, KCONV - 1, C_CONV, generator=g, device=device).to(act_dtype)
    ssm = torch.randn(N, HV, DV, DK, generator=g, device=device) * 0.02
    return conv, ssm


N_EMBD = 2048                        # output width of the ssm_out projection


def out_proj_weight(seed: int, act_dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """ssm_out.weight [2048][4096] ~ N(0, 1/64) (std), so outputs keep the input
    scale; rounded once to the activation dtype."""
    g = _gen(seed + 800_000, device)
    return (torch.randn(N_EMBD, D_INNER, generator=g, device=device) / 64.0).to(act_dtype)


def in_proj_weights(seed: int, act_dtype=torch.bfloat16, device="cpu"):
    """(attn_qkv [8192][2048], attn_gate [4096][2048], ssm_alpha [32][2048],
    ssm_beta [32][2048]) ~ N(0, 1/2048) (variance), so the projected streams are
    ~N(0, 1) like the synthetic streams; rounded once to the activation dtype."""
    g = _gen(seed + 850_000, device)
    sd = 1.0 / math.sqrt(N_EMBD)
    return tuple((torch.randn(r, N_EMBD, generator=g, device=device) * sd).to(act_dtype)
                 for r in (C_CONV, D_INNER, HV, HV))


ATTN_HQ, ATTN_HKV, ATTN_D = 16, 2, 256   # full-attention layers: 16 query / 2 KV heads, head_dim 256


@dataclass
class AttnInputs:
    q: torch.Tensor          # [B][16][256] bf16
    k_cache: torch.Tensor    # [B][2][Lmax][256] bf16
    v_cache: torch.Tensor    # [B][2][Lmax][256] bf16
    ctx_len: torch.Tensor    # [B] int32
    z: torch.Tensor          # [B][16][256] bf16

    def to(self, device) -> "AttnInputs":
        return AttnInputs(*(t.to(device) for t in (self.q, self.k_cache, self.v_cache, self.ctx_len, self.z)))


def attn_inputs(seed: int, B: int, Lmax: int, ctx_len=None, device="cpu") -> AttnInputs:
    """One decode step of a full-attention layer. q and the cached keys come out
    of per-head RMSNorms (unit RMS per head, then partial RoPE, a rotation), so
    they are drawn N(0, 1) per element; values and the gate logits z too. Rows
    at or past each sequence's ctx_len hold NaN, which the attention must
    never let through. ctx_len defaults to Lmax for every sequence."""
    g = _gen(seed + 950_000, device)
    q = torch.randn(B, ATTN_HQ, ATTN_D, generator=g, device=device).to(torch.bfloat16)
    k = torch.randn(B, ATTN_HKV, Lmax, ATTN_D, generator=g, device=device)
    v = torch.randn(B, ATTN_HKV, Lmax, ATTN_D, generator=g, device=device)
    z = torch.randn(B, ATTN_HQ, ATTN_D, generator=g, device=device).to(torch.bfloat16)
    cl = torch.full((B,), Lmax, dtype=torch.int32) if ctx_len is None else \
        torch.as_tensor(ctx_len, dtype=torch.int32).reshape(B)
    pos = torch.arange(Lmax, device=device)
    past = (pos[None, :] >= cl.to(device)[:, None])[:, None, :, None]
    k = torch.where(past, torch.full_like(k, float("nan")), k)
    v = torch.where(past, torch.full_like(v, float("nan")), v)
    return AttnInputs(q, k.to(torch.bfloat16), v.to(torch.bfloat16), cl.to(device), z)


def varlen_lengths(seed: int, n: int = 8, lo: int = 256, hi: int = 32768) -> list[int]:
    """Sequence lengths drawn log-uniformly in [lo, hi] and rounded."""
    g = _gen(seed + 700_000, "cpu")
    u = torch.rand(n, generator=g, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]


def cu_seqlens(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


# The five workloads (sizes as stated for the benchmark and parity suite).
WORKLOADS = {
    0: dict(name="prefill_T64_fp32", kind="prefill", T=64, B=1, act="f32", zero_state=True),
    1: dict(name="decode_B64_x128_bf16", kind="decode", B=64, steps=128, layers=1, act="bf16"),
    2: dict(name="prefill_T4096_bf16", kind="prefill", T=4096, B=1, act="bf16", zero_state=True,
            chunk=64),
    3: dict(name="decode_30L_B256_x32_bf16", kind="decode", B=256, steps=32, layers=30, act="bf16"),
    4: dict(name="varlen_prefill_8seq_bf16", kind="varlen", n_seq=8, act="bf16", zero_state=False),
}


def seed_of(workload: int, layer: int = 0) -> int:
    return 1000 * int(workload) + int(layer)
