"""Thin ctypes binding of libgdn.so (include/gdn.h), with the same names.

This layer only marshals arguments. It checks the tensors' shapes, dtypes,
devices and contiguity, passes their device pointers and the current CUDA
stream, and turns a non-OK status into ``GdnError``. Every step of the mixer
runs in the library's CUDA kernels. If the library is missing, loading fails
loudly: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import inputs as _inp

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE, GDN_ERR_CUDA, GDN_ERR_TIMEOUT = range(6)
GDN_F32, GDN_BF16 = 0, 1
_DT = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16}

HV, HK, DK, DV, KC, CC, DI = _inp.HV, _inp.HK, _inp.DK, _inp.DV, _inp.KCONV, _inp.C_CONV, _inp.D_INNER
N_EMBD = _inp.N_EMBD


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}" + (f" ({detail})" if detail else ""))


class gdn_params(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("norm_w", ctypes.c_void_p), ("norm_eps", ctypes.c_float), ("l2_eps", ctypes.c_float)]


_lib = None
_vp, _int, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """The loaded libgdn.so. Raises if it has not been built: the mixer has
    no CPU or library fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        L.gdn_conv_step.restype = _int
        L.gdn_conv_step.argtypes = [_vp, _vp, _vp, _vp, _int, _int, _vp]
        L.gdn_decode_step.restype = _int
        L.gdn_decode_step.argtypes = [ctypes.POINTER(gdn_params)] + [_vp] * 7 + [_int, _int, _int, _vp]
        L.gdn_decode_multi.restype = _int
        L.gdn_decode_multi.argtypes = [ctypes.POINTER(gdn_params)] + [_vp] * 7 + [_int, _int, _int, _int, _vp]
        L.gdn_in_proj.restype = _int
        L.gdn_in_proj.argtypes = [_vp] * 6 + [_int, _int, _vp]
        L.gdn_out_proj.restype = _int
        L.gdn_out_proj.argtypes = [_vp, _vp, _vp, _int, _int, _vp]
        L.gdn_in_proj_conv.restype = _int
        L.gdn_in_proj_conv.argtypes = [ctypes.POINTER(gdn_params), _vp, _vp, _vp, _int, _int] + [_vp] * 6 + [_vp]
        L.gdn_prefill_xhat.restype = _int
        L.gdn_prefill_xhat.argtypes = [ctypes.POINTER(gdn_params)] + [_vp] * 5 + [_int, _int] + [_vp] * 3 + \
            [_int, _vp, _sz, _vp]
        L.gdn_gated_out_proj.restype = _int
        L.gdn_gated_out_proj.argtypes = [_vp, ctypes.c_float, _vp, _vp, _vp, _vp, _int, _int, _int, _vp]
        L.gdn_prefill.restype = _int
        L.gdn_prefill.argtypes = [ctypes.POINTER(gdn_params)] + [_vp] * 5 + [_int, _int] + [_vp] * 5 + \
            [_int, _int, _int, _vp, _sz, _vp]
        L.gdn_prefill_static.restype = _int
        L.gdn_prefill_static.argtypes = [ctypes.POINTER(gdn_params)] + [_vp] * 5 + [_int, _int] + [_vp] * 5 + \
            [_int, _int, _int, _vp]
        L.gdn_attn_decode.restype = _int
        L.gdn_attn_decode.argtypes = [_vp] * 6 + [_int, _int, _vp, _sz, _int, _vp]
        L.gdn_attn_decode_workspace_size.restype = _sz
        L.gdn_attn_decode_workspace_size.argtypes = [_int, _int]
        L.gdn_prefill_workspace_size.restype = _sz
        L.gdn_prefill_workspace_size.argtypes = [_int, _int, _int, _int]
        L.gdn_selftest_wait_timeout.restype = _int
        L.gdn_selftest_wait_timeout.argtypes = [_vp]
        L.gdn_device_error.restype = _int
        L.gdn_device_error.argtypes = [_vp]
        L.gdn_get_device_error.restype = _int
        L.gdn_get_device_error.argtypes = [_vp, _vp]
        L.gdn_status_string.restype = ctypes.c_char_p
        L.gdn_status_string.argtypes = [_int]
        L.gdn_last_error.restype = ctypes.c_char_p
        L.gdn_last_error.argtypes = []
        L.gdn_abi_version.restype = _int
        L.gdn_abi_version.argtypes = []
        _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().gdn_status_string(int(s)).decode()


def last_error() -> str:
    return lib().gdn_last_error().decode()


def abi_version() -> int:
    return lib().gdn_abi_version()


def _check(status: int, where: str):
    if status != GDN_OK:
        raise GdnError(status, where, last_error())


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if isinstance(stream, torch.cuda.Stream) else int(stream)


def _ptr(t: torch.Tensor | None, name: str, shape=None, dtype=None, device=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def make_params(p) -> gdn_params:
    """gdn_params from anything with conv_w, A_log, dt_bias, norm_w fp32 CUDA
    tensors and norm_eps, l2_eps floats (e.g. inputs.LayerParams).

    The struct holds raw device pointers, so it also keeps references to the
    four tensors: they stay alive as long as the struct does, even when the
    caller passed a temporary such as ``make_params(lp.to("cuda"))``."""
    cp = gdn_params(_ptr(p.conv_w, "conv_w", (CC, KC), torch.float32),
                    _ptr(p.A_log, "A_log", (HV,), torch.float32),
                    _ptr(p.dt_bias, "dt_bias", (HV,), torch.float32),
                    _ptr(p.norm_w, "norm_w", (DV,), torch.float32),
                    float(p.norm_eps), float(p.l2_eps))
    cp._keep_alive = (p.conv_w, p.A_log, p.dt_bias, p.norm_w)
    return cp


def _act_dtype(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise ValueError(f"activation dtype {t.dtype} unsupported (float32 or bfloat16)")
    return _DT[t.dtype]


def conv_step(conv_w, qkv_in, qkv_out, conv_state, stream=None):
    """gdn_conv_step: qkv_out = SiLU(causal conv(conv_state, qkv_in)); conv_state shifts."""
    B = qkv_in.shape[0]
    act = _act_dtype(qkv_in)
    st = lib().gdn_conv_step(_ptr(conv_w, "conv_w", (CC, KC), torch.float32),
                             _ptr(qkv_in, "qkv_in", (B, CC)), _ptr(qkv_out, "qkv_out", (B, CC), qkv_in.dtype),
                             _ptr(conv_state, "conv_state", (B, KC - 1, CC), qkv_in.dtype), B, act,
                             _stream(stream))
    _check(st, "gdn_conv_step")


def decode_step(params, qkv, z, alpha, beta, conv_state, ssm_state, out, stream=None,
                cparams: gdn_params | None = None):
    """gdn_decode_step: one token for B sequences, states updated in place."""
    B = qkv.shape[0]
    dt = qkv.dtype
    act = _act_dtype(qkv)
    od = _act_dtype(out)
    cp = cparams if cparams is not None else make_params(params)
    st = lib().gdn_decode_step(ctypes.byref(cp), _ptr(qkv, "qkv", (B, CC)), _ptr(z, "z", (B, DI), dt),
                               _ptr(alpha, "alpha", (B, HV), dt), _ptr(beta, "beta", (B, HV), dt),
                               _ptr(conv_state, "conv_state", (B, KC - 1, CC), dt),
                               _ptr(ssm_state, "ssm_state", (B, HV, DV, DK), torch.float32),
                               _ptr(out, "out", (B, DI)), B, act, od, _stream(stream))
    _check(st, "gdn_decode_step")


def decode_multi(params, qkv, z, alpha, beta, conv_state, ssm_state, out, stream=None,
                 cparams: gdn_params | None = None):
    """gdn_decode_multi: T consecutive tokens for each of B sequences (qkv
    [B][T][8192]), states updated in place."""
    B, T = qkv.shape[0], qkv.shape[1]
    dt = qkv.dtype
    act = _act_dtype(qkv)
    od = _act_dtype(out)
    cp = cparams if cparams is not None else make_params(params)
    st = lib().gdn_decode_multi(ctypes.byref(cp), _ptr(qkv, "qkv", (B, T, CC)), _ptr(z, "z", (B, T, DI), dt),
                                _ptr(alpha, "alpha", (B, T, HV), dt), _ptr(beta, "beta", (B, T, HV), dt),
                                _ptr(conv_state, "conv_state", (B, KC - 1, CC), dt),
                                _ptr(ssm_state, "ssm_state", (B, HV, DV, DK), torch.float32),
                                _ptr(out, "out", (B, T, DI)), B, T, act, od, _stream(stream))
    _check(st, "gdn_decode_multi")


IN_PROJ_ROWS = CC + DI + 2 * HV   # GDN_IN_PROJ_ROWS


def in_proj(h, w_in, qkv, z, alpha, beta, stream=None):
    """gdn_in_proj: the four input projections of the normed hidden states h
    [M][2048] (bf16) through the stacked weight w_in [12352][2048] (bf16), into
    qkv [M][8192], z [M][4096], alpha [M][32], beta [M][32] (fp32 or bf16)."""
    M = h.shape[0]
    act = _act_dtype(qkv)
    dt = qkv.dtype
    st = lib().gdn_in_proj(_ptr(h, "h", (M, N_EMBD), torch.bfloat16),
                           _ptr(w_in, "w_in", (IN_PROJ_ROWS, N_EMBD), torch.bfloat16),
                           _ptr(qkv, "qkv", (M, CC)), _ptr(z, "z", (M, DI), dt), _ptr(alpha, "alpha", (M, HV), dt),
                           _ptr(beta, "beta", (M, HV), dt), M, act, _stream(stream))
    _check(st, "gdn_in_proj")


def out_proj(x, w, y, stream=None):
    """gdn_out_proj: y = x w^T on the tensor cores (x [M][4096] bf16, w
    [2048][4096] bf16, y [M][2048] fp32 or bf16)."""
    M = x.shape[0]
    od = _act_dtype(y)
    st = lib().gdn_out_proj(_ptr(x, "x", (M, DI), torch.bfloat16), _ptr(w, "w", (N_EMBD, DI), torch.bfloat16),
                            _ptr(y, "y", (M, N_EMBD)), M, od, _stream(stream))
    _check(st, "gdn_out_proj")


def in_proj_conv(params, h, w_in, cu_seqlens, xhat, z, alpha, beta, conv_state_in=None, conv_state_out=None,
                 stream=None, cparams: gdn_params | None = None):
    """gdn_in_proj_conv: the input projections with the conv, SiLU and q/k L2
    norms in the GEMM's epilogue (h [M][2048] bf16, w_in [12352][2048] bf16)
    into xhat [M][8192] fp16, z [M][4096], alpha/beta [M][32] bf16, and
    conv_state_out [N][3][8192] bf16."""
    M = h.shape[0]
    N = cu_seqlens.shape[0] - 1
    cp = cparams if cparams is not None else make_params(params)
    st = lib().gdn_in_proj_conv(ctypes.byref(cp), _ptr(h, "h", (M, N_EMBD), torch.bfloat16),
                                _ptr(w_in, "w_in", (IN_PROJ_ROWS, N_EMBD), torch.bfloat16),
                                _ptr(cu_seqlens, "cu_seqlens", (N + 1,), torch.int32), N, M,
                                _ptr(conv_state_in, "conv_state_in", (N, KC - 1, CC), torch.bfloat16),
                                _ptr(conv_state_out, "conv_state_out", (N, KC - 1, CC), torch.bfloat16),
                                _ptr(xhat, "xhat", (M, CC), torch.float16), _ptr(z, "z", (M, DI), torch.bfloat16),
                                _ptr(alpha, "alpha", (M, HV), torch.bfloat16), _ptr(beta, "beta", (M, HV), torch.bfloat16),
                                _stream(stream))
    _check(st, "gdn_in_proj_conv")


def prefill_xhat(params, xhat, z, alpha, beta, cu_seqlens, out, ssm_state_in=None, ssm_state_out=None,
                 workspace=None, stream=None, cparams: gdn_params | None = None):
    """gdn_prefill_xhat: the chunked prefill from gdn_in_proj_conv's activations.
    Allocates the workspace through torch when none is given."""
    T = xhat.shape[0]
    N = cu_seqlens.shape[0] - 1
    if workspace is None:
        workspace = torch.empty(max(prefill_workspace_size(N, T, torch.bfloat16, 64), 256), dtype=torch.uint8,
                                device=xhat.device)
    cp = cparams if cparams is not None else make_params(params)
    st = lib().gdn_prefill_xhat(ctypes.byref(cp), _ptr(xhat, "xhat", (T, CC), torch.float16),
                                _ptr(z, "z", (T, DI), torch.bfloat16), _ptr(alpha, "alpha", (T, HV), torch.bfloat16),
                                _ptr(beta, "beta", (T, HV), torch.bfloat16),
                                _ptr(cu_seqlens, "cu_seqlens", (N + 1,), torch.int32), N, T,
                                _ptr(ssm_state_in, "ssm_state_in", (N, HV, DV, DK), torch.float32),
                                _ptr(ssm_state_out, "ssm_state_out", (N, HV, DV, DK), torch.float32),
                                _ptr(out, "out", (T, DI)), _act_dtype(out), _ptr(workspace, "workspace"),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "gdn_prefill_xhat")
    return workspace


def gated_out_proj(norm_w, norm_eps, y, z, w, out, stream=None):
    """gdn_gated_out_proj: out = (gated RMSNorm(y) . silu(z)) w^T in one
    tensor-core GEMM. y and z [M][4096] in the same dtype (fp32 or bf16; y is
    the mixer's output with the norm left out), norm_w [128] fp32, w
    [2048][4096] bf16, out [M][2048] fp32 or bf16."""
    M = y.shape[0]
    act = _act_dtype(y)
    st = lib().gdn_gated_out_proj(_ptr(norm_w, "norm_w", (DV,), torch.float32), float(norm_eps),
                                  _ptr(y, "y", (M, DI)), _ptr(z, "z", (M, DI), y.dtype),
                                  _ptr(w, "w", (N_EMBD, DI), torch.bfloat16), _ptr(out, "out", (M, N_EMBD)),
                                  M, act, _act_dtype(out), _stream(stream))
    _check(st, "gdn_gated_out_proj")


ATTN_HQ, ATTN_HKV, ATTN_D = 16, 2, 256   # GDN_ATTN_Q_HEADS, GDN_ATTN_KV_HEADS, GDN_ATTN_HEAD_DIM


def attn_decode_workspace_size(B: int, Lmax: int) -> int:
    return int(lib().gdn_attn_decode_workspace_size(int(B), int(Lmax)))


def attn_decode(q, k_cache, v_cache, ctx_len, z, out, workspace=None, stream=None):
    """gdn_attn_decode: one decode step of GQA attention (16 query / 2 KV heads,
    head_dim 256) with the sigmoid output gate. q, z [B][16][256] bf16; caches
    [B][2][Lmax][256] bf16; ctx_len [B] int32; out [B][16][256] fp32 or bf16.
    Allocates the workspace through torch when none is given."""
    B = q.shape[0]
    Lmax = k_cache.shape[2] if k_cache.dim() == 4 else 0
    od = _act_dtype(out)
    need = attn_decode_workspace_size(B, Lmax) if B > 0 else 0
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().gdn_attn_decode(_ptr(q, "q", (B, ATTN_HQ, ATTN_D), torch.bfloat16),
                               _ptr(k_cache, "k_cache", (B, ATTN_HKV, Lmax, ATTN_D), torch.bfloat16),
                               _ptr(v_cache, "v_cache", (B, ATTN_HKV, Lmax, ATTN_D), torch.bfloat16),
                               _ptr(ctx_len, "ctx_len", (B,), torch.int32),
                               _ptr(z, "z", (B, ATTN_HQ, ATTN_D), torch.bfloat16),
                               _ptr(out, "out", (B, ATTN_HQ, ATTN_D)), B, Lmax, _ptr(workspace, "workspace"),
                               workspace.numel() * workspace.element_size(), od, _stream(stream))
    _check(st, "gdn_attn_decode")
    return workspace


def prefill_workspace_size(N: int, T_total: int, act=torch.bfloat16, chunk_size: int = 0) -> int:
    return int(lib().gdn_prefill_workspace_size(int(N), int(T_total), _DT[act], int(chunk_size)))


def prefill(params, qkv, z, alpha, beta, cu_seqlens, out, conv_state_in=None, conv_state_out=None,
            ssm_state_in=None, ssm_state_out=None, chunk_size: int = 0, workspace=None, stream=None,
            cparams: gdn_params | None = None):
    """gdn_prefill over N packed sequences (cu_seqlens: int32 CUDA [N+1]).
    Allocates the workspace through torch when none is given."""
    T = qkv.shape[0]
    N = cu_seqlens.shape[0] - 1
    dt = qkv.dtype
    act = _act_dtype(qkv)
    od = _act_dtype(out)
    need = prefill_workspace_size(N, T, dt, chunk_size)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=qkv.device)
    cp = cparams if cparams is not None else make_params(params)
    st = lib().gdn_prefill(ctypes.byref(cp), _ptr(qkv, "qkv", (T, CC)), _ptr(z, "z", (T, DI), dt),
                           _ptr(alpha, "alpha", (T, HV), dt), _ptr(beta, "beta", (T, HV), dt),
                           _ptr(cu_seqlens, "cu_seqlens", (N + 1,), torch.int32), N, T,
                           _ptr(conv_state_in, "conv_state_in", (N, KC - 1, CC), dt),
                           _ptr(conv_state_out, "conv_state_out", (N, KC - 1, CC), dt),
                           _ptr(ssm_state_in, "ssm_state_in", (N, HV, DV, DK), torch.float32),
                           _ptr(ssm_state_out, "ssm_state_out", (N, HV, DV, DK), torch.float32),
                           _ptr(out, "out", (T, DI)), act, od, int(chunk_size),
                           _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                           _stream(stream))
    _check(st, "gdn_prefill")
    return workspace


def device_error(stream=None) -> int:
    """Synchronises the stream, then reads and clears the library's device error
    word: GDN_OK, or GDN_ERR_TIMEOUT if a bounded device-side wait gave up."""
    return lib().gdn_device_error(_stream(stream))


def selftest_wait_timeout(stream=None) -> None:
    """gdn_selftest_wait_timeout: enqueue the kernel whose bounded wait runs
    out (about 2 s); the next device_error() then reports GDN_ERR_TIMEOUT."""
    _check(lib().gdn_selftest_wait_timeout(_stream(stream)), "gdn_selftest_wait_timeout")


def static_scratch_bytes() -> int:
    """Bytes of the fixed scratch gdn_prefill_static uses, from the library."""
    L = lib()
    L.gdn_static_scratch_bytes.restype = _sz
    L.gdn_static_scratch_bytes.argtypes = []
    return int(L.gdn_static_scratch_bytes())


DECODE_MAX_T = 8   # GDN_DECODE_MAX_T: tokens per sequence of gdn_decode_multi, at most


def prefill_static(params, qkv, z, alpha, beta, cu_seqlens, out, conv_state_in=None, conv_state_out=None,
                   ssm_state_in=None, ssm_state_out=None, chunk_size: int = 0, stream=None,
                   cparams: gdn_params | None = None):
    """gdn_prefill_static: gdn_prefill without a workspace argument, for callers
    that cannot allocate device memory. The library's fixed 64 MiB device
    scratch is used instead, shared by every call on the device."""
    T = qkv.shape[0]
    N = cu_seqlens.shape[0] - 1
    dt = qkv.dtype
    cp = cparams if cparams is not None else make_params(params)
    st = lib().gdn_prefill_static(ctypes.byref(cp), _ptr(qkv, "qkv", (T, CC)), _ptr(z, "z", (T, DI), dt),
                                  _ptr(alpha, "alpha", (T, HV), dt), _ptr(beta, "beta", (T, HV), dt),
                                  _ptr(cu_seqlens, "cu_seqlens", (N + 1,), torch.int32), N, T,
                                  _ptr(conv_state_in, "conv_state_in", (N, KC - 1, CC), dt),
                                  _ptr(conv_state_out, "conv_state_out", (N, KC - 1, CC), dt),
                                  _ptr(ssm_state_in, "ssm_state_in", (N, HV, DV, DK), torch.float32),
                                  _ptr(ssm_state_out, "ssm_state_out", (N, HV, DV, DK), torch.float32),
                                  _ptr(out, "out", (T, DI)), _act_dtype(qkv), _act_dtype(out), int(chunk_size),
                                  _stream(stream))
    _check(st, "gdn_prefill_static")
