"""The C ABI without a GPU.

These tests check that libgdn.so loads and exports every function
include/gdn.h declares, and that the host-side argument checks reject bad
calls before any CUDA work. No call here reaches the device: every case
fails a check first, which the status and message confirm.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def ops():
    from gated_deltanet_linear_02_gb300 import build, ops
    build.build()
    return ops


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(gdn_[a-z_0-9]+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gdn_conv_step", "gdn_decode_step", "gdn_decode_multi", "gdn_prefill", "gdn_prefill_workspace_size",
              "gdn_in_proj", "gdn_out_proj", "gdn_attn_decode", "gdn_attn_decode_workspace_size",
              "gdn_selftest_wait_timeout",
              "gdn_device_error", "gdn_get_device_error", "gdn_status_string", "gdn_last_error", "gdn_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(ops):
    L = ops.lib()
    for n in declared_functions():
        assert hasattr(L, n), f"{n} declared in gdn.h but not exported by libgdn.so"


def test_exports_are_c_symbols(ops):
    # extern "C": the dynamic symbol table holds the plain names (no C++ mangling)
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", ops.LIB_PATH], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in declared_functions():
        assert n in syms


def test_version_and_status_strings(ops):
    assert ops.abi_version() == 1
    assert ops.status_string(ops.GDN_OK) == "GDN_OK"
    assert ops.status_string(ops.GDN_ERR_TIMEOUT) == "GDN_ERR_TIMEOUT"
    assert ops.status_string(99) == "GDN_STATUS_UNKNOWN"


def test_workspace_size_arithmetic(ops):
    L = ops.lib()
    # per-token bytes of the exact scan path: x (8192) + gates (64) + y (4096) fp32, plus a 256 B header
    for T in (0, 1, 64, 4096):
        body = 4 * (8192 + 64 + 4096) * T
        assert L.gdn_prefill_workspace_size(1, T, ops.GDN_F32, 1) == 256 + ((body + 255) // 256) * 256
    assert L.gdn_prefill_workspace_size(-1, 10, ops.GDN_F32, 1) == 0
    assert L.gdn_prefill_workspace_size(1, -1, ops.GDN_F32, 1) == 0
    assert L.gdn_prefill_workspace_size(1, 10, 7, 1) == 0
    assert L.gdn_prefill_workspace_size(1, 10, ops.GDN_F32, 3) == 0
    assert L.gdn_prefill_workspace_size(70000, 10, ops.GDN_F32, 1) == 0


def test_chunked_workspace_is_bounded(ops):
    """The chunked form runs the packed tokens in windows, so its default
    workspace stops growing with the prompt: one sequence of 4096 tokens, of
    32768 tokens and of 2^24 tokens all get the size of one 4096-token window.
    Shorter prompts get less, and the size grows with N only through the
    per-sequence tables (at most one 4096-token window's worth of sequences)."""
    L = ops.lib()
    a = L.gdn_prefill_workspace_size(1, 4096, ops.GDN_BF16, 64)
    assert a == L.gdn_prefill_workspace_size(1, 32768, ops.GDN_BF16, 64)
    assert a == L.gdn_prefill_workspace_size(1, 1 << 24, ops.GDN_BF16, 64)
    assert L.gdn_prefill_workspace_size(1, 64, ops.GDN_BF16, 64) < L.gdn_prefill_workspace_size(1, 1000, ops.GDN_BF16, 64) < a
    assert L.gdn_prefill_workspace_size(8, 70264, ops.GDN_BF16, 64) == L.gdn_prefill_workspace_size(8, 4096, ops.GDN_BF16, 64)
    assert L.gdn_prefill_workspace_size(65535, 1 << 20, ops.GDN_BF16, 64) == \
        L.gdn_prefill_workspace_size(4096, 1 << 20, ops.GDN_BF16, 64)
    # one 4096-token window: 64 chunks x 32 V-heads of 72 KiB operand blobs
    # (144 MiB), 64 MiB of fp16 activations, 32 MiB of fp16 y, the gate records
    # and the tables
    assert 240 << 20 < a < 256 << 20


FAKE = 0x10000          # 16-byte aligned, never dereferenced: every case fails a host check first
MIS = 0x10004           # misaligned


def _params(ops, **kw):
    p = ops.gdn_params(FAKE, FAKE, FAKE, FAKE, 1e-6, 1e-6)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_decode_argument_checks(ops):
    L = ops.lib()
    p = _params(ops)
    ok_args = [FAKE] * 7
    call = lambda pp, args, B, act=ops.GDN_BF16, od=ops.GDN_F32: L.gdn_decode_step(
        ctypes.byref(pp) if pp is not None else None, *args, B, act, od, None)
    assert call(p, ok_args, 0) == ops.GDN_OK                                # empty batch: no-op
    assert call(p, ok_args, -1) == ops.GDN_ERR_INVALID_ARG
    assert call(p, ok_args, 65536) == ops.GDN_ERR_INVALID_ARG
    assert call(None, ok_args, 4) == ops.GDN_ERR_INVALID_ARG
    assert "params" in ops.last_error()
    assert call(p, ok_args, 4, act=5) == ops.GDN_ERR_INVALID_ARG
    for i in range(7):
        bad = list(ok_args)
        bad[i] = 0
        assert call(p, bad, 4) == ops.GDN_ERR_INVALID_ARG
        bad[i] = MIS
        assert call(p, bad, 4) == ops.GDN_ERR_INVALID_ARG
    assert call(_params(ops, conv_w=MIS), ok_args, 4) == ops.GDN_ERR_INVALID_ARG
    assert call(_params(ops, norm_eps=-1.0), ok_args, 4) == ops.GDN_ERR_INVALID_ARG
    assert call(_params(ops, l2_eps=float("nan")), ok_args, 4) == ops.GDN_ERR_INVALID_ARG


def test_decode_multi_argument_checks(ops):
    L = ops.lib()
    p = _params(ops)
    ok_args = [FAKE] * 7
    call = lambda pp, args, B, T, act=ops.GDN_BF16, od=ops.GDN_F32: L.gdn_decode_multi(
        ctypes.byref(pp) if pp is not None else None, *args, B, T, act, od, None)
    assert call(p, ok_args, 0, 4) == ops.GDN_OK                             # empty batch: no-op
    assert call(p, ok_args, 0, 0) == ops.GDN_ERR_INVALID_ARG                # T checked even then
    assert call(p, ok_args, 4, 0) == ops.GDN_ERR_INVALID_ARG
    assert call(p, ok_args, 4, ops.DECODE_MAX_T + 1) == ops.GDN_ERR_INVALID_ARG
    assert "T out of range" in ops.last_error()
    assert call(p, ok_args, -1, 2) == ops.GDN_ERR_INVALID_ARG
    assert call(p, ok_args, 65536, 2) == ops.GDN_ERR_INVALID_ARG
    assert call(None, ok_args, 4, 2) == ops.GDN_ERR_INVALID_ARG
    assert call(p, ok_args, 4, 2, od=7) == ops.GDN_ERR_INVALID_ARG
    for i in range(7):
        bad = list(ok_args)
        bad[i] = 0
        assert call(p, bad, 4, 2) == ops.GDN_ERR_INVALID_ARG
        bad[i] = MIS
        assert call(p, bad, 4, 2) == ops.GDN_ERR_INVALID_ARG


def test_in_proj_argument_checks(ops):
    L = ops.lib()
    assert L.gdn_in_proj(*([FAKE] * 6), 0, ops.GDN_BF16, None) == ops.GDN_OK      # empty: no-op
    assert L.gdn_in_proj(*([FAKE] * 6), -1, ops.GDN_BF16, None) == ops.GDN_ERR_INVALID_ARG
    assert L.gdn_in_proj(*([FAKE] * 6), 4, 3, None) == ops.GDN_ERR_INVALID_ARG
    for i in range(6):
        args = [FAKE] * 6
        args[i] = 0
        assert L.gdn_in_proj(*args, 4, ops.GDN_BF16, None) == ops.GDN_ERR_INVALID_ARG
        args[i] = MIS
        assert L.gdn_in_proj(*args, 4, ops.GDN_BF16, None) == ops.GDN_ERR_INVALID_ARG


def test_out_proj_argument_checks(ops):
    L = ops.lib()
    assert L.gdn_out_proj(FAKE, FAKE, FAKE, 0, ops.GDN_BF16, None) == ops.GDN_OK      # empty: no-op
    assert L.gdn_out_proj(FAKE, FAKE, FAKE, -1, ops.GDN_BF16, None) == ops.GDN_ERR_INVALID_ARG
    assert L.gdn_out_proj(FAKE, FAKE, FAKE, (1 << 24) + 1, ops.GDN_BF16, None) == ops.GDN_ERR_INVALID_ARG
    assert L.gdn_out_proj(FAKE, FAKE, FAKE, 4, 9, None) == ops.GDN_ERR_INVALID_ARG
    for i in range(3):
        args = [FAKE, FAKE, FAKE]
        args[i] = 0
        assert L.gdn_out_proj(*args, 4, ops.GDN_F32, None) == ops.GDN_ERR_INVALID_ARG
        args[i] = MIS
        assert L.gdn_out_proj(*args, 4, ops.GDN_F32, None) == ops.GDN_ERR_INVALID_ARG


def test_attn_decode_argument_checks(ops):
    L = ops.lib()
    ws = L.gdn_attn_decode_workspace_size(256, 4096)
    # 256 sequences x 2 KV heads x 4 blocks of 1024 positions, each 8 x 256 outputs + 8 (max, sum) pairs
    assert ws == 256 * 2 * 4 * (8 * 256 + 16) * 4
    assert L.gdn_attn_decode_workspace_size(1, 300) == 2 * 3 * (8 * 256 + 16) * 4   # small batch: 1-tile blocks
    assert L.gdn_attn_decode_workspace_size(0, 10) == 0 and L.gdn_attn_decode_workspace_size(3, 0) == 0
    assert L.gdn_attn_decode_workspace_size(3, 1 << 28) == 0                        # B * 2 * Lmax > 2^30

    def call(q=FAKE, k=FAKE, v=FAKE, cl=FAKE, z=FAKE, out=FAKE, B=4, Lmax=64, w=FAKE, wb=1 << 30, od=1):
        return L.gdn_attn_decode(q, k, v, cl, z, out, B, Lmax, w, wb, od, None)

    assert call(B=0) == ops.GDN_OK                                        # empty: no-op
    assert call(B=-1) == ops.GDN_ERR_INVALID_ARG
    assert call(B=65536) == ops.GDN_ERR_INVALID_ARG
    assert call(Lmax=0) == ops.GDN_ERR_INVALID_ARG
    assert call(B=3, Lmax=1 << 28) == ops.GDN_ERR_INVALID_ARG
    assert call(od=7) == ops.GDN_ERR_INVALID_ARG
    for name in ("q", "k", "v", "z", "out"):
        assert call(**{name: 0}) == ops.GDN_ERR_INVALID_ARG
        assert call(**{name: MIS}) == ops.GDN_ERR_INVALID_ARG
    assert call(cl=0) == ops.GDN_ERR_INVALID_ARG
    assert call(cl=FAKE + 2) == ops.GDN_ERR_INVALID_ARG
    assert call(w=0) == ops.GDN_ERR_WORKSPACE
    assert call(wb=L.gdn_attn_decode_workspace_size(4, 64) - 1) == ops.GDN_ERR_WORKSPACE


def test_conv_step_argument_checks(ops):
    L = ops.lib()
    assert L.gdn_conv_step(FAKE, FAKE, FAKE + 16, FAKE + 32, 0, ops.GDN_BF16, None) == ops.GDN_OK
    assert L.gdn_conv_step(FAKE, FAKE, FAKE, FAKE + 32, 3, ops.GDN_BF16, None) == ops.GDN_ERR_INVALID_ARG
    assert L.gdn_conv_step(None, FAKE, FAKE + 16, FAKE + 32, 3, ops.GDN_BF16, None) == ops.GDN_ERR_INVALID_ARG
    assert L.gdn_conv_step(FAKE, FAKE, FAKE + 16, FAKE + 32, 3, 2, None) == ops.GDN_ERR_INVALID_ARG


def test_prefill_argument_checks(ops):
    L = ops.lib()
    p = _params(ops)

    def call(N=2, T=100, chunk=1, act=ops.GDN_F32, ws=FAKE, ws_bytes=1 << 40, cu=FAKE, ins=(None,) * 4,
             streams=(FAKE,) * 4, out=FAKE, pp=p):
        return L.gdn_prefill(ctypes.byref(pp), *streams, cu, N, T, *ins, out, act, ops.GDN_F32, chunk, ws,
                             ws_bytes, None)

    assert call(N=0, T=0) == ops.GDN_OK
    assert call(N=0, T=5) == ops.GDN_ERR_INVALID_ARG
    assert call(N=-1) == ops.GDN_ERR_INVALID_ARG
    assert call(T=-1) == ops.GDN_ERR_INVALID_ARG
    assert call(T=(1 << 24) + 1) == ops.GDN_ERR_INVALID_ARG
    assert call(N=65536) == ops.GDN_ERR_INVALID_ARG
    assert call(chunk=7) == ops.GDN_ERR_UNSUPPORTED
    assert call(cu=None) == ops.GDN_ERR_INVALID_ARG
    assert call(out=MIS) == ops.GDN_ERR_INVALID_ARG
    assert call(out=None) == ops.GDN_ERR_INVALID_ARG
    assert call(streams=(FAKE, None, FAKE, FAKE)) == ops.GDN_ERR_INVALID_ARG
    assert call(ins=(MIS, None, None, None)) == ops.GDN_ERR_INVALID_ARG
    assert call(ws=None) == ops.GDN_ERR_WORKSPACE
    assert call(ws=FAKE + 16) == ops.GDN_ERR_WORKSPACE          # not 256-byte aligned
    need = L.gdn_prefill_workspace_size(2, 100, ops.GDN_F32, 1)
    assert call(ws_bytes=need - 1) == ops.GDN_ERR_WORKSPACE
    assert "workspace" in ops.last_error()


def test_binding_refuses_cpu_tensors(ops):
    import torch
    from gated_deltanet_linear_02_gb300 import inputs
    lp = inputs.layer_params(1)
    with pytest.raises(ValueError):
        ops.make_params(lp)           # CPU tensors: the binding only passes device memory


def test_gated_out_proj_argument_checks_host(ops):
    L = ops.lib()
    call = lambda ptrs, M, act=ops.GDN_BF16, od=ops.GDN_F32, eps=1e-6: L.gdn_gated_out_proj(
        ptrs[0], ctypes.c_float(eps), *ptrs[1:], M, act, od, None)
    ok = [FAKE] * 5                     # norm_w, y, z, w, out
    assert call(ok, 0) == ops.GDN_OK                                          # M == 0: no-op
    assert call(ok, -1) == ops.GDN_ERR_INVALID_ARG
    assert call(ok, (1 << 24) + 1) == ops.GDN_ERR_INVALID_ARG
    assert call(ok, 4, act=2) == ops.GDN_ERR_INVALID_ARG
    assert call(ok, 4, od=9) == ops.GDN_ERR_INVALID_ARG
    assert call(ok, 4, eps=-1.0) == ops.GDN_ERR_INVALID_ARG
    for i in range(5):
        for badp in (0, MIS):
            bad = list(ok)
            bad[i] = badp
            assert call(bad, 4) == ops.GDN_ERR_INVALID_ARG


def test_in_proj_conv_argument_checks(ops):
    L = ops.lib()
    p = _params(ops)
    # h, w_in, cu | N, M | cs_in, cs_out, xhat, z, alpha, beta
    call = lambda pp, head, N, M, tail: L.gdn_in_proj_conv(
        ctypes.byref(pp) if pp is not None else None, *head, N, M, *tail, None)
    head, tail = [FAKE] * 3, [None, None] + [FAKE] * 4
    assert call(p, head, 0, 0, tail) == ops.GDN_OK                            # no sequences: no-op
    assert call(p, head, 0, 5, tail) == ops.GDN_ERR_INVALID_ARG
    assert call(p, head, -1, 0, tail) == ops.GDN_ERR_INVALID_ARG
    assert call(p, head, 2, -1, tail) == ops.GDN_ERR_INVALID_ARG
    assert call(None, head, 2, 8, tail) == ops.GDN_ERR_INVALID_ARG
    assert call(_params(ops, conv_w=MIS), head, 2, 8, tail) == ops.GDN_ERR_INVALID_ARG
    assert call(_params(ops, l2_eps=-1.0), head, 2, 8, tail) == ops.GDN_ERR_INVALID_ARG
    for i in range(3):
        bad = list(head)
        bad[i] = 0
        assert call(p, bad, 2, 8, tail) == ops.GDN_ERR_INVALID_ARG
    for i in range(2, 6):
        bad = list(tail)
        bad[i] = MIS
        assert call(p, head, 2, 8, bad) == ops.GDN_ERR_INVALID_ARG
    bad = list(tail)
    bad[0] = MIS                                                              # a misaligned state
    assert call(p, head, 2, 8, bad) == ops.GDN_ERR_INVALID_ARG
    same = [FAKE, FAKE] + [FAKE] * 4                                          # in and out states overlap
    assert call(p, head, 2, 8, same) == ops.GDN_ERR_INVALID_ARG
    assert "overlap" in ops.last_error()


def test_prefill_xhat_argument_checks(ops):
    L = ops.lib()
    p = _params(ops)
    # xhat, z, alpha, beta, cu | N, T | S_in, S_out, out | out_dt, ws, ws_bytes
    call = lambda pp, five, N, T, three, od=ops.GDN_F32, ws=FAKE * 16, wsb=1 << 30: L.gdn_prefill_xhat(
        ctypes.byref(pp) if pp is not None else None, *five, N, T, *three, od, ws, wsb, None)
    five, three = [FAKE] * 5, [None, None, FAKE]
    assert call(p, five, 0, 0, three) == ops.GDN_OK                           # no sequences: no-op
    assert call(p, five, 0, 3, three) == ops.GDN_ERR_INVALID_ARG
    assert call(p, five, 1, -1, three) == ops.GDN_ERR_INVALID_ARG
    assert call(p, five, 1, 64, three, od=4) == ops.GDN_ERR_INVALID_ARG
    assert call(None, five, 1, 64, three) == ops.GDN_ERR_INVALID_ARG
    for i in range(5):
        bad = list(five)
        bad[i] = 0
        assert call(p, bad, 1, 64, three) == ops.GDN_ERR_INVALID_ARG
    assert call(p, five, 1, 64, [MIS, None, FAKE]) == ops.GDN_ERR_INVALID_ARG
    assert call(p, five, 1, 64, three, ws=None) == ops.GDN_ERR_WORKSPACE
    assert call(p, five, 1, 64, three, wsb=1024) == ops.GDN_ERR_WORKSPACE
    assert call(p, five, 1, 64, three, ws=FAKE * 16 + 16) == ops.GDN_ERR_WORKSPACE   # not 256-byte aligned
