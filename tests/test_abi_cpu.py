"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/sl8.h declares, and rejects bad arguments
synchronously, before anything is launched."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import w8a8_int8_flashattention_gb300 as sl8
from w8a8_int8_flashattention_gb300 import build as sl8_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sl8_build.build()
    return sl8.lib()


def test_exports_every_header_function(lib):
    names = sl8.header_functions()
    assert len(names) >= 19
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding declares a signature for each of them
    assert set(names) == set(sl8._SIGNATURES)


def test_exported_symbols_are_only_the_abi(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", sl8.LIB_PATH], capture_output=True, text=True).stdout
    sl8_syms = sorted(set(re.findall(r"\b(sl8_[a-z0-9_]+)\b", out)))
    assert sl8_syms == sl8.header_functions()


def test_status_strings_and_version(lib):
    assert lib.sl8_status_string(0) == b"ok"
    assert b"workspace" in lib.sl8_status_string(3)
    assert lib.sl8_status_string(99) == b"unknown status"
    assert lib.sl8_version() >= 100


def test_workspace_sizes(lib):
    # dense: codes for Q and K (bf16) + scales + table; grows with N and heads
    a = lib.sl8_attn_int8_fwd_workspace_size(1, 32, 8, 4096, 128, 0)
    assert a >= 32 * 4096 * 128 * 2 + 8 * 4096 * 128 * 2
    assert lib.sl8_attn_int8_fwd_workspace_size(1, 32, 8, 4097, 128, 0) > a
    # varlen bound: total tokens + 127 per sequence of padding
    v = lib.sl8_attn_int8_fwd_workspace_size(32, 64, 8, 3000, 128, 48000)
    assert v >= (48000 + 32 * 127) // 128 * 128 * 72 * 128 * 2 * 0.99
    assert lib.sl8_attn_int8_fwd_workspace_size(-1, 32, 8, 4096, 128, 0) == 0
    assert lib.sl8_k_channel_mean_workspace_size(2, 8, 8192, 256) > 0


def test_decode_split_plan(lib):
    # The decode kernel streams the cache in stages of 160 tokens for d = 128 (ten
    # compute warps x 16 tokens).  Explicit requests: split size = ceil(Lmax / n) rounded
    # up to whole stages (to 16 tokens below one stage).
    stage = 160
    assert lib.sl8_attn_decode_num_splits(64, 8, 8192, 128, 5) == 5
    assert lib.sl8_attn_decode_split_size(64, 8, 8192, 128, 5) == 1760
    assert lib.sl8_attn_decode_split_size(2, 2, 600, 128, 4) == 160
    assert lib.sl8_attn_decode_num_splits(2, 2, 600, 128, 3) == 2       # 200 -> 320 tokens
    assert lib.sl8_attn_decode_split_size(2, 2, 300, 128, 3) == 112
    assert lib.sl8_attn_decode_num_splits(64, 8, 8192, 128, 1) == 1
    assert lib.sl8_attn_decode_num_splits(1, 1, 10, 128, 64) == 1       # one 16-token split
    assert lib.sl8_attn_decode_num_splits(64, 8, 100, 96, 0) == 0       # unsupported head dim
    # head dim 32: the same 160-token stages
    assert lib.sl8_attn_decode_split_size(64, 8, 8192, 32, 5) == 1760
    assert lib.sl8_attn_decode_num_splits(0, 8, 100, 128, 0) == 0
    # every plan: 16-token aligned splits (whole stages from one stage up), all non-empty
    # at Lmax, covering Lmax, and the combine's split size (from Lmax and S alone) is the
    # split kernel's
    for B, Hkv in ((1, 1), (64, 8), (3, 2)):
        for lmax in range(1, 3000, 37):
            for n in (0, 1, 3, 40, 500):
                S = lib.sl8_attn_decode_num_splits(B, Hkv, lmax, 128, n)
                ss = lib.sl8_attn_decode_split_size(B, Hkv, lmax, 128, n)
                assert S >= 1 and ss % 16 == 0 and ss * S >= lmax and (S - 1) * ss < lmax
                per = -(-lmax // S)
                step = stage if per >= stage else 16
                assert ss == (per + step - 1) // step * step
                if n == 0:
                    assert S <= -(-lmax // stage)


def _host_buf(nbytes):
    # 16-byte aligned host memory: only used for argument checks that fail before any access
    raw = np.zeros(nbytes + 32, np.uint8)
    off = (-raw.ctypes.data) % 16
    return raw, raw.ctypes.data + off


def test_prefill_argument_errors(lib):
    keep, p = _host_buf(1 << 12)
    f = lib.sl8_attn_int8_fwd
    # (q, k, v, qk_dtype, v_dtype, B, Hq, Hkv, N, d, cu, T, causal, smooth, out, out_dtype, lse, ws, ws_bytes, stream)
    base = [p, p, p, sl8.SL8_BF16, sl8.SL8_BF16, 1, 4, 2, 128, 128, None, 0, 1, 1, p, sl8.SL8_BF16, None, p, 16, None]

    def call(**kw):
        args = list(base)
        idx = dict(q=0, k=1, v=2, qk=3, vdt=4, B=5, Hq=6, Hkv=7, N=8, d=9, out=14, odt=15, ws=17, wsb=18)
        for k, val in kw.items():
            args[idx[k]] = val
        return f(*args)

    assert call(q=None) == sl8.SL8_ERR_INVALID_ARG
    assert call(q=p + 2) == sl8.SL8_ERR_INVALID_ARG           # misaligned
    assert call(Hkv=3) == sl8.SL8_ERR_INVALID_ARG             # Hq % Hkv != 0
    assert call(d=32) == sl8.SL8_ERR_WORKSPACE               # head dim 32 is accepted (runs as 64)
    assert call(d=96) == sl8.SL8_ERR_UNSUPPORTED
    assert call(d=16) == sl8.SL8_ERR_UNSUPPORTED
    assert call(qk=sl8.SL8_F32) == sl8.SL8_ERR_INVALID_ARG
    assert call(odt=sl8.SL8_F16) == sl8.SL8_ERR_INVALID_ARG   # out must be V's dtype or F32
    assert call(ws=None) == sl8.SL8_ERR_WORKSPACE
    assert call(wsb=16) == sl8.SL8_ERR_WORKSPACE
    assert call(B=0) == sl8.SL8_OK                            # empty: nothing to do
    assert call(N=0) == sl8.SL8_OK


def test_chunk_cache_argument_errors(lib):
    keep, p = _host_buf(1 << 12)
    f = lib.sl8_attn_int8_fwd_chunk_cache
    # (q, q_dtype, k_cache, k_scale, v_cache, v_scale, B, Hq, Hkv, Nq, Nk, Lmax, d, causal, out, out_dtype, lse,
    #  ws, ws_bytes, stream)
    base = [p, sl8.SL8_BF16, p, p, p, p, 1, 4, 2, 16, 64, 64, 128, 1, p, sl8.SL8_BF16, None, p, 16, None]

    def call(**kw):
        args = list(base)
        idx = dict(q=0, qdt=1, kc=2, ks=3, vc=4, vs=5, B=6, Hq=7, Hkv=8, Nq=9, Nk=10, Lmax=11, d=12, out=14, odt=15,
                   ws=17, wsb=18)
        for k, val in kw.items():
            args[idx[k]] = val
        return f(*args)

    assert call(kc=None) == sl8.SL8_ERR_INVALID_ARG
    assert call(vs=None) == sl8.SL8_ERR_INVALID_ARG
    assert call(vc=p + 4) == sl8.SL8_ERR_INVALID_ARG          # misaligned cache
    assert call(Hkv=3) == sl8.SL8_ERR_INVALID_ARG             # Hq % Hkv != 0
    assert call(Nq=65) == sl8.SL8_ERR_INVALID_ARG             # Nq > Nk
    assert call(Nk=65) == sl8.SL8_ERR_INVALID_ARG             # Nk > Lmax
    assert call(qdt=sl8.SL8_F32) == sl8.SL8_ERR_INVALID_ARG   # q must be fp16 or bf16
    assert call(odt=sl8.SL8_F32) == sl8.SL8_ERR_WORKSPACE     # any output dtype (F16, BF16, F32)
    assert call(d=96) == sl8.SL8_ERR_UNSUPPORTED
    assert call(d=32) == sl8.SL8_ERR_WORKSPACE               # head dim 32 is accepted (runs as 64)
    assert call(ws=None) == sl8.SL8_ERR_WORKSPACE
    assert call(B=0) == sl8.SL8_OK                            # empty: nothing to do
    assert call(Nq=0) == sl8.SL8_OK


def test_w8a8_argument_errors(lib):
    keep, p = _host_buf(1 << 12)
    f = lib.sl8_attn_w8a8_fwd
    # (..., causal, smooth, q_group, k_group, ratio, out, out_dtype, lse, ws, ws_bytes, stream)
    base = [p, p, p, sl8.SL8_BF16, sl8.SL8_BF16, 1, 4, 2, 128, 128, None, 0, 1, 1, 32, 32, 4.0, p, sl8.SL8_BF16,
            None, p, 16, None]

    def call(**kw):
        args = list(base)
        idx = dict(gq=14, gk=15, tau=16, wsb=21)
        for k, val in kw.items():
            args[idx[k]] = val
        return f(*args)

    assert call() == sl8.SL8_ERR_WORKSPACE                    # valid groups reach the workspace check
    for g in (0, 3, 48, 128, -32):
        assert call(gq=g) == sl8.SL8_ERR_INVALID_ARG
        assert call(gk=g) == sl8.SL8_ERR_INVALID_ARG
    for g in (1, 2, 64):
        assert call(gq=g, gk=g) == sl8.SL8_ERR_WORKSPACE
    assert call(tau=-1.0) == sl8.SL8_ERR_INVALID_ARG
    assert call(tau=float("nan")) == sl8.SL8_ERR_INVALID_ARG
    assert call(tau=float("inf")) == sl8.SL8_ERR_INVALID_ARG
    assert call(tau=0.0) == sl8.SL8_ERR_WORKSPACE
    d = lib.sl8_attn_w8a8_qk_logits_debug
    assert d(p, p, sl8.SL8_BF16, 1, 4, 2, 128, 128, None, 0, 1, 5, 32, 4.0, 0, 1, p, None, None, None, None, p, 16,
             None) == sl8.SL8_ERR_INVALID_ARG


def test_decode_and_quant_argument_errors(lib):
    keep, p = _host_buf(1 << 12)
    f = lib.sl8_attn_int8_decode_splitkv
    ok_args = [p, sl8.SL8_BF16, p, p, p, p, p, 64, 32, 8, 8192, 128, 0, p, p, None]
    a = list(ok_args); a[0] = None
    assert f(*a) == sl8.SL8_ERR_INVALID_ARG
    a = list(ok_args); a[8] = 30; a[9] = 4                   # Hq not a multiple of Hkv
    assert f(*a) == sl8.SL8_ERR_INVALID_ARG
    vf = lib.sl8_attn_int8_decode_verify                     # verify: Hq/Hkv = 16 > 8 is refused
    assert vf(p, sl8.SL8_BF16, p, p, p, p, p, p, 4, 64, 64, 4, 8192, 128, 0, p, p, p, sl8.SL8_BF16, None,
              None) == sl8.SL8_ERR_UNSUPPORTED
    a = list(ok_args); a[11] = 80
    assert f(*a) == sl8.SL8_ERR_UNSUPPORTED
    a = list(ok_args); a[7] = 0
    assert f(*a) == sl8.SL8_OK
    q = lib.sl8_quant_rowwise
    assert q(None, sl8.SL8_F32, 4, 4, 4, None, 0, p, p, None) == sl8.SL8_ERR_INVALID_ARG
    assert q(p, sl8.SL8_I8, 4, 4, 4, None, 0, p, p, None) == sl8.SL8_ERR_INVALID_ARG
    assert q(p, sl8.SL8_F32, 4, 4, 2, None, 0, p, p, None) == sl8.SL8_ERR_INVALID_ARG  # stride < cols
    assert q(p, sl8.SL8_F32, 4, 4, 4, p, 0, p, p, None) == sl8.SL8_ERR_INVALID_ARG    # group size 0
    assert q(p, sl8.SL8_F32, 0, 4, 4, None, 0, p, p, None) == sl8.SL8_OK
    c = lib.sl8_attn_decode_combine
    assert c(p, p, p, 2, 4, 100, 128, 0, p, sl8.SL8_BF16, None, None) == sl8.SL8_ERR_INVALID_ARG
    assert c(p, p, p, 2, 4, 100, 128, 1, p, sl8.SL8_I8, None, None) == sl8.SL8_ERR_INVALID_ARG


def test_spin_limit_knob(lib):
    old = sl8.get_spin_limit_ns()
    sl8.set_spin_limit_ns(12345)
    assert sl8.get_spin_limit_ns() == 12345
    sl8.set_spin_limit_ns(old)


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(4, 64)
    with pytest.raises(ValueError):
        sl8.quant_rowwise(x)


def test_oracle_builds_independently():
    import oracle
    path = oracle.build()
    assert os.path.exists(path)
    # the oracle shares no code with the library: no include of csrc or the ABI header
    src = open(os.path.join(ROOT, "oracle", "sl8_oracle.c")).read()
    assert "csrc" not in src and "sl8.h" not in src
    for f in os.listdir(os.path.join(ROOT, "w8a8_int8_flashattention_gb300", "csrc")):
        assert "oracle" not in open(os.path.join(ROOT, "w8a8_int8_flashattention_gb300", "csrc", f)).read().lower()


def test_page_table_and_paginate_round_trip():
    import workloads as W
    w = W.custom(3301, kind="decode", B=4, Hq=4, Hkv=2, d=64, extra={"lengths": [0, 17, 64, 100]})
    lens = W.seq_lengths(w)
    table, num_pages = W.page_table(w, lens, 16, max_blocks=8, spare=2)
    need = (lens + 15) // 16
    assert num_pages == int(need.sum()) + 2
    used = np.concatenate([table[b, :need[b]] for b in range(4)])
    assert len(set(used.tolist())) == len(used) and used.min() >= 0 and used.max() < num_pages
    assert all(np.all(table[b, need[b]:] == -1) for b in range(4))
    rng = np.random.default_rng(5)
    cache = rng.integers(-127, 128, size=(4, 2, 128, 64)).astype(np.int8)
    scales = rng.uniform(0.01, 1.0, size=(4, 2, 128)).astype(np.float32)
    pages, spages = W.paginate(cache, scales, table, lens, 16, num_pages)
    for b in range(4):
        for t in range(int(lens[b])):
            np.testing.assert_array_equal(pages[table[b, t // 16], :, t % 16], cache[b, :, t])
            np.testing.assert_array_equal(spages[table[b, t // 16], :, t % 16], scales[b, :, t])
    shared, _ = W.page_table(w, lens, 16, max_blocks=8, shared_prefix=1)
    assert shared[2, 0] == shared[0, 0] or lens[0] == 0


def test_decode_workspace_size(lib):
    """The decode scratch query: o_partial [B,Hq,S,d] fp32 at 0, lse_partial [B,Hq,S] fp32
    at a 256-byte aligned offset after it, for the effective split count S."""
    for B, Hq, Hkv, lmax, d, n in ((64, 32, 8, 8192, 128, 0), (64, 32, 8, 8192, 128, 5), (3, 4, 4, 1024, 64, 7),
                                   (2, 16, 2, 2000, 256, 0), (1, 1, 1, 10, 128, 64)):
        S = lib.sl8_attn_decode_num_splits(B, Hkv, lmax, d, n)
        assert S >= 1
        off = lib.sl8_attn_decode_lse_offset(B, Hq, Hkv, lmax, d, n)
        size = lib.sl8_attn_decode_workspace_size(B, Hq, Hkv, lmax, d, n)
        o_bytes = B * Hq * S * d * 4
        assert off % 256 == 0 and o_bytes <= off < o_bytes + 256
        assert size == off + B * Hq * S * 4
    # invalid or unsupported shapes size to 0
    assert lib.sl8_attn_decode_workspace_size(64, 30, 8, 8192, 128, 0) == 0   # Hq % Hkv != 0
    assert lib.sl8_attn_decode_workspace_size(64, 32, 8, 8192, 96, 0) == 0    # head dim
    assert lib.sl8_attn_decode_workspace_size(0, 32, 8, 8192, 128, 0) == 0
    assert lib.sl8_attn_decode_workspace_size(4, 32, 8, 0, 128, 0) == 0
