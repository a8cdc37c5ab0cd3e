"""The no-allocation decode entry point, called through the C ABI.

sl8_attn_int8_decode_noalloc is for callers that cannot allocate GPU memory where
they run decode (a fixed memory budget after warm-up, tensors owned by another
framework, a C caller without an allocator).  It keeps its split partials in a
fixed array inside the library instead of caller scratch.  Its output must match
the regular split + combine entry points within the tests' tolerance, on two calls
in a row with different inputs (so stale scratch from the first call cannot leak
into the second), including the largest ordinary case (d = 256, eight query heads
per kv head) and a shape whose automatic split count asks for more partials than the
array holds, so that the entry point has to lower it.  One call is also checked
against the oracle directly.

This file is named to be collected last; it also runs on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
import w8a8_int8_flashattention_gb300 as sl8
from _parity import check_f32, check_half, to_np32

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"
SCRATCH_BYTES = 16 << 20  # SL8_NOALLOC_SCRATCH_BYTES in include/sl8.h


@pytest.fixture(scope="module", autouse=True)
def _built():
    from w8a8_int8_flashattention_gb300 import build
    build.build()
    sl8.lib()


def _cache(wid, B, Hq, Hkv, d, lens, lmax):
    w = W.custom(wid, kind="decode", B=B, Hq=Hq, Hkv=Hkv, d=d, dtype="bf16", extra={"lengths": lens})
    kc = torch.zeros((B, Hkv, lmax, d), dtype=torch.int8, device=DEV)
    vc = torch.zeros_like(kc)
    ks = torch.zeros((B, Hkv, lmax), dtype=torch.float32, device=DEV)
    vs = torch.zeros_like(ks)
    for b, L in enumerate(lens):
        for name, c, s in (("k", kc, ks), ("v", vc, vs)):
            cc, sc = sl8.quant_rowwise(torch.from_numpy(W.decode_cache_values(w, b, name)).to(DEV))
            c[b, :, :L], s[b, :, :L] = cc, sc
    q = W.decode_query(w).to(DEV)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    return q, kc, ks, vc, vs, seq


def _noalloc(q, kc, ks, vc, vs, seq, out):
    B, Hq, d = q.shape
    _, Hkv, Lmax, _ = kc.shape
    return sl8.lib().sl8_attn_int8_decode_noalloc(
        q.data_ptr(), sl8.SL8_BF16, kc.data_ptr(), ks.data_ptr(), vc.data_ptr(), vs.data_ptr(), seq.data_ptr(),
        B, Hq, Hkv, Lmax, d, out.data_ptr(), sl8._DTYPES[out.dtype], torch.cuda.current_stream().cuda_stream)


def test_noalloc_decode_matches_oracle():
    """fp32 and bf16 outputs of the no-allocation decode against the CPU oracle."""
    wid, B, Hq, Hkv, d, lens, lmax = 7101, 3, 8, 2, 128, [900, 1, 333], 900
    q, kc, ks, vc, vs, seq = _cache(wid, B, Hq, Hkv, d, lens, lmax)
    w = W.custom(wid, kind="decode", B=B, Hq=Hq, Hkv=Hkv, d=d, dtype="bf16", extra={"lengths": lens})
    ok = {n: np.zeros((B, Hkv, lmax, d), np.int8) for n in ("k", "v")}
    os_ = {n: np.zeros((B, Hkv, lmax), np.float32) for n in ("k", "v")}
    for b, L in enumerate(lens):
        for n in ("k", "v"):
            ok[n][b, :, :L], os_[n][b, :, :L] = oracle.quant_rowwise(W.decode_cache_values(w, b, n))
    ref = oracle.attn_decode(q.float().cpu().numpy(), ok["k"], os_["k"], ok["v"], os_["v"], np.asarray(lens))
    o32 = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device=DEV)
    ob = torch.zeros((B, Hq, d), dtype=torch.bfloat16, device=DEV)
    for out in (o32, ob):
        rc = _noalloc(q, kc, ks, vc, vs, seq, out)
        assert rc == sl8.SL8_OK, sl8.status_string(rc)
    torch.cuda.synchronize()
    check_f32(to_np32(o32), ref["out"], "noalloc vs oracle f32")
    check_half(ob, ref["out"], "noalloc vs oracle bf16")


def test_noalloc_decode_matches_regular_entry_points():
    cases = [
        # two calls in a row: different caches, lengths and shapes
        (7001, 4, 8, 2, 128, [300, 1, 0, 700], 700),
        (7002, 3, 4, 4, 64, [513, 129, 20], 600),
        # the most partial bytes per SM the automatic split count gives (d = 256, G = 8)
        (7003, 8, 64, 8, 256, [8192, 77, 300, 1, 5, 999, 2048, 17], 8192),
    ]
    for wid, B, Hq, Hkv, d, lens, lmax in cases:
        q, kc, ks, vc, vs, seq = _cache(wid, B, Hq, Hkv, d, lens, lmax)
        ref = sl8.attn_int8_decode(q, kc, ks, vc, vs, seq, out_dtype=torch.float32)
        out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device=DEV)
        rc = _noalloc(q, kc, ks, vc, vs, seq, out)
        assert rc == sl8.SL8_OK, sl8.status_string(rc)
        torch.cuda.synchronize()
        check_f32(to_np32(out), to_np32(ref).astype(np.float64), f"noalloc w{wid}")
        st, site = sl8.last_device_status()
        assert st == sl8.SL8_OK, (st, site)


def test_noalloc_lowers_the_split_count_to_the_array():
    """A shape whose automatic split count needs more partials than the array holds:
    many sequences of one kv head, d = 256, Lmax just above 17 stages of 128 tokens.
    The entry point lowers the count to fit and must still agree with the regular path
    (which uses the full automatic count)."""
    Hq, Hkv, d, lmax = 8, 1, 256, 2200
    floats = SCRATCH_BYTES // 4
    pick = None
    for B in range(150, 1200):
        S = sl8.decode_num_splits(B, Hkv, lmax, d, 0)
        if S > floats // (B * Hq * (d + 1)):
            pick = B
            break
    assert pick is not None, "no shape in the searched range needs lowering on this part"
    B = pick
    rng = np.random.default_rng(7201)
    lens = [int(x) for x in rng.integers(1, lmax + 1, size=B)]
    lens[:4] = [lmax, 2100, 2049, 2150]
    q, kc, ks, vc, vs, seq = _cache(7201, B, Hq, Hkv, d, lens, lmax)
    ref = sl8.attn_int8_decode(q, kc, ks, vc, vs, seq, out_dtype=torch.float32)
    for _ in range(2):
        out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device=DEV)
        rc = _noalloc(q, kc, ks, vc, vs, seq, out)
        assert rc == sl8.SL8_OK, sl8.status_string(rc)
        torch.cuda.synchronize()
        check_f32(to_np32(out), to_np32(ref).astype(np.float64), f"noalloc lowered B={B}")
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_OK, (st, site)


def test_noalloc_refuses_problems_beyond_the_array():
    # one split of B * Hq * (d + 1) fp32 values needs more than the fixed array: refused, no launch
    B, Hq, Hkv, d, L = 1040, 32, 8, 128, 16
    assert B * Hq * (d + 1) * 4 > SCRATCH_BYTES
    q = torch.zeros((B, Hq, d), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((B, Hkv, L, d), dtype=torch.int8, device=DEV)
    ks = torch.ones((B, Hkv, L), dtype=torch.float32, device=DEV)
    seq = torch.full((B,), L, dtype=torch.int32, device=DEV)
    out = torch.zeros((B, Hq, d), dtype=torch.float32, device=DEV)
    assert _noalloc(q, kc, ks, kc, ks, seq, out) == sl8.SL8_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 0)
