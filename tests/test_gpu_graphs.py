"""The hot path inside CUDA graphs: prefill and decode captured once by stream capture
and replayed on new inputs give the same bits as eager calls.

The library makes no allocation, host synchronisation or attribute call on its launch
paths once a kernel has run on the device, so a serving loop can capture a step and
replay it.  Operations: the "SuperL8" README, "Attention kernels" table (attn_int8_fwd,
attn_decode); the "Engine" table lists graphed decode.
"""
import numpy as np
import pytest
import torch

import workloads as W
import w8a8_int8_flashattention_gb300 as sl8

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from w8a8_int8_flashattention_gb300 import build
    build.build()
    sl8.lib()


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                      # eager run on the side stream first
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_prefill_graph_replay():
    w = W.custom(2801, B=1, Hq=8, Hkv=2, N=700, d=128, dtype="bf16", k_bias_std=1.0)
    q, k, v = W.prefill_dense(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    ws = torch.empty(sl8.prefill_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(qd)
    g = _capture(lambda: sl8.attn_int8_fwd(qd, kd, vd, causal=True, smooth_k=True, workspace=ws, out=out))
    for seed in (1, 2):
        gen = torch.Generator(device="cpu").manual_seed(seed)
        qd.copy_(torch.randn(qd.shape, generator=gen).to(torch.bfloat16))
        kd.copy_(torch.randn(kd.shape, generator=gen).to(torch.bfloat16))
        g.replay()
        eager = sl8.attn_int8_fwd(qd, kd, vd, causal=True, smooth_k=True)
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_OK, (st, site)


def test_decode_graph_replay():
    B, Hq, Hkv, d, lmax = 8, 16, 4, 128, 2048
    gen = torch.Generator(device="cpu").manual_seed(3)
    kc = torch.randint(-127, 128, (B, Hkv, lmax, d), generator=gen, dtype=torch.int8).to(DEV)
    vc = torch.randint(-127, 128, (B, Hkv, lmax, d), generator=gen, dtype=torch.int8).to(DEV)
    ks = (torch.rand((B, Hkv, lmax), generator=gen) * 0.05 + 1e-3).to(DEV)
    vs = (torch.rand((B, Hkv, lmax), generator=gen) * 0.05 + 1e-3).to(DEV)
    seq = torch.tensor([1, 100, 500, 1024, 1500, 2040, 7, 640], dtype=torch.int32, device=DEV)
    q = torch.randn((B, Hq, d), generator=gen).to(torch.bfloat16).to(DEV)
    S = sl8.decode_num_splits(B, Hkv, lmax, d, 0)
    op = torch.empty((B, Hq, S, d), dtype=torch.float32, device=DEV)
    lp = torch.empty((B, Hq, S), dtype=torch.float32, device=DEV)
    out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=DEV)
    g = _capture(lambda: sl8.attn_int8_decode(q, kc, ks, vc, vs, seq, o_partial=op, lse_partial=lp, out=out))
    for step in range(3):
        q.copy_(torch.randn((B, Hq, d), generator=gen).to(torch.bfloat16))
        seq.add_(1)                                # one more cached token per step
        g.replay()
        eager = sl8.attn_int8_decode(q, kc, ks, vc, vs, seq)
        torch.cuda.synchronize()
        assert torch.equal(out, eager), step
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_OK, (st, site)


def test_chunk_onto_cache_graph_replay():
    """A serving loop's prefill chunk onto the int8 cache, captured once: replays on new
    queries and a grown cache give the bits of eager calls (the short chunk takes the
    key-split path, so the merge launch is captured too)."""
    B, Hq, Hkv, d, lmax, nq = 1, 8, 2, 128, 2048, 128
    gen = torch.Generator(device="cpu").manual_seed(4)
    kc = torch.randint(-127, 128, (B, Hkv, lmax, d), generator=gen, dtype=torch.int8).to(DEV)
    vc = torch.randint(-127, 128, (B, Hkv, lmax, d), generator=gen, dtype=torch.int8).to(DEV)
    ks = (torch.rand((B, Hkv, lmax), generator=gen) * 0.05 + 1e-3).to(DEV)
    vs = (torch.rand((B, Hkv, lmax), generator=gen) * 0.05 + 1e-3).to(DEV)
    q = torch.randn((B, Hq, nq, d), generator=gen).to(torch.bfloat16).to(DEV)
    nk = 1500
    ws = torch.empty(int(sl8.lib().sl8_attn_int8_fwd_chunk_workspace_size(B, Hq, Hkv, nq, nk, d)), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty_like(q)
    g = _capture(lambda: sl8.attn_int8_fwd_chunk_cache(q, kc, ks, vc, vs, Nk=nk, workspace=ws, out=out))
    for step in range(2):
        q.copy_(torch.randn(q.shape, generator=gen).to(torch.bfloat16))
        vs.mul_(2.0 ** (8 * step + 6))             # V scales grow 2^6, then 2^14 more: a new V exponent
        g.replay()
        eager = sl8.attn_int8_fwd_chunk_cache(q, kc, ks, vc, vs, Nk=nk)
        torch.cuda.synchronize()
        assert torch.equal(out, eager), step
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_OK, (st, site)
