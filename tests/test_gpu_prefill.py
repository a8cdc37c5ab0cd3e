"""GPU parity of the W8A8 INT8 prefill against the CPU oracle, through the C ABI.

Operation: the "SuperL8" README, "Attention kernels" table (attn_int8_fwd: causal
GQA/MQA prefill at head dims 64/128/256; attn_varlen_fwd: ragged prefill) and its
"Quick start" layouts.  Bit-exact: int8 codes, scales, K means and int32 logits;
outputs within the tolerances of tests/_parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
import w8a8_int8_flashattention_gb300 as sl8
from _parity import check_f32, check_half, sample_rows, to_np32

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from w8a8_int8_flashattention_gb300 import build
    build.build()
    sl8.lib()


def _np(t):
    return t.float().numpy()


def _status_ok():
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_OK, f"device status {st} at site {site}"


# ------------------------------------------------------------------ codes and logits

CODE_CASES = [
    # wid, B, Hq, Hkv, N, d, dtype, smooth, k_bias, outlier
    (2001, 1, 4, 2, 256, 64, "f16", True, 0.0, 0.01),
    (2002, 2, 4, 1, 300, 128, "bf16", True, 2.0, 0.0),
    (2003, 1, 2, 2, 200, 256, "bf16", True, 0.0, 0.0),
    (2004, 1, 8, 8, 129, 128, "bf16", False, 0.0, 0.0),
    (2005, 1, 2, 1, 1, 64, "bf16", True, 1.0, 0.0),
    (2006, 1, 4, 2, 200, 32, "bf16", True, 1.0, 0.0),
    (2007, 2, 2, 1, 129, 32, "f16", False, 0.0, 0.0),
]


@pytest.mark.parametrize("case", CODE_CASES, ids=[f"w{c[0]}_N{c[4]}_d{c[5]}" for c in CODE_CASES])
def test_codes_scales_logits_bit_exact(case):
    wid, B, Hq, Hkv, N, d, dt, smooth, bias, outl = case
    w = W.custom(wid, B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, dtype=dt, k_bias_std=bias, k_outlier_frac=outl)
    q, k, v = W.prefill_dense(w)
    res = sl8.attn_int8_qk_logits_debug(q.to(DEV), k.to(DEV), smooth_k=smooth)
    torch.cuda.synchronize()
    _status_ok()
    ref = oracle.attn_prefill(_np(q), _np(k), _np(v), causal=False, smooth_k=smooth,
                              rows=[(b, h, i) for b in range(B) for h in range(Hq) for i in range(N)],
                              want_logits=True)
    np.testing.assert_array_equal(res["q_codes"].cpu().numpy(), ref["q_codes"])
    np.testing.assert_array_equal(res["q_scales"].cpu().numpy(), ref["q_scales"])
    np.testing.assert_array_equal(res["k_codes"].cpu().numpy(), ref["k_codes"])
    np.testing.assert_array_equal(res["k_scales"].cpu().numpy(), ref["k_scales"])
    lg = res["logits"].cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            want = np.stack([ref["logits"][(b, h, i)] for i in range(N)])
            np.testing.assert_array_equal(lg[b, h], want)


def test_k_mean_bit_exact_dense_and_varlen():
    w = W.custom(2010, B=2, Hq=2, Hkv=2, N=300, d=128, dtype="bf16", k_bias_std=3.0)
    q, k, v = W.prefill_dense(w)
    mu = sl8.k_channel_mean(k.to(DEV)).cpu().numpy()
    for b in range(2):
        for h in range(2):
            np.testing.assert_array_equal(mu[b, h], oracle.k_channel_mean(_np(k[b, h])))
    wv = W.custom(2011, kind="varlen", B=4, Hq=2, Hkv=2, d=64, dtype="f16", k_bias_std=1.0,
                  extra={"lengths": [1, 64, 65, 200]})
    qv, kv, vv, cu = W.prefill_varlen(wv)
    muv = sl8.k_channel_mean(kv.to(DEV), cu.to(DEV), max_seqlen=200).cpu().numpy()
    c = cu.numpy()
    for s in range(4):
        for h in range(2):
            np.testing.assert_array_equal(muv[s, h], oracle.k_channel_mean(_np(kv[c[s]:c[s + 1], h])))


# ------------------------------------------------------------------ outputs, small shapes

OUT_CASES = [
    # wid, B, Hq, Hkv, N, d, dtype, causal, smooth, k_bias
    (2101, 1, 4, 2, 256, 64, "f16", True, True, 0.0),
    (2102, 1, 4, 2, 256, 64, "f16", True, False, 0.0),
    (2103, 2, 8, 2, 300, 128, "bf16", True, True, 2.0),
    (2104, 1, 4, 4, 200, 256, "bf16", True, True, 0.0),
    (2105, 1, 8, 1, 129, 64, "bf16", False, True, 0.0),
    (2106, 1, 2, 2, 1, 128, "bf16", True, True, 0.0),
    (2107, 1, 2, 1, 17, 128, "bf16", True, True, 0.0),
    (2108, 1, 2, 1, 127, 128, "bf16", True, True, 0.0),
    (2109, 1, 2, 1, 128, 128, "bf16", True, True, 0.0),
    (2110, 1, 4, 1, 255, 128, "bf16", False, False, 0.0),
    (2111, 1, 2, 2, 384, 256, "f16", False, True, 1.0),
    (2112, 1, 4, 2, 300, 32, "f16", True, True, 1.0),
    (2113, 2, 8, 2, 129, 32, "bf16", True, True, 0.0),
    (2114, 1, 2, 2, 200, 32, "bf16", False, False, 0.0),
]


@pytest.mark.parametrize("case", OUT_CASES, ids=[f"w{c[0]}_N{c[4]}_d{c[5]}_{'c' if c[7] else 'nc'}" for c in OUT_CASES])
def test_prefill_outputs_small(case):
    wid, B, Hq, Hkv, N, d, dt, causal, smooth, bias = case
    w = W.custom(wid, B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, dtype=dt, k_bias_std=bias)
    q, k, v = W.prefill_dense(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o32, lse = sl8.attn_int8_fwd(qd, kd, vd, causal=causal, smooth_k=smooth, out_dtype=torch.float32,
                                 return_lse=True)
    oh = sl8.attn_int8_fwd(qd, kd, vd, causal=causal, smooth_k=smooth)
    torch.cuda.synchronize()
    _status_ok()
    ref = oracle.attn_prefill(_np(q), _np(k), _np(v), causal=causal, smooth_k=smooth)
    check_f32(to_np32(o32), ref["out"], f"w{wid} f32")
    check_half(oh, ref["out"], f"w{wid} {dt}")
    np.testing.assert_allclose(to_np32(lse), ref["lse"], rtol=0, atol=1e-4)
    if causal:
        # row 0 sees only key 0: its output is v_0 exactly (up to the output rounding)
        g = Hq // Hkv
        for h in range(Hq):
            assert torch.equal(oh[:, h, 0].cpu(), v[:, h // g, 0]), f"row 0 of head {h} is not v_0"


def test_tiny_workload_all_rows():
    w = W.get("tiny")
    q, k, v = W.prefill_dense(w)
    for smooth in (True, False):
        o32 = sl8.attn_int8_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, smooth_k=smooth,
                                out_dtype=torch.float32)
        oh = sl8.attn_int8_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, smooth_k=smooth)
        torch.cuda.synchronize()
        ref = oracle.attn_prefill(_np(q), _np(k), _np(v), causal=True, smooth_k=smooth)
        check_f32(to_np32(o32), ref["out"], f"tiny smooth={smooth}")
        check_half(oh, ref["out"], f"tiny fp16 smooth={smooth}")
    _status_ok()


def test_varlen_small():
    w = W.custom(2201, kind="varlen", B=6, Hq=8, Hkv=2, d=128, dtype="bf16", k_bias_std=1.0,
                 extra={"lengths": [1, 17, 130, 256, 3, 300]})
    q, k, v, cu = W.prefill_varlen(w)
    o32, lse = sl8.attn_int8_fwd(q.to(DEV), k.to(DEV), v.to(DEV), cu_seqlens=cu.to(DEV), max_seqlen=300,
                                 out_dtype=torch.float32, return_lse=True)
    oh = sl8.attn_int8_fwd(q.to(DEV), k.to(DEV), v.to(DEV), cu_seqlens=cu.to(DEV), max_seqlen=300)
    torch.cuda.synchronize()
    _status_ok()
    ref = oracle.attn_prefill(_np(q), _np(k), _np(v), causal=True, smooth_k=True, cu_seqlens=cu.numpy())
    check_f32(to_np32(o32), ref["out"], "varlen f32")
    check_half(oh, ref["out"], "varlen bf16")
    np.testing.assert_allclose(to_np32(lse), ref["lse"], rtol=0, atol=1e-4)


def test_varlen_head_dim_32():
    """Head dim 32 (run as 64 with zero channels) on ragged sequences."""
    w = W.custom(2202, kind="varlen", B=4, Hq=4, Hkv=2, d=32, dtype="bf16", k_bias_std=1.0,
                 extra={"lengths": [1, 130, 77, 256]})
    q, k, v, cu = W.prefill_varlen(w)
    o32, lse = sl8.attn_int8_fwd(q.to(DEV), k.to(DEV), v.to(DEV), cu_seqlens=cu.to(DEV), max_seqlen=256,
                                 out_dtype=torch.float32, return_lse=True)
    torch.cuda.synchronize()
    _status_ok()
    ref = oracle.attn_prefill(_np(q), _np(k), _np(v), causal=True, smooth_k=True, cu_seqlens=cu.numpy())
    check_f32(to_np32(o32), ref["out"], "varlen d32 f32")
    np.testing.assert_allclose(to_np32(lse), ref["lse"], rtol=0, atol=1e-4)


def test_deterministic_bytes():
    w = W.custom(2301, B=1, Hq=8, Hkv=2, N=700, d=128, dtype="bf16", k_bias_std=2.0)
    q, k, v = (t.to(DEV) for t in W.prefill_dense(w))
    a = sl8.attn_int8_fwd(q, k, v)
    b = sl8.attn_int8_fwd(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_guard_canaries_untouched():
    """Outputs are written exactly inside their bounds: canaries around out stay intact."""
    w = W.custom(2302, B=1, Hq=4, Hkv=2, N=130, d=64, dtype="bf16")
    q, k, v = (t.to(DEV) for t in W.prefill_dense(w))
    n = q.numel()
    buf = torch.full((n + 2048,), 12345, dtype=torch.int16, device=DEV)
    out = buf[1024:1024 + n].view(torch.bfloat16).view(q.shape)
    sl8.attn_int8_fwd(q, k, v, out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:1024] == 12345) and torch.all(buf[1024 + n:] == 12345)


# ------------------------------------------------------------------ full-size workloads (sampled rows)

@pytest.mark.parametrize("name", ["qwen3_8b", "gemma3_d256"])
def test_full_size_dense_workload(name):
    w = W.get(name)
    q, k, v = W.prefill_dense(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o32 = sl8.attn_int8_fwd(qd, kd, vd, causal=True, smooth_k=w.smooth_k, out_dtype=torch.float32)
    oh = sl8.attn_int8_fwd(qd, kd, vd, causal=True, smooth_k=w.smooth_k)
    dbg = sl8.attn_int8_qk_logits_debug(qd, kd, smooth_k=w.smooth_k, row_begin=w.N - 64, row_end=w.N)
    torch.cuda.synchronize()
    _status_ok()
    rng = np.random.default_rng(7)
    rows = sample_rows(rng, [w.N] * w.B, w.Hq, per_head=6)
    logit_rows = [(b, h, i) for b in range(w.B) for h in range(0, w.Hq, max(1, w.Hq // 4))
                  for i in range(w.N - 64, w.N, 16)]
    ref = oracle.attn_prefill(_np(q), _np(k), _np(v), causal=True, smooth_k=w.smooth_k, rows=rows)
    np.testing.assert_array_equal(dbg["q_codes"].cpu().numpy(), ref["q_codes"])
    np.testing.assert_array_equal(dbg["k_codes"].cpu().numpy(), ref["k_codes"])
    np.testing.assert_array_equal(dbg["q_scales"].cpu().numpy(), ref["q_scales"])
    np.testing.assert_array_equal(dbg["k_scales"].cpu().numpy(), ref["k_scales"])
    sel = np.zeros(q.shape[:-1], bool)
    for (b, h, i) in rows:
        sel[b, h, i] = True
    refo = np.where(sel[..., None], ref["out"], np.nan)
    check_f32(to_np32(o32), refo, f"{name} f32")
    check_half(oh, refo, f"{name} bf16")
    lref = oracle.attn_prefill(_np(q), _np(k), _np(v), causal=False, smooth_k=w.smooth_k, rows=logit_rows,
                               want_logits=True)
    lg = dbg["logits"].cpu().numpy()
    for (b, h, i) in logit_rows:
        np.testing.assert_array_equal(lg[b, h, i - (w.N - 64)], lref["logits"][(b, h, i)])


def test_full_size_varlen_workload():
    w = W.get("varlen")
    q, k, v, cu = W.prefill_varlen(w)
    lens = np.diff(cu.numpy())
    o32 = sl8.attn_int8_fwd(q.to(DEV), k.to(DEV), v.to(DEV), cu_seqlens=cu.to(DEV), max_seqlen=int(lens.max()),
                            out_dtype=torch.float32)
    oh = sl8.attn_int8_fwd(q.to(DEV), k.to(DEV), v.to(DEV), cu_seqlens=cu.to(DEV), max_seqlen=int(lens.max()))
    torch.cuda.synchronize()
    _status_ok()
    rng = np.random.default_rng(8)
    rows = sample_rows(rng, lens, w.Hq, per_head=2, edge=False)
    rows += [(s, h, i) for s in (0, len(lens) - 1) for h in (0, w.Hq - 1) for i in range(min(3, lens[s]))]
    ref = oracle.attn_prefill(_np(q), _np(k), _np(v), causal=True, smooth_k=True, cu_seqlens=cu.numpy(), rows=rows)
    check_f32(to_np32(o32), ref["out"], "varlen full f32")
    check_half(oh, ref["out"], "varlen full bf16")


# ------------------------------------------------------------------ query chunks (Nq < Nk)

CHUNK_CASES = [
    # wid, B, Hq, Hkv, Nq, Nk, d, dtype, causal
    (2601, 1, 4, 2, 100, 700, 64, "f16", True),
    (2602, 2, 4, 1, 128, 300, 128, "bf16", True),
    (2603, 1, 8, 4, 1, 513, 128, "bf16", True),
    (2604, 1, 2, 2, 200, 200, 256, "bf16", True),
    (2605, 1, 4, 2, 300, 777, 256, "bf16", True),
    (2606, 1, 4, 4, 70, 400, 128, "bf16", False),
    (2607, 2, 8, 2, 257, 1000, 128, "bf16", True),
    (2608, 1, 4, 2, 100, 333, 32, "f16", True),
]


@pytest.mark.parametrize("case", CHUNK_CASES, ids=[f"w{c[0]}_Nq{c[4]}_Nk{c[5]}_d{c[6]}" for c in CHUNK_CASES])
def test_prefill_query_chunk(case):
    """A chunk of the last Nq queries against Nk keys (bottom-right alignment) against the
    oracle, and against the rows Nk-Nq.. of the full prefill computed by the same library."""
    wid, B, Hq, Hkv, Nq, Nk, d, dt, causal = case
    w = W.custom(wid, B=B, Hq=Hq, Hkv=Hkv, N=Nk, d=d, dtype=dt, k_bias_std=1.0)
    q, k, v = W.prefill_dense(w)
    qc = q[:, :, Nk - Nq:].contiguous()
    o32, lse = sl8.attn_int8_fwd_chunk(qc.to(DEV), k.to(DEV), v.to(DEV), causal=causal, smooth_k=True,
                                       out_dtype=torch.float32, return_lse=True)
    oh = sl8.attn_int8_fwd_chunk(qc.to(DEV), k.to(DEV), v.to(DEV), causal=causal, smooth_k=True)
    full = sl8.attn_int8_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, smooth_k=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    _status_ok()
    ref = oracle.attn_prefill(_np(qc), _np(k), _np(v), causal=causal, smooth_k=True)
    check_f32(to_np32(o32), ref["out"], f"w{wid} chunk f32")
    check_half(oh, ref["out"], f"w{wid} chunk {dt}")
    np.testing.assert_allclose(to_np32(lse), ref["lse"], rtol=0, atol=1e-4)
    # the chunk's rows are the full prefill's last rows (same codes, same tiles of keys)
    np.testing.assert_allclose(to_np32(o32), to_np32(full[:, :, Nk - Nq:]), rtol=0, atol=1e-6)
