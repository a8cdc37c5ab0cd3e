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


def test_k_mean_bit_exact_f32_keys():
    """fp32 keys (rows twice as wide as the half-precision ones), dense and ragged."""
    w = W.custom(2012, B=1, Hq=2, Hkv=2, N=200, d=256, dtype="bf16", k_bias_std=2.0)
    _, k, _ = W.prefill_dense(w)
    k32 = k.float() * 1.0009765625  # off the bf16 grid
    mu = sl8.k_channel_mean(k32.to(DEV)).cpu().numpy()
    for h in range(2):
        np.testing.assert_array_equal(mu[0, h], oracle.k_channel_mean(k32[0, h].numpy()))
    wv = W.custom(2013, kind="varlen", B=3, Hq=2, Hkv=2, d=128, dtype="bf16", k_bias_std=1.0,
                  extra={"lengths": [65, 1, 190]})
    _, kv, _, cu = W.prefill_varlen(wv)
    kv32 = kv.float() * 1.0009765625
    muv = sl8.k_channel_mean(kv32.to(DEV), cu.to(DEV), max_seqlen=190).cpu().numpy()
    c = cu.numpy()
    for s in range(3):
        for h in range(2):
            np.testing.assert_array_equal(muv[s, h], oracle.k_channel_mean(kv32[c[s]:c[s + 1], h].numpy()))


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


# ------------------------------------------------------------------ full-size workloads (every row)
#
# At the benchmark sizes every output row is compared with the oracle (fp32 and bf16
# outputs, LSE), the codes and scales of every Q and K row bit for bit, and the exact
# int32 logits on a seeded sample: for every head the first and the last 128-row tile
# and 64 random rows (whole rows, every key of the sequence), and for two heads every
# diagonal 128 x 128 tile (the tiles the causal mask cuts).  Only these launches reach
# late causal rows, run-time item claiming across all SMs, head pairs at G = 4 and the
# d = 256 kernel's double S buffer.

LOGIT_RANDOM_ROWS = 64
TILE = 128


def _logit_sample(rng, lens, Hq, diag_heads, packed=False):
    """({(s, h): rows} whole-row sample, {(s, h): rows} diagonal-tile rows), rows being
    indices within sequence s.  Per head: the first and the last 128-row tile and 64
    random rows of every sequence (dense), or of the packed token stream (packed=True:
    varlen input, whose first and last tiles then lie in its first and last sequences)."""
    lens = [int(x) for x in lens]
    starts = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    spans = [(0, int(starts[-1]))] if packed else [(int(starts[s]), int(starts[s + 1])) for s in range(len(lens))]
    whole = {}
    for h in range(Hq):
        for a, e in spans:
            picks = set(range(a, min(a + TILE, e))) | set(range(max(a, e - TILE), e))
            picks |= set(int(t) for t in rng.integers(a, e, size=LOGIT_RANDOM_ROWS))
            for t in picks:
                s = int(np.searchsorted(starts, t, side="right") - 1)
                whole.setdefault((s, h), set()).add(t - int(starts[s]))
    diag = {(s, h): set(range(lens[s])) for (s, h) in diag_heads}
    return ({k: sorted(v) for k, v in whole.items()}, {k: sorted(v) for k, v in diag.items()})


def _gpu_logits(qd, kd, smooth, lens, N, whole, diag, cu=None, chunk=1024):
    """Run the debug view in row chunks and keep, per (s, h), the whole rows of `whole`
    ({(s, h, i): int32 [L_s]}) and, of `diag`, each row's diagonal tile
    ({(s, h, i): int32 [tile width]})."""
    got_whole, got_diag = {}, {}
    ws = torch.empty(max(sl8.prefill_workspace_bytes(len(lens), qd.shape[-3] if cu is None else qd.shape[-2],
                                                     kd.shape[1] if cu is None else kd.shape[-2], N, qd.shape[-1],
                                                     0 if cu is None else qd.shape[0]), 16),
                     dtype=torch.uint8, device=DEV)
    for r0 in range(0, N, chunk):
        r1 = min(N, r0 + chunk)
        res = sl8.attn_int8_qk_logits_debug(qd, kd, smooth_k=smooth, row_begin=r0, row_end=r1, want_codes=False,
                                            cu_seqlens=cu, max_seqlen=None if cu is None else N, workspace=ws)
        lg = res["logits"]
        for (s, h), rows in whole.items():
            sel = [i for i in rows if r0 <= i < r1]
            if sel:
                block = lg[s, h, torch.tensor(sel, device=DEV) - r0, :lens[s]].cpu().numpy()
                for i, row in zip(sel, block):
                    got_whole[(s, h, i)] = row
        for (s, h), rows in diag.items():
            lo, hi = r0, min(r1, lens[s])
            for t0 in range(lo, hi, TILE):
                t1 = min(t0 + TILE, hi)
                blk = lg[s, h, t0 - r0:t1 - r0, t0:min(t0 + TILE, lens[s])].cpu().numpy()
                for i in range(t0, t1):
                    got_diag[(s, h, i)] = blk[i - t0]
        del res, lg
    return got_whole, got_diag


def _check_logits(q, k, v, smooth, got_whole, got_diag, whole, diag, lens, cu=None):
    rows = [(s, h, i) for (s, h), rr in whole.items() for i in rr]
    ref = oracle.attn_prefill(q, k, v, causal=False, smooth_k=smooth, rows=rows, want_logits=True,
                              cu_seqlens=cu)
    for key in rows:
        np.testing.assert_array_equal(got_whole[key], ref["logits"][key], err_msg=f"logits row {key}")
    del ref
    for (s, h), rr in diag.items():
        ref = oracle.attn_prefill(q, k, v, causal=False, smooth_k=smooth, rows=[(s, h, i) for i in rr],
                                  want_logits=True, cu_seqlens=cu)
        for i in rr:
            t0 = i // TILE * TILE
            want = ref["logits"][(s, h, i)][t0:min(t0 + TILE, lens[s])]
            np.testing.assert_array_equal(got_diag[(s, h, i)], want, err_msg=f"diagonal tile row {(s, h, i)}")
        del ref


@pytest.mark.parametrize("name", ["qwen3_8b", "gemma3_d256"])
def test_full_size_dense_workload(name):
    w = W.get(name)
    q, k, v = W.prefill_dense(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o32, lse = sl8.attn_int8_fwd(qd, kd, vd, causal=True, smooth_k=w.smooth_k, out_dtype=torch.float32,
                                 return_lse=True)
    oh = sl8.attn_int8_fwd(qd, kd, vd, causal=True, smooth_k=w.smooth_k)
    codes = sl8.attn_int8_qk_logits_debug(qd, kd, smooth_k=w.smooth_k, row_begin=0, row_end=0, want_logits=False)
    torch.cuda.synchronize()
    _status_ok()
    qn, kn, vn = _np(q), _np(k), _np(v)
    ref = oracle.attn_prefill(qn, kn, vn, causal=True, smooth_k=w.smooth_k)
    for c in ("q_codes", "q_scales", "k_codes", "k_scales"):
        np.testing.assert_array_equal(codes[c].cpu().numpy(), ref[c], err_msg=c)
    check_f32(to_np32(o32), ref["out"], f"{name} f32, every row")
    check_half(oh, ref["out"], f"{name} bf16, every row")
    np.testing.assert_allclose(to_np32(lse), ref["lse"], rtol=0, atol=1e-4)
    del ref, o32, oh, lse
    whole, diag = _logit_sample(np.random.default_rng(7), [w.N] * w.B, w.Hq, [(0, 0), (w.B - 1, w.Hq - 1)])
    got_whole, got_diag = _gpu_logits(qd, kd, w.smooth_k, [w.N] * w.B, w.N, whole, diag)
    _status_ok()
    _check_logits(qn, kn, vn, w.smooth_k, got_whole, got_diag, whole, diag, [w.N] * w.B)


def test_full_size_varlen_workload():
    w = W.get("varlen")
    q, k, v, cu = W.prefill_varlen(w)
    lens = [int(x) for x in np.diff(cu.numpy())]
    N = max(lens)
    qd, kd, vd, cud = q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV)
    o32, lse = sl8.attn_int8_fwd(qd, kd, vd, cu_seqlens=cud, max_seqlen=N, out_dtype=torch.float32,
                                 return_lse=True)
    oh = sl8.attn_int8_fwd(qd, kd, vd, cu_seqlens=cud, max_seqlen=N)
    codes = sl8.attn_int8_qk_logits_debug(qd, kd, smooth_k=True, row_begin=0, row_end=0, want_logits=False,
                                          cu_seqlens=cud, max_seqlen=N)
    torch.cuda.synchronize()
    _status_ok()
    qn, kn, vn = _np(q), _np(k), _np(v)
    ref = oracle.attn_prefill(qn, kn, vn, causal=True, smooth_k=True, cu_seqlens=cu.numpy())
    for c in ("q_codes", "q_scales", "k_codes", "k_scales"):
        np.testing.assert_array_equal(codes[c].cpu().numpy(), ref[c], err_msg=c)
    check_f32(to_np32(o32), ref["out"], "varlen f32, every row")
    check_half(oh, ref["out"], "varlen bf16, every row")
    np.testing.assert_allclose(to_np32(lse), ref["lse"], rtol=0, atol=1e-4)
    del ref, o32, oh, lse
    whole, diag = _logit_sample(np.random.default_rng(8), lens, w.Hq, [(0, 0), (len(lens) - 1, w.Hq - 1)],
                                packed=True)
    got_whole, got_diag = _gpu_logits(qd, kd, True, lens, N, whole, diag, cu=cud, chunk=256)
    _status_ok()
    _check_logits(qn, kn, vn, True, got_whole, got_diag, whole, diag, lens, cu=cu.numpy())


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
    (2609, 1, 4, 2, 100, 2100, 64, "f16", True),  # 4 items: keys split into 8 parts
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
    # the default workspace lets a small chunk split its keys across CTAs and merge the
    # parts: the same attention, with P rounded to fp16 against each part's own running max
    # (so within that rounding of the unsplit rows; the oracle checks above are the bar)
    np.testing.assert_allclose(to_np32(o32), to_np32(full[:, :, Nk - Nq:]), rtol=0, atol=2e-4)
    # with only the plain prefill workspace the chunk is not split: its rows are the full
    # prefill's last rows (same codes, same tiles of keys, same order)
    base_ws = torch.empty(sl8.prefill_workspace_bytes(B, Hq, Hkv, Nk, d), dtype=torch.uint8, device=DEV)
    o32b, lseb = sl8.attn_int8_fwd_chunk(qc.to(DEV), k.to(DEV), v.to(DEV), causal=causal, smooth_k=True,
                                         out_dtype=torch.float32, return_lse=True, workspace=base_ws)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_np32(o32b), to_np32(full[:, :, Nk - Nq:]), rtol=0, atol=1e-6)
    np.testing.assert_allclose(to_np32(lseb), to_np32(lse), rtol=0, atol=1e-4)
    _status_ok()


def test_chunk_key_split_is_used_and_matches():
    """A 256-query chunk of the Qwen3-8B-shaped prefill: 32 (query tile, head pair) items
    for the GPU's SMs, so the default workspace splits each item's keys.  The split form
    and the unsplit form (plain workspace) agree with each other and with the oracle on
    sampled rows.  The 1024-query chunk (128 items) is left unsplit."""
    w = W.get("qwen3_8b")
    q, k, v = W.prefill_dense(w)
    small = sl8.prefill_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d)
    assert sl8.lib().sl8_attn_int8_fwd_chunk_workspace_size(w.B, w.Hq, w.Hkv, 1024, w.N, w.d) == small
    nq = 256
    qc = q[:, :, w.N - nq:].contiguous()
    qd, kd, vd = qc.to(DEV), k.to(DEV), v.to(DEV)
    big = sl8.lib().sl8_attn_int8_fwd_chunk_workspace_size(w.B, w.Hq, w.Hkv, nq, w.N, w.d)
    assert big > small
    o_split, l_split = sl8.attn_int8_fwd_chunk(qd, kd, vd, out_dtype=torch.float32, return_lse=True)
    o_one, l_one = sl8.attn_int8_fwd_chunk(qd, kd, vd, out_dtype=torch.float32, return_lse=True,
                                           workspace=torch.empty(small, dtype=torch.uint8, device=DEV))
    torch.cuda.synchronize()
    _status_ok()
    np.testing.assert_allclose(to_np32(o_split), to_np32(o_one), rtol=0, atol=2e-4)
    np.testing.assert_allclose(to_np32(l_split), to_np32(l_one), rtol=0, atol=1e-4)
    rng = np.random.default_rng(11)
    rows = [(0, h, int(i)) for h in range(w.Hq) for i in rng.integers(0, nq, size=8)]
    ref = oracle.attn_prefill(_np(qc), _np(k), _np(v), causal=True, smooth_k=True, rows=rows)
    check_f32(to_np32(o_split), ref["out"], "chunk 256 split f32")
