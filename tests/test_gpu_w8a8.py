"""GPU parity of attn_w8a8_fwd (grouped "per-warp" scales, outlier-aware Q) against
the CPU oracle, through the C ABI.

Operation: the "SuperL8" README, "Attention kernels" table, attn_w8a8_fwd row (a W8A8
forward with scales set per warp that takes outliers into account) and the
"Quantization" table's per-row int8 row (outlier detection for Q).  Bit-exact: the int8 codes, the fp32 scales and the int32
logits; outputs within the tolerances of tests/_parity.py.
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


def _plant_outliers(q, rng, frac=0.03, gain=40.0):
    """Scale a few query rows of every head up (rows whose max|x| stands far above
    their group's), in the input dtype."""
    q = q.clone()
    rows = q.reshape(-1, q.shape[-1])
    pick = rng.choice(rows.shape[0], size=max(1, int(frac * rows.shape[0])), replace=False)
    rows[torch.from_numpy(pick)] = (rows[torch.from_numpy(pick)].float() * gain).to(q.dtype)
    return q


CODE_CASES = [
    # wid, B, Hq, Hkv, N, d, dtype, smooth, q_group, k_group, tau
    (2701, 1, 4, 2, 256, 64, "f16", True, 32, 32, 4.0),
    (2702, 2, 4, 1, 300, 128, "bf16", True, 32, 64, 4.0),
    (2703, 1, 2, 2, 200, 256, "bf16", True, 64, 16, 1.5),
    (2704, 1, 8, 8, 129, 128, "bf16", False, 8, 8, 0.0),
    (2705, 1, 2, 1, 1, 64, "bf16", True, 32, 32, 4.0),
    (2706, 1, 4, 2, 200, 32, "bf16", True, 16, 32, 2.0),
    (2707, 2, 2, 1, 77, 128, "f16", False, 2, 4, 1.0),
]


@pytest.mark.parametrize("case", CODE_CASES, ids=[f"w{c[0]}_N{c[4]}_d{c[5]}_g{c[8]}" for c in CODE_CASES])
def test_grouped_codes_scales_logits_bit_exact(case):
    wid, B, Hq, Hkv, N, d, dt, smooth, gq, gk, tau = case
    w = W.custom(wid, B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, dtype=dt, k_bias_std=1.0)
    q, k, v = W.prefill_dense(w)
    q = _plant_outliers(q, np.random.default_rng(wid))
    res = sl8.attn_int8_qk_logits_debug(q.to(DEV), k.to(DEV), smooth_k=smooth, groups=(gq, gk, tau))
    torch.cuda.synchronize()
    _status_ok()
    ref = oracle.attn_prefill(_np(q), _np(k), _np(v), causal=False, smooth_k=smooth,
                              rows=[(b, h, i) for b in range(B) for h in range(Hq) for i in range(N)],
                              want_logits=True, q_group=gq, k_group=gk, q_outlier_ratio=tau)
    np.testing.assert_array_equal(res["q_scales"].cpu().numpy(), ref["q_scales"])
    np.testing.assert_array_equal(res["q_codes"].cpu().numpy(), ref["q_codes"])
    np.testing.assert_array_equal(res["k_scales"].cpu().numpy(), ref["k_scales"])
    np.testing.assert_array_equal(res["k_codes"].cpu().numpy(), ref["k_codes"])
    lg = res["logits"].cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            want = np.stack([ref["logits"][(b, h, i)] for i in range(N)])
            np.testing.assert_array_equal(lg[b, h], want)
    if tau > 0 and gq > 1 and N >= 2 * gq:
        # the planted rows were found: some group holds a row with a scale of its own
        qs = ref["q_scales"][..., :N // gq * gq].reshape(B, Hq, -1, gq)
        assert np.any(qs.max(axis=-1) != qs.min(axis=-1))


OUT_CASES = [
    # wid, B, Hq, Hkv, N, d, dtype, causal, smooth, q_group, k_group, tau
    (2711, 1, 4, 2, 256, 64, "f16", True, True, 32, 32, 4.0),
    (2712, 2, 8, 2, 300, 128, "bf16", True, True, 32, 32, 4.0),
    (2713, 1, 4, 4, 200, 256, "bf16", True, True, 64, 64, 4.0),
    (2714, 1, 8, 1, 129, 64, "bf16", False, True, 16, 32, 0.0),
    (2715, 1, 4, 2, 300, 32, "f16", True, True, 32, 8, 2.0),
    (2716, 1, 2, 1, 1, 128, "bf16", True, True, 32, 32, 4.0),
]


@pytest.mark.parametrize("case", OUT_CASES, ids=[f"w{c[0]}_N{c[4]}_d{c[5]}_g{c[9]}" for c in OUT_CASES])
def test_w8a8_outputs_small(case):
    wid, B, Hq, Hkv, N, d, dt, causal, smooth, gq, gk, tau = case
    w = W.custom(wid, B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, dtype=dt, k_bias_std=1.0)
    q, k, v = W.prefill_dense(w)
    q = _plant_outliers(q, np.random.default_rng(wid))
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    kw = dict(causal=causal, smooth_k=smooth, q_group=gq, k_group=gk, q_outlier_ratio=tau)
    o32, lse = sl8.attn_w8a8_fwd(qd, kd, vd, out_dtype=torch.float32, return_lse=True, **kw)
    oh = sl8.attn_w8a8_fwd(qd, kd, vd, **kw)
    torch.cuda.synchronize()
    _status_ok()
    ref = oracle.attn_prefill(_np(q), _np(k), _np(v), causal=causal, smooth_k=smooth, q_group=gq, k_group=gk,
                              q_outlier_ratio=tau)
    check_f32(to_np32(o32), ref["out"], f"w{wid} f32")
    check_half(oh, ref["out"], f"w{wid} {dt}")
    np.testing.assert_allclose(to_np32(lse), ref["lse"], rtol=0, atol=1e-4)


def test_group_one_is_attn_int8_fwd_bytes():
    w = W.custom(2721, B=1, Hq=8, Hkv=2, N=333, d=128, dtype="bf16", k_bias_std=1.0)
    q, k, v = W.prefill_dense(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    a = sl8.attn_int8_fwd(qd, kd, vd)
    b = sl8.attn_w8a8_fwd(qd, kd, vd, q_group=1, k_group=1, q_outlier_ratio=0.0)
    torch.cuda.synchronize()
    _status_ok()
    assert torch.equal(a, b)


def test_w8a8_varlen_ragged_groups():
    """Sequence ends inside a group: the group's scale covers its valid rows only."""
    w = W.custom(2722, kind="varlen", B=6, Hq=8, Hkv=2, d=128, dtype="bf16", k_bias_std=1.0,
                 extra={"lengths": [1, 17, 130, 256, 3, 300]})
    q, k, v, cu = W.prefill_varlen(w)
    q = _plant_outliers(q, np.random.default_rng(2722))
    kw = dict(q_group=32, k_group=64, q_outlier_ratio=4.0, cu_seqlens=cu.to(DEV), max_seqlen=300)
    o32, lse = sl8.attn_w8a8_fwd(q.to(DEV), k.to(DEV), v.to(DEV), out_dtype=torch.float32, return_lse=True, **kw)
    oh = sl8.attn_w8a8_fwd(q.to(DEV), k.to(DEV), v.to(DEV), **kw)
    torch.cuda.synchronize()
    _status_ok()
    ref = oracle.attn_prefill(_np(q), _np(k), _np(v), causal=True, smooth_k=True, cu_seqlens=cu.numpy(),
                              q_group=32, k_group=64, q_outlier_ratio=4.0)
    check_f32(to_np32(o32), ref["out"], "w8a8 varlen f32")
    check_half(oh, ref["out"], "w8a8 varlen bf16")
    np.testing.assert_allclose(to_np32(lse), ref["lse"], rtol=0, atol=1e-4)


def test_w8a8_full_size_dense_workload():
    """The Qwen3-8B-shaped prefill (B1 Hq32 Hkv8 N4096 d128) with warp groups and outlier
    rows: all codes and scales bit-exact, sampled rows of the output."""
    w = W.get("qwen3_8b")
    q, k, v = W.prefill_dense(w)
    q = _plant_outliers(q, np.random.default_rng(2731), frac=0.005)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    kw = dict(q_group=32, k_group=32, q_outlier_ratio=4.0)
    o32 = sl8.attn_w8a8_fwd(qd, kd, vd, smooth_k=w.smooth_k, out_dtype=torch.float32, **kw)
    oh = sl8.attn_w8a8_fwd(qd, kd, vd, smooth_k=w.smooth_k, **kw)
    dbg = sl8.attn_int8_qk_logits_debug(qd, kd, smooth_k=w.smooth_k, row_begin=w.N - 1, row_end=w.N,
                                        groups=(32, 32, 4.0))
    torch.cuda.synchronize()
    _status_ok()
    rng = np.random.default_rng(9)
    rows = sample_rows(rng, [w.N] * w.B, w.Hq, per_head=3)
    ref = oracle.attn_prefill(_np(q), _np(k), _np(v), causal=True, smooth_k=w.smooth_k, rows=rows,
                              q_group=32, k_group=32, q_outlier_ratio=4.0)
    np.testing.assert_array_equal(dbg["q_scales"].cpu().numpy(), ref["q_scales"])
    np.testing.assert_array_equal(dbg["q_codes"].cpu().numpy(), ref["q_codes"])
    np.testing.assert_array_equal(dbg["k_scales"].cpu().numpy(), ref["k_scales"])
    np.testing.assert_array_equal(dbg["k_codes"].cpu().numpy(), ref["k_codes"])
    sel = np.zeros(q.shape[:-1], bool)
    for (b, h, i) in rows:
        sel[b, h, i] = True
    refo = np.where(sel[..., None], ref["out"], np.nan)
    check_f32(to_np32(o32), refo, "qwen3_8b w8a8 f32")
    check_half(oh, refo, "qwen3_8b w8a8 bf16")
