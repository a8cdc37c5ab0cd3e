"""Pins for the oracle's grouped quantiser and the attn_w8a8_fwd prefill built on it.

Operation: "SuperL8" README (github.com/jajmangold/superl8), "Attention kernels" table,
attn_w8a8_fwd row (a W8A8 forward with scales set per warp that takes outliers into
account), and the "Quantization" table's per-row int8 row (outlier detection for Q).  The reading (groups of
G consecutive rows share the scale of their non-outlier rows; a row above tau times
its group's lower median max|x| keeps its own scale) is restated in the oracle.

What fixes the oracle here, independently of its code:
  - hand-derived golden cases (tests/golden/quant_groups_cases.txt), including ties
    and a case that tells the lower median from the upper median and from the mean;
  - G = 1 reduces to the per-row quantiser, which has its own pins;
  - invariants: a permutation of rows inside a group permutes the result, groups are
    independent of one another, power-of-two scaling moves only the scales, the
    round-trip bound |x - s q| <= s / 2, each group's largest inlier reaches +-127;
  - brute force: a planted outlier row quantises like a row of its own, and the rest of
    its group like the group without it; a short last group like those rows alone;
  - the attention on grouped codes equals textbook fp64 attention (torch's
    scaled_dot_product_attention in float64) on the dequantised Q and K.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    with open(os.path.join(GOLDEN, "quant_groups_cases.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                yield line.rstrip("\n")


def _mat(txt, dtype):
    return np.array([[float(t) for t in r.split()] for r in txt.split(";")], dtype)


def test_quant_groups_golden_cases():
    n = 0
    for line in _cases():
        head, rows, a_txt, flags_txt, codes_txt = (p.strip() for p in line.split("|"))
        g, tau = head.split()
        x = _mat(rows, np.float32)
        codes, scales, flags = oracle.quant_groups(x, int(g), float(tau))
        want_s = np.array([np.float32(float(t)) / np.float32(127) for t in a_txt.split()], np.float32)
        np.testing.assert_array_equal(scales, want_s, err_msg=line)
        np.testing.assert_array_equal(flags, np.array([t == "1" for t in flags_txt.split()]), err_msg=line)
        np.testing.assert_array_equal(codes, _mat(codes_txt, np.float64).astype(np.int8), err_msg=line)
        n += 1
    assert n == 5


def _rows(rng, n, d, spread=20.0):
    return (rng.standard_normal((n, d)) * rng.uniform(0.05, spread, size=(n, 1))).astype(np.float32)


def test_group_one_is_the_per_row_quantiser():
    rng = np.random.default_rng(40)
    x = _rows(rng, 97, 64)
    mu = (rng.standard_normal(64) * 0.5).astype(np.float32)
    for m in (None, mu):
        for tau in (0.0, 4.0):
            c1, s1, f1 = oracle.quant_groups(x, 1, tau, m)
            c0, s0 = oracle.quant_rowwise(x, None if m is None else m[None, :], len(x))
            np.testing.assert_array_equal(c1, c0)
            np.testing.assert_array_equal(s1, s0)
            assert not f1.any()


@pytest.mark.parametrize("group,tau", [(8, 0.0), (32, 0.0), (32, 4.0), (16, 1.5)])
def test_group_invariants(group, tau):
    rng = np.random.default_rng(41 + group)
    n, d = 4 * group + group // 2 + 1, 32          # a ragged last group
    x = _rows(rng, n, d)
    codes, scales, flags = oracle.quant_groups(x, group, tau)
    assert codes.min() >= -127 and codes.max() <= 127
    err = np.abs(x.astype(np.float64) - scales[:, None].astype(np.float64) * codes)
    assert np.all(err <= scales[:, None].astype(np.float64) / 2 * (1 + 1e-6))
    amax = np.abs(x).max(axis=1)
    for g0 in range(0, n, group):
        sl = slice(g0, min(g0 + group, n))
        inl = ~flags[sl]
        # the inliers share one scale, set by the largest of them, whose codes reach 127
        assert len(set(scales[sl][inl].tolist())) <= 1
        if inl.any():
            top = np.argmax(np.where(inl, amax[sl], -1.0))
            assert np.abs(codes[sl][top]).max() == 127
        # outliers quantise like rows of their own
        for r in np.nonzero(flags[sl])[0] + g0:
            c, s = oracle.quant_rowwise(x[r:r + 1])
            np.testing.assert_array_equal(codes[r], c[0])
            assert scales[r] == s[0]
    # a permutation inside each group permutes the result
    perm = np.concatenate([g0 + rng.permutation(min(group, n - g0)) for g0 in range(0, n, group)])
    c2, s2, f2 = oracle.quant_groups(x[perm], group, tau)
    np.testing.assert_array_equal(c2, codes[perm])
    np.testing.assert_array_equal(s2, scales[perm])
    np.testing.assert_array_equal(f2, flags[perm])
    # groups are independent: rescaling the second group leaves the others alone
    y = x.copy()
    y[group:2 * group] *= np.float32(37.0)
    c3, s3, _ = oracle.quant_groups(y, group, tau)
    keep = np.r_[0:group, 2 * group:n]
    np.testing.assert_array_equal(c3[keep], codes[keep])
    np.testing.assert_array_equal(s3[keep], scales[keep])
    # power-of-two scaling moves only the scales (x / s is unchanged exactly)
    c4, s4, f4 = oracle.quant_groups(x * np.float32(2.0 ** -7), group, tau)
    np.testing.assert_array_equal(c4, codes)
    np.testing.assert_array_equal(s4, scales * np.float32(2.0 ** -7))
    np.testing.assert_array_equal(f4, flags)
    # the short last group quantises like those rows alone
    tail = (n // group) * group
    c5, s5, f5 = oracle.quant_groups(x[tail:], group, tau)
    np.testing.assert_array_equal(c5, codes[tail:])
    np.testing.assert_array_equal(s5, scales[tail:])


def test_planted_outlier_rows():
    rng = np.random.default_rng(43)
    group, d = 32, 64
    x = (rng.standard_normal((3 * group, d))).astype(np.float32)
    planted = [5, group + 17, 2 * group + 31]
    for r in planted:
        x[r] *= np.float32(100.0)
    codes, scales, flags = oracle.quant_groups(x, group, 4.0)
    assert sorted(np.nonzero(flags)[0].tolist()) == planted
    for gi, r in enumerate(planted):
        g0 = gi * group
        rest = [i for i in range(g0, g0 + group) if i != r]
        c_rest, s_rest, _ = oracle.quant_groups(x[rest], group, 0.0)
        np.testing.assert_array_equal(codes[rest], c_rest)
        np.testing.assert_array_equal(scales[rest], s_rest)
    # without the outlier test the planted rows set every scale of their group
    c0, s0, f0 = oracle.quant_groups(x, group, 0.0)
    assert not f0.any()
    for gi, r in enumerate(planted):
        assert np.all(s0[gi * group:(gi + 1) * group] == scales[r])


def test_smoothed_groups_subtract_the_mean_first():
    rng = np.random.default_rng(44)
    x = _rows(rng, 64, 32)
    mu = (rng.standard_normal(32) * 3).astype(np.float32)
    c, s, _ = oracle.quant_groups(x, 16, 0.0, mu)
    c2, s2, _ = oracle.quant_groups((x - mu[None, :]).astype(np.float32), 16, 0.0)
    np.testing.assert_array_equal(c, c2)
    np.testing.assert_array_equal(s, s2)


@pytest.mark.parametrize("smooth", [False, True])
def test_grouped_attention_is_textbook_attention_on_dequantised_qk(smooth):
    rng = np.random.default_rng(45)
    B, Hq, Hkv, N, d = 1, 4, 2, 77, 32
    q = rng.standard_normal((B, Hq, N, d)).astype(np.float32)
    q[0, 1, 40] *= 30.0                                 # an outlier query row
    k = (rng.standard_normal((B, Hkv, N, d)) + 0.5).astype(np.float32)
    v = rng.standard_normal((B, Hkv, N, d)).astype(np.float32)
    res = oracle.attn_prefill(q, k, v, causal=True, smooth_k=smooth, q_group=32, k_group=16,
                              q_outlier_ratio=4.0)
    # the codes are those of the grouped quantiser (K after its channel mean)
    for h in range(Hq):
        c, s, f = oracle.quant_groups(q[0, h], 32, 4.0)
        np.testing.assert_array_equal(res["q_codes"][0, h], c)
        np.testing.assert_array_equal(res["q_scales"][0, h], s)
        assert f[40] == (h == 1)
    for h in range(Hkv):
        mu = oracle.k_channel_mean(k[0, h]) if smooth else None
        c, s, _ = oracle.quant_groups(k[0, h], 16, 0.0, mu)
        np.testing.assert_array_equal(res["k_codes"][0, h], c)
        np.testing.assert_array_equal(res["k_scales"][0, h], s)
    qd = torch.from_numpy(res["q_codes"].astype(np.float64) * res["q_scales"][..., None].astype(np.float64))
    kd = torch.from_numpy(res["k_codes"].astype(np.float64) * res["k_scales"][..., None].astype(np.float64))
    kd = kd.repeat_interleave(Hq // Hkv, dim=1)
    vd = torch.from_numpy(v.astype(np.float64)).repeat_interleave(Hq // Hkv, dim=1)
    want = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, is_causal=True).numpy()
    np.testing.assert_allclose(res["out"], want, rtol=0, atol=1e-12)


def test_default_groups_are_the_int8_path():
    rng = np.random.default_rng(46)
    q = rng.standard_normal((1, 2, 40, 32)).astype(np.float32)
    k = rng.standard_normal((1, 1, 40, 32)).astype(np.float32)
    v = rng.standard_normal((1, 1, 40, 32)).astype(np.float32)
    a = oracle.attn_prefill(q, k, v, smooth_k=True)
    b = oracle.attn_prefill(q, k, v, smooth_k=True, q_group=1, k_group=1, q_outlier_ratio=0.0)
    np.testing.assert_array_equal(a["out"], b["out"])
