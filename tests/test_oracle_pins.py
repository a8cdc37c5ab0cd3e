"""Pins for the CPU oracle: facts fixed by the pages' definitions or by mathematics,
independent of the oracle's own code.

Operation sources (the "SuperL8" README, github.com/jajmangold/superl8): "Supporting
kernels" table (quant_rowwise), "Quantization" table (per-row int8, K-smoothing),
"Attention kernels" table (attn_int8_fwd causal GQA/MQA prefill, attn_varlen_fwd,
attn_decode split-KV over an int8 cache) and the "Quick start" section (layouts).

Each pin is built so that a plausible slip in the oracle (a dropped term, a wrong sign
or index, a transposed operand, a wrong rounding mode or summation order) fails it:
  - hand-derived golden cases (tests/golden/) for the quantiser's rounding and division
    and for the K-mean summation order;
  - closed forms: the round-trip bound |x - s q| <= s/2, exact codes for integer x 2^k rows;
  - textbook fp64 attention (torch's scaled_dot_product_attention in float64) on
    quantisation-exact inputs, where the W8A8 path has no quantisation error at all;
  - invariants: softmax rows sum to 1, causal row 0 returns v_0, zero Q averages V,
    GQA equals MHA with repeated K/V, K-smoothing leaves exact-case outputs unchanged,
    split-count invariance of split-KV decode, decode equals the prefill's last row;
  - brute force: int64 matmul of the codes gives the int32 logits.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def exact_rows(rng, shape, emin=-6, emax=1):
    """Rows of integers in [-127, 127] (each row holding a +-127) times a per-row 2^e.

    Symmetric per-row int8 quantisation reproduces such rows exactly: s = 2^e and the
    codes are the integers.  Returns (x fp32, codes int8, scales fp32)."""
    *lead, d = shape
    codes = rng.integers(-127, 128, size=shape).astype(np.int64)
    flat = codes.reshape(-1, d)
    pos = rng.integers(0, d, size=flat.shape[0])
    sign = rng.choice([-1, 1], size=flat.shape[0])
    flat[np.arange(flat.shape[0]), pos] = 127 * sign
    e = rng.integers(emin, emax + 1, size=flat.shape[0])
    scales = np.ldexp(np.ones(flat.shape[0]), e).astype(np.float32).reshape(lead)
    x = (codes.astype(np.float64) * scales[..., None].astype(np.float64)).astype(np.float32)
    return x, codes.astype(np.int8), scales


def textbook(q, k, v, causal):
    """fp64 softmax(q k^T / sqrt(d)) v via torch; q [B,Hq,N,d], k/v [B,Hkv,N,d]."""
    g = q.shape[1] // k.shape[1]
    qt = torch.from_numpy(np.asarray(q, np.float64))
    kt = torch.from_numpy(np.asarray(k, np.float64)).repeat_interleave(g, dim=1)
    vt = torch.from_numpy(np.asarray(v, np.float64)).repeat_interleave(g, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal)
    return o.numpy()


def read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ---------------------------------------------------------------- quantiser

def test_quant_golden_cases():
    for line in read_rows("quant_rowwise_cases.txt"):
        s_txt, x_txt, c_txt = (p.strip() for p in line.split("|"))
        x = np.array([float(t) for t in x_txt.split()], np.float32)[None, :]
        want = np.array([int(t) for t in c_txt.split()], np.int8)
        codes, scales = oracle.quant_rowwise(x)
        assert scales[0] == np.float32(float(s_txt)), line
        np.testing.assert_array_equal(codes[0], want, err_msg=line)


def test_quant_round_trip_bound_and_range():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((512, 128)) * rng.uniform(0.01, 50, size=(512, 1))).astype(np.float32)
    x[7, 3] *= 1000.0  # an outlier row
    codes, s = oracle.quant_rowwise(x)
    assert codes.min() >= -127 and codes.max() <= 127
    err = np.abs(x.astype(np.float64) - s[:, None].astype(np.float64) * codes)
    assert np.all(err <= s[:, None].astype(np.float64) / 2 * (1 + 1e-6))
    # the row maximum always lands on +-127 (s = max/127 makes max/s round to 127)
    assert np.all(np.abs(codes).max(axis=1) == 127)
    # scale is max|x|/127 in fp32
    np.testing.assert_array_equal(s, (np.abs(x).max(axis=1) / np.float32(127)).astype(np.float32))


def test_quant_exact_rows():
    rng = np.random.default_rng(2)
    x, c, s = exact_rows(rng, (64, 64))
    codes, scales = oracle.quant_rowwise(x)
    np.testing.assert_array_equal(codes, c)
    np.testing.assert_array_equal(scales, s)


def test_quant_smoothing_subtracts_group_mean():
    rng = np.random.default_rng(3)
    x, c, s = exact_rows(rng, (6, 32))
    mu = np.array([rng.integers(-4, 5, 32), rng.integers(-4, 5, 32)], np.float32) * np.float32(0.25)
    shifted = x.copy()
    shifted[:3] += mu[0]
    shifted[3:] += mu[1]
    # the shifted values are exact in fp32 (few significant bits), so x + mu - mu == x
    codes, scales = oracle.quant_rowwise(shifted, mu, rows_per_group=3)
    np.testing.assert_array_equal(codes, c)
    np.testing.assert_array_equal(scales, s)


# ---------------------------------------------------------------- K mean

def test_k_mean_golden_order():
    (line,) = read_rows("k_mean_order.txt")
    n, first, other, want = line.split()
    k = np.full((int(n), 1), np.float32(float(other)), np.float32)
    k[0, 0] = np.float32(float(first))
    mu = oracle.k_channel_mean(k)
    assert mu[0] == np.float32(float(want))


def test_k_mean_close_to_exact_mean():
    rng = np.random.default_rng(4)
    for n in (1, 63, 64, 65, 1000, 4097):
        k = (rng.standard_normal((n, 16)) * 3 + rng.standard_normal(16) * 2).astype(np.float32)
        mu = oracle.k_channel_mean(k)
        exact = k.astype(np.float64).mean(axis=0)
        bound = n * 2.0 ** -23 * np.abs(k.astype(np.float64)).sum(axis=0) / n + 1e-30
        assert np.all(np.abs(mu - exact) <= bound), n


def test_k_mean_integer_data_is_exact():
    rng = np.random.default_rng(5)
    k = rng.integers(-1000, 1000, size=(777, 8)).astype(np.float32)
    mu = oracle.k_channel_mean(k)
    np.testing.assert_array_equal(mu, (k.astype(np.float64).sum(axis=0) / 777).astype(np.float32))


# ---------------------------------------------------------------- prefill

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv,d", [(4, 2, 64), (3, 1, 32), (2, 2, 128)])
def test_prefill_equals_textbook_on_exact_inputs(causal, hq, hkv, d):
    rng = np.random.default_rng(10 + d + hq)
    B, N = 2, 37
    q, _, _ = exact_rows(rng, (B, hq, N, d))
    k, _, _ = exact_rows(rng, (B, hkv, N, d))
    v = rng.standard_normal((B, hkv, N, d)).astype(np.float32)
    r = oracle.attn_prefill(q, k, v, causal=causal, smooth_k=False)
    ref = textbook(q, k, v, causal)
    np.testing.assert_allclose(r["out"], ref, rtol=0, atol=1e-10)


def test_prefill_lse_matches_logsumexp():
    rng = np.random.default_rng(11)
    q, _, _ = exact_rows(rng, (1, 2, 20, 64))
    k, _, _ = exact_rows(rng, (1, 2, 20, 64))
    v = rng.standard_normal((1, 2, 20, 64)).astype(np.float32)
    r = oracle.attn_prefill(q, k, v, causal=True)
    s = np.einsum("bhid,bhjd->bhij", q.astype(np.float64), k.astype(np.float64)) / math.sqrt(64)
    s = np.where(np.tril(np.ones((20, 20), bool)), s, -np.inf)
    want = np.log(np.exp(s - s.max(-1, keepdims=True)).sum(-1)) + s.max(-1)
    np.testing.assert_allclose(r["lse"], want, rtol=0, atol=1e-10)


def test_prefill_rows_sum_to_one_and_row0():
    rng = np.random.default_rng(12)
    q = rng.standard_normal((1, 4, 50, 64)).astype(np.float32)
    k = (rng.standard_normal((1, 2, 50, 64)) * 3).astype(np.float32)
    ones = np.ones((1, 2, 50, 64), np.float32)
    r = oracle.attn_prefill(q, k, ones, causal=True, smooth_k=True)
    np.testing.assert_allclose(r["out"], 1.0, rtol=0, atol=1e-14)
    v = rng.standard_normal((1, 2, 50, 64)).astype(np.float32)
    r = oracle.attn_prefill(q, k, v, causal=True, smooth_k=True)
    for hq in range(4):
        np.testing.assert_array_equal(r["out"][0, hq, 0], v[0, hq // 2, 0].astype(np.float64))


def test_prefill_zero_q_averages_v():
    rng = np.random.default_rng(13)
    q = np.zeros((1, 2, 40, 32), np.float32)
    k = rng.standard_normal((1, 1, 40, 32)).astype(np.float32)
    v = rng.standard_normal((1, 1, 40, 32)).astype(np.float32)
    r = oracle.attn_prefill(q, k, v, causal=True)
    assert np.all(r["q_scales"] == 0) and np.all(r["q_codes"] == 0)
    want = np.cumsum(v[0, 0].astype(np.float64), axis=0) / np.arange(1, 41)[:, None]
    for h in range(2):
        np.testing.assert_allclose(r["out"][0, h], want, rtol=0, atol=1e-13)
    # non-causal: every row is the full mean
    r = oracle.attn_prefill(q, k, v, causal=False)
    np.testing.assert_allclose(r["out"][0, 0], np.broadcast_to(want[-1], (40, 32)), rtol=0, atol=1e-13)


def test_prefill_output_inside_v_hull():
    rng = np.random.default_rng(14)
    q = rng.standard_normal((1, 2, 64, 64)).astype(np.float32)
    k = rng.standard_normal((1, 2, 64, 64)).astype(np.float32)
    v = rng.standard_normal((1, 2, 64, 64)).astype(np.float32)
    r = oracle.attn_prefill(q, k, v, causal=True, smooth_k=True)
    for i in range(64):
        lo = v[0, :, : i + 1].min(axis=1)
        hi = v[0, :, : i + 1].max(axis=1)
        assert np.all(r["out"][0, :, i] >= lo - 1e-12) and np.all(r["out"][0, :, i] <= hi + 1e-12)


def test_gqa_equals_repeated_kv_mha():
    rng = np.random.default_rng(15)
    q = rng.standard_normal((2, 8, 33, 64)).astype(np.float32)
    k = (rng.standard_normal((2, 2, 33, 64)) + rng.standard_normal(64)).astype(np.float32)
    v = rng.standard_normal((2, 2, 33, 64)).astype(np.float32)
    a = oracle.attn_prefill(q, k, v, causal=True, smooth_k=True)
    b = oracle.attn_prefill(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), causal=True, smooth_k=True)
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["lse"], b["lse"])


def test_smoothing_invariance_exact_case():
    """K = K0 + mu with K0 quantisation-exact and zero channel means: smoothing recovers
    K0 exactly, and attention against K0 equals attention against K (a per-channel
    constant shifts each row's logits by q.mu, which the softmax removes)."""
    rng = np.random.default_rng(16)
    N, d = 40, 64
    q, _, _ = exact_rows(rng, (1, 2, N, d))
    half, _, _ = exact_rows(rng, (1, 1, N // 2, d), emin=-3, emax=-3)
    k0 = np.concatenate([half, -half], axis=2)  # every channel sums to exactly 0
    k0 = k0[:, :, rng.permutation(N)]
    mu = (rng.integers(-16, 17, size=d) * 0.125).astype(np.float32)
    k = (k0 + mu).astype(np.float32)
    assert np.array_equal(k - mu, k0)
    v = rng.standard_normal((1, 1, N, d)).astype(np.float32)
    r = oracle.attn_prefill(q, k, v, causal=True, smooth_k=True)
    np.testing.assert_array_equal(r["k_mean"][0, 0], mu)
    np.testing.assert_allclose(r["out"], textbook(q, k0, v, True), rtol=0, atol=1e-10)
    np.testing.assert_allclose(r["out"], textbook(q, k, v, True), rtol=0, atol=1e-10)


def test_logits_brute_force_int_matmul():
    rng = np.random.default_rng(17)
    q = rng.standard_normal((1, 4, 29, 128)).astype(np.float32) * 5
    k = rng.standard_normal((1, 2, 29, 128)).astype(np.float32) * 5
    v = rng.standard_normal((1, 2, 29, 128)).astype(np.float32)
    r = oracle.attn_prefill(q, k, v, causal=True, smooth_k=True, want_logits=True)
    for hq in range(4):
        full = r["q_codes"][0, hq].astype(np.int64) @ r["k_codes"][0, hq // 2].astype(np.int64).T
        for i in range(29):
            np.testing.assert_array_equal(r["logits"][(0, hq, i)], full[i, : i + 1])


def test_varlen_equals_per_sequence_dense():
    rng = np.random.default_rng(18)
    lens = [1, 17, 64, 130]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = cu[-1]
    q = rng.standard_normal((T, 4, 64)).astype(np.float32)
    k = (rng.standard_normal((T, 2, 64)) + 2 * rng.standard_normal(64)).astype(np.float32)
    v = rng.standard_normal((T, 2, 64)).astype(np.float32)
    r = oracle.attn_prefill(q, k, v, causal=True, smooth_k=True, cu_seqlens=cu)
    for s, L in enumerate(lens):
        a = cu[s]
        sl = slice(a, a + L)
        dq = q[sl].transpose(1, 0, 2)[None]
        dk = k[sl].transpose(1, 0, 2)[None]
        dv = v[sl].transpose(1, 0, 2)[None]
        rd = oracle.attn_prefill(dq, dk, dv, causal=True, smooth_k=True)
        np.testing.assert_array_equal(r["out"][sl], rd["out"][0].transpose(1, 0, 2))
        np.testing.assert_array_equal(r["k_codes"][sl], rd["k_codes"][0].transpose(1, 0, 2))


def test_row_subset_matches_full():
    rng = np.random.default_rng(19)
    q = rng.standard_normal((1, 2, 70, 64)).astype(np.float32)
    k = rng.standard_normal((1, 1, 70, 64)).astype(np.float32)
    v = rng.standard_normal((1, 1, 70, 64)).astype(np.float32)
    full = oracle.attn_prefill(q, k, v, causal=True)
    rows = [(0, 1, 0), (0, 1, 69), (0, 0, 33)]
    part = oracle.attn_prefill(q, k, v, causal=True, rows=rows)
    for (b, h, i) in rows:
        np.testing.assert_array_equal(part["out"][b, h, i], full["out"][b, h, i])


# ---------------------------------------------------------------- decode

def _decode_case(rng, B=3, hq=4, hkv=2, lmax=300, d=64, lens=(1, 150, 300)):
    kf, kc, ks = exact_rows(rng, (B, hkv, lmax, d))
    vf, vc, vs = exact_rows(rng, (B, hkv, lmax, d))
    q, _, _ = exact_rows(rng, (B, hq, d))
    return q, kf, kc, ks, vf, vc, vs, np.array(lens, np.int64)


def test_decode_equals_textbook_and_prefill_last_row():
    rng = np.random.default_rng(20)
    q, kf, kc, ks, vf, vc, vs, lens = _decode_case(rng)
    r = oracle.attn_decode(q, kc, ks, vc, vs, lens, num_splits=1)
    for b, L in enumerate(lens):
        qq = q[b][:, None, :][None]                                  # [1, Hq, 1, d]
        ref = textbook(qq, kf[b][None, :, :L], vf[b][None, :, :L], causal=False)[0, :, 0]
        np.testing.assert_allclose(r["out"][b], ref, rtol=0, atol=1e-10)
        # prefill oracle: query placed at row L-1 of a causal sequence of length L
        qp = np.zeros((1, q.shape[1], L, q.shape[2]), np.float32)
        qp[0, :, L - 1] = q[b]
        rp = oracle.attn_prefill(qp, kf[b][None, :, :L], vf[b][None, :, :L], causal=True,
                                 rows=[(0, h, L - 1) for h in range(q.shape[1])])
        np.testing.assert_allclose(r["out"][b], rp["out"][0, :, L - 1], rtol=0, atol=1e-12)


def test_decode_split_count_invariance():
    rng = np.random.default_rng(21)
    q = rng.standard_normal((2, 4, 64)).astype(np.float32)
    kc = rng.integers(-127, 128, size=(2, 2, 513, 64)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(2, 2, 513, 64)).astype(np.int8)
    ks = rng.uniform(0.001, 0.05, size=(2, 2, 513)).astype(np.float32)
    vs = rng.uniform(0.001, 0.05, size=(2, 2, 513)).astype(np.float32)
    lens = np.array([513, 77])
    one = oracle.attn_decode(q, kc, ks, vc, vs, lens, num_splits=1)
    for ns in (2, 5, 16, 64):
        many = oracle.attn_decode(q, kc, ks, vc, vs, lens, num_splits=ns)
        np.testing.assert_allclose(many["out"], one["out"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(many["lse"], one["lse"], rtol=0, atol=1e-12)
        # splits past a sequence's end are empty: lse -inf
        assert np.all(np.isneginf(many["lse_partial"][1][:, -1])) or ns <= 6


def test_decode_logits_and_empty_context():
    rng = np.random.default_rng(22)
    q = rng.standard_normal((2, 2, 64)).astype(np.float32)
    kc = rng.integers(-127, 128, size=(2, 1, 40, 64)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(2, 1, 40, 64)).astype(np.int8)
    ks = np.full((2, 1, 40), 0.01, np.float32)
    vs = np.full((2, 1, 40), 0.02, np.float32)
    lens = np.array([40, 0])
    r = oracle.attn_decode(q, kc, ks, vc, vs, lens, num_splits=3, want_logits=True)
    qc, _ = oracle.quant_rowwise(q)
    for h in range(2):
        np.testing.assert_array_equal(r["logits"][(0, h)], kc[0, 0].astype(np.int64) @ qc[0, h].astype(np.int64))
    assert np.all(r["out"][1] == 0) and np.all(np.isneginf(r["lse"][1]))


def test_combine_weights():
    o = np.array([[[1.0, 2.0], [3.0, 4.0], [9.0, 9.0]]])
    lse = np.array([[math.log(1.0), math.log(3.0), -math.inf]])
    out, l = oracle.decode_combine(o, lse)
    np.testing.assert_allclose(out[0], [(1 * 1 + 3 * 3) / 4, (2 * 1 + 4 * 3) / 4], rtol=0, atol=1e-15)
    np.testing.assert_allclose(l[0], math.log(4.0), rtol=0, atol=1e-15)


# ---------------------------------------------------------------- paged (k8v8) decode

def _contiguous_from_pages(pages, spages, table, lens, page):
    """The contiguous cache [B, Hkv, max_blocks * page, d] that a paged cache stands for,
    read token by token (t -> row t % page of page table[b, t // page])."""
    B, lmax = table.shape[0], table.shape[1] * page
    H, d = pages.shape[1], pages.shape[3]
    c = np.zeros((B, H, lmax, d), pages.dtype)
    s = np.zeros((B, H, lmax), spages.dtype)
    for b in range(B):
        for t in range(int(lens[b])):
            c[b, :, t] = pages[table[b, t // page], :, t % page]
            s[b, :, t] = spages[table[b, t // page], :, t % page]
    return c, s


def _assert_same_decode(a, b):
    for key in ("out", "lse", "o_partial", "lse_partial", "q_codes", "q_scales"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    assert a["logits"].keys() == b["logits"].keys()
    for k in a["logits"]:
        np.testing.assert_array_equal(a["logits"][k], b["logits"][k])


def test_paged_decode_hand_layout():
    # page size 2, one kv head, d 64: tokens 0,1 live in page 1 and token 2 in row 0 of
    # page 0 (row 1 of page 0 holds junk that a length-3 sequence never reads)
    rng = np.random.default_rng(40)
    d = 64
    tok_k = rng.integers(-127, 128, size=(3, d)).astype(np.int8)
    tok_v = rng.integers(-127, 128, size=(3, d)).astype(np.int8)
    tok_ks = np.array([0.01, 0.02, 0.03], np.float32)
    tok_vs = np.array([0.5, 0.25, 0.125], np.float32)
    kp = np.zeros((2, 1, 2, d), np.int8)
    vp = np.zeros((2, 1, 2, d), np.int8)
    ksp = np.zeros((2, 1, 2), np.float32)
    vsp = np.zeros((2, 1, 2), np.float32)
    kp[1, 0, 0], kp[1, 0, 1], kp[0, 0, 0] = tok_k
    vp[1, 0, 0], vp[1, 0, 1], vp[0, 0, 0] = tok_v
    ksp[1, 0, 0], ksp[1, 0, 1], ksp[0, 0, 0] = tok_ks
    vsp[1, 0, 0], vsp[1, 0, 1], vsp[0, 0, 0] = tok_vs
    kp[0, 0, 1] = 127
    vp[0, 0, 1] = -127
    ksp[0, 0, 1] = vsp[0, 0, 1] = 1e3
    table = np.array([[1, 0]], np.int32)
    q = rng.standard_normal((1, 2, d)).astype(np.float32)
    paged = oracle.attn_paged_decode(q, kp, ksp, vp, vsp, table, [3], num_splits=2, want_logits=True)
    kc = np.zeros((1, 1, 4, d), np.int8)
    vc = np.zeros((1, 1, 4, d), np.int8)
    kc[0, 0, :3], vc[0, 0, :3] = tok_k, tok_v
    ks = np.zeros((1, 1, 4), np.float32)
    vs = np.zeros((1, 1, 4), np.float32)
    ks[0, 0, :3], vs[0, 0, :3] = tok_ks, tok_vs
    flat = oracle.attn_decode(q, kc, ks, vc, vs, [3], num_splits=2, want_logits=True)
    _assert_same_decode(paged, flat)
    # and the logits are the plain int dots with the tokens in order
    qc, _ = oracle.quant_rowwise(q)
    np.testing.assert_array_equal(paged["logits"][(0, 1)], tok_k.astype(np.int64) @ qc[0, 1].astype(np.int64))


@pytest.mark.parametrize("page", [16, 64])
def test_paged_decode_equals_contiguous(page):
    rng = np.random.default_rng(41 + page)
    B, hq, hkv, d, max_blocks = 5, 8, 2, 64, 6
    lens = np.array([0, 1, page - 1, page + 1, max_blocks * page])
    need = (lens + page - 1) // page
    num_pages = int(need.sum()) + 3                      # three pages nobody uses
    perm = rng.permutation(num_pages)
    table = np.full((B, max_blocks), -1, np.int32)
    nxt = 0
    for b in range(B):
        table[b, :need[b]] = perm[nxt:nxt + need[b]]
        nxt += need[b]
    kp = rng.integers(-127, 128, size=(num_pages, hkv, page, d)).astype(np.int8)
    vp = rng.integers(-127, 128, size=(num_pages, hkv, page, d)).astype(np.int8)
    ksp = rng.uniform(0.001, 0.05, size=(num_pages, hkv, page)).astype(np.float32)
    vsp = rng.uniform(0.001, 0.05, size=(num_pages, hkv, page)).astype(np.float32)
    q = rng.standard_normal((B, hq, d)).astype(np.float32)
    kc, ks = _contiguous_from_pages(kp, ksp, table, lens, page)
    vc, vs = _contiguous_from_pages(vp, vsp, table, lens, page)
    for ns in (1, 3):
        paged = oracle.attn_paged_decode(q, kp, ksp, vp, vsp, table, lens, num_splits=ns, want_logits=True)
        flat = oracle.attn_decode(q, kc, ks, vc, vs, lens, num_splits=ns, want_logits=True)
        _assert_same_decode(paged, flat)


def test_paged_decode_shared_prefix_pages():
    # sequences 1 and 2 reuse sequence 0's first two pages (a common prompt prefix)
    rng = np.random.default_rng(43)
    page, d, hkv = 16, 64, 1
    table = np.array([[3, 0, 5], [3, 0, 1], [3, 0, 4]], np.int32)
    lens = np.array([40, 33, 48])
    kp = rng.integers(-127, 128, size=(6, hkv, page, d)).astype(np.int8)
    vp = rng.integers(-127, 128, size=(6, hkv, page, d)).astype(np.int8)
    ksp = rng.uniform(0.001, 0.05, size=(6, hkv, page)).astype(np.float32)
    vsp = rng.uniform(0.001, 0.05, size=(6, hkv, page)).astype(np.float32)
    q = np.repeat(rng.standard_normal((1, 2, d)).astype(np.float32), 3, axis=0)
    paged = oracle.attn_paged_decode(q, kp, ksp, vp, vsp, table, lens, num_splits=2)
    kc, ks = _contiguous_from_pages(kp, ksp, table, lens, page)
    vc, vs = _contiguous_from_pages(vp, vsp, table, lens, page)
    flat = oracle.attn_decode(q, kc, ks, vc, vs, lens, num_splits=2)
    _assert_same_decode(paged, flat)
    # the shared prefix really is shared: the 32 common tokens are identical rows
    np.testing.assert_array_equal(kc[0, :, :32], kc[1, :, :32])
    np.testing.assert_array_equal(kc[0, :, :32], kc[2, :, :32])


# ---------------------------------------------------------------- decode with an fp16 V cache

def test_decode_f16v_equals_textbook():
    """fp16-V decode on quantisation-exact K and q rows: no quantisation error is left, so
    it is fp64 softmax attention over the fp16 V values."""
    rng = np.random.default_rng(50)
    B, hq, hkv, lmax, d = 3, 4, 2, 300, 64
    kf, kc, ks = exact_rows(rng, (B, hkv, lmax, d))
    q, _, _ = exact_rows(rng, (B, hq, d))
    v16 = rng.standard_normal((B, hkv, lmax, d)).astype(np.float16)
    lens = np.array([1, 150, 300])
    r = oracle.attn_decode_f16v(q, kc, ks, v16, lens, num_splits=3)
    for b, L in enumerate(lens):
        qq = q[b][:, None, :][None]
        ref = textbook(qq, kf[b][None, :, :L], v16[b][None, :, :L].astype(np.float64), causal=False)[0, :, 0]
        np.testing.assert_allclose(r["out"][b], ref, rtol=0, atol=1e-10)


def test_decode_f16v_equals_int8v_on_exact_v():
    """When every fp16 V value is s_v * code exactly (s_v = 2^-7), the fp16-V decode and the
    int8-V decode are the same sum (up to the order of one fp64 product)."""
    rng = np.random.default_rng(51)
    B, hq, hkv, lmax, d = 2, 8, 2, 200, 128
    q = rng.standard_normal((B, hq, d)).astype(np.float32)
    kc = rng.integers(-127, 128, size=(B, hkv, lmax, d)).astype(np.int8)
    ks = rng.uniform(0.001, 0.05, size=(B, hkv, lmax)).astype(np.float32)
    vc = rng.integers(-127, 128, size=(B, hkv, lmax, d)).astype(np.int8)
    vs = np.full((B, hkv, lmax), 2.0 ** -7, np.float32)
    v16 = (vc.astype(np.float32) * np.float32(2.0 ** -7)).astype(np.float16)
    assert np.array_equal(v16.astype(np.float32), vc.astype(np.float32) / 128)
    lens = np.array([200, 37])
    a = oracle.attn_decode_f16v(q, kc, ks, v16, lens, num_splits=2, want_logits=True)
    b = oracle.attn_decode(q, kc, ks, vc, vs, lens, num_splits=2, want_logits=True)
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(a["lse"], b["lse"])
    for key in b["logits"]:
        np.testing.assert_array_equal(a["logits"][key], b["logits"][key])


# ---------------------------------------------------------------- query chunks (Nq < Nk)

@pytest.mark.parametrize("causal", [True, False])
def test_chunk_equals_tail_of_full_prefill(causal):
    """A chunk of the last Nq queries against all Nk keys is the same computation as rows
    Nk-Nq .. Nk-1 of the full prefill (bottom-right alignment; same K mean and codes)."""
    rng = np.random.default_rng(60)
    B, hq, hkv, nk, d = 2, 4, 2, 200, 64
    qf = rng.standard_normal((B, hq, nk, d)).astype(np.float32)
    k = (rng.standard_normal((B, hkv, nk, d)) + 3.0).astype(np.float32)
    v = rng.standard_normal((B, hkv, nk, d)).astype(np.float32)
    full = oracle.attn_prefill(qf, k, v, causal=causal, smooth_k=True, want_logits=True)
    for nq in (1, 57, 200):
        off = nk - nq
        part = oracle.attn_prefill(qf[:, :, off:], k, v, causal=causal, smooth_k=True, want_logits=True)
        np.testing.assert_array_equal(part["out"], full["out"][:, :, off:])
        np.testing.assert_array_equal(part["lse"], full["lse"][:, :, off:])
        np.testing.assert_array_equal(part["k_codes"], full["k_codes"])
        for (s, h, i), lg in part["logits"].items():
            np.testing.assert_array_equal(lg, full["logits"][(s, h, i + off)])


def test_chunk_equals_textbook_bottom_right_mask():
    rng = np.random.default_rng(61)
    B, hq, hkv, nq, nk, d = 1, 4, 2, 40, 100, 64
    qf, _, _ = exact_rows(rng, (B, hq, nq, d))
    kf, _, _ = exact_rows(rng, (B, hkv, nk, d))
    v = rng.standard_normal((B, hkv, nk, d)).astype(np.float32)
    r = oracle.attn_prefill(qf, kf, v, causal=True, smooth_k=False)
    g = hq // hkv
    mask = torch.ones((nq, nk), dtype=torch.bool).tril(diagonal=nk - nq)   # j <= i + nk - nq
    qt = torch.from_numpy(qf.astype(np.float64))
    kt = torch.from_numpy(kf.astype(np.float64)).repeat_interleave(g, dim=1)
    vt = torch.from_numpy(v.astype(np.float64)).repeat_interleave(g, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask).numpy()
    np.testing.assert_allclose(r["out"], ref, rtol=0, atol=1e-10)
    assert mask[0].sum() == nk - nq + 1 and mask[-1].all()


# ---------------------------------------------------------------- verify mask (speculative decoding)

def _verify_case(rng, B=2, T=4, hq=4, hkv=2, lmax=64, d=64, lens=(40, 64)):
    q = rng.standard_normal((B, T, hq, d)).astype(np.float32)
    kc = rng.integers(-127, 128, size=(B, hkv, lmax, d)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(B, hkv, lmax, d)).astype(np.int8)
    ks = rng.uniform(0.001, 0.05, size=(B, hkv, lmax)).astype(np.float32)
    vs = rng.uniform(0.001, 0.05, size=(B, hkv, lmax)).astype(np.float32)
    return q, kc, ks, vc, vs, np.array(lens)


def test_verify_chain_mask_equals_decode_prefixes():
    """A chain of drafts (query t sees drafts 0..t) is decode of query t at length
    L - T + t + 1."""
    rng = np.random.default_rng(70)
    q, kc, ks, vc, vs, lens = _verify_case(rng)
    T = q.shape[1]
    chain = np.array([[(1 << (t + 1)) - 1 for t in range(T)]] * len(lens), np.uint32)
    r = oracle.attn_decode_verify(q, kc, ks, vc, vs, lens, chain)
    for t in range(T):
        ref = oracle.attn_decode(q[:, t], kc, ks, vc, vs, lens - T + t + 1, num_splits=1)
        np.testing.assert_allclose(r["out"][:, t], ref["out"], rtol=0, atol=1e-13)
        np.testing.assert_allclose(r["lse"][:, t], ref["lse"], rtol=0, atol=1e-13)


def test_verify_full_mask_equals_decode():
    rng = np.random.default_rng(71)
    q, kc, ks, vc, vs, lens = _verify_case(rng)
    T = q.shape[1]
    full = np.full((len(lens), T), (1 << T) - 1, np.uint32)
    r = oracle.attn_decode_verify(q, kc, ks, vc, vs, lens, full)
    for t in range(T):
        ref = oracle.attn_decode(q[:, t], kc, ks, vc, vs, lens, num_splits=1)
        np.testing.assert_allclose(r["out"][:, t], ref["out"], rtol=0, atol=1e-13)


def test_verify_tree_mask_drops_siblings():
    """Two sibling drafts (each sees only itself): query 1 must not see draft 0, i.e. it
    equals decode over a cache with draft 0's row removed."""
    rng = np.random.default_rng(72)
    q, kc, ks, vc, vs, lens = _verify_case(rng, B=1, T=2, lens=(30,))
    mask = np.array([[0b01, 0b10]], np.uint32)
    r = oracle.attn_decode_verify(q, kc, ks, vc, vs, lens, mask)
    keep = [i for i in range(30) if i != 28]                      # draft 0 sits at position 28
    kc2, ks2 = kc[:, :, keep], ks[:, :, keep]
    vc2, vs2 = vc[:, :, keep], vs[:, :, keep]
    ref = oracle.attn_decode(q[:, 1], kc2, ks2, vc2, vs2, [29], num_splits=1)
    np.testing.assert_allclose(r["out"][:, 1], ref["out"], rtol=0, atol=1e-13)
    ref0 = oracle.attn_decode(q[:, 0], kc, ks, vc, vs, [29], num_splits=1)   # draft 0 sees positions 0..28
    np.testing.assert_allclose(r["out"][:, 0], ref0["out"], rtol=0, atol=1e-13)


def _chunk_cache_case(rng, B=2, hq=4, hkv=2, nq=5, nk=40, lmax=48, d=64):
    q = rng.standard_normal((B, hq, nq, d)).astype(np.float32)
    kc = rng.integers(-127, 128, size=(B, hkv, lmax, d)).astype(np.int8)
    # every key row reaches +-127, so that re-quantising code * scale gives the codes back
    kc[..., 0] = np.where(rng.random((B, hkv, lmax)) < 0.5, 127, -127).astype(np.int8)
    vc = rng.integers(-127, 128, size=(B, hkv, lmax, d)).astype(np.int8)
    ks = rng.uniform(0.001, 0.05, size=(B, hkv, lmax)).astype(np.float32)
    vs = rng.uniform(0.001, 0.05, size=(B, hkv, lmax)).astype(np.float32)
    return q, kc, ks, vc, vs, nk


@pytest.mark.parametrize("causal", [True, False])
def test_chunk_cache_equals_prefill_chunk_on_dequantised_cache(causal):
    """The chunk against an int8 cache is the prefill chunk (bottom-right, no smoothing)
    whose K and V are the cache's code * scale: the prefill's own per-row quantisation of
    K returns the cache's codes (every row holds a +-127), up to fp32 rounding of the
    products."""
    rng = np.random.default_rng(80)
    q, kc, ks, vc, vs, nk = _chunk_cache_case(rng)
    r = oracle.attn_chunk_cache(q, kc, ks, vc, vs, nk, causal=causal)
    kf = (kc[:, :, :nk].astype(np.float32) * ks[:, :, :nk, None]).astype(np.float32)
    vf = (vc[:, :, :nk].astype(np.float32) * vs[:, :, :nk, None]).astype(np.float32)
    ref = oracle.attn_prefill(q, kf, vf, causal=causal, smooth_k=False)
    np.testing.assert_allclose(r["out"], ref["out"], rtol=0, atol=1e-6)
    np.testing.assert_allclose(r["lse"], ref["lse"], rtol=0, atol=1e-6)


def test_chunk_cache_single_query_is_decode():
    """A one-query chunk is the decode of that query over the whole cache (length nk)."""
    rng = np.random.default_rng(81)
    q, kc, ks, vc, vs, nk = _chunk_cache_case(rng, nq=1)
    r = oracle.attn_chunk_cache(q, kc, ks, vc, vs, nk)
    ref = oracle.attn_decode(q[:, :, 0], kc, ks, vc, vs, np.full(q.shape[0], nk), num_splits=1)
    np.testing.assert_allclose(r["out"][:, :, 0], ref["out"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["lse"][:, :, 0], ref["lse"], rtol=0, atol=1e-13)
