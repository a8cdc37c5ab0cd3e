"""GPU parity of the split-KV int8-cache decode (and its combine) against the oracle.

Operation: the "SuperL8" README, "Attention kernels" table, attn_decode (split-KV
decode with an int8 KV cache, int8-V variant).  The cache is built from the same
seeded fp32 values on both sides: the GPU path quantises them with
sl8_quant_rowwise, the oracle with its own quantiser, and the two caches must be
byte-identical.  Bit-exact: q codes/scales and int32 logits; outputs within the
tolerances of tests/_parity.py.
"""
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    from w8a8_int8_flashattention_gb300 import build
    build.build()
    sl8.lib()


def build_cache(w, lmax, batches=None):
    """GPU and oracle caches for workload w: codes [B,Hkv,Lmax,d] int8, scales [B,Hkv,Lmax]."""
    B, Hkv, d = w.B, w.Hkv, w.d
    lens = W.seq_lengths(w)
    g = {n: torch.zeros((B, Hkv, lmax, d), dtype=torch.int8, device=DEV) for n in ("k", "v")}
    gs = {n: torch.zeros((B, Hkv, lmax), dtype=torch.float32, device=DEV) for n in ("k", "v")}
    o = {n: np.zeros((B, Hkv, lmax, d), np.int8) for n in ("k", "v")}
    os_ = {n: np.zeros((B, Hkv, lmax), np.float32) for n in ("k", "v")}
    for b in range(B):
        L = int(lens[b])
        for n in ("k", "v"):
            vals = W.decode_cache_values(w, b, n)  # [Hkv, L, d] fp32
            c, s = sl8.quant_rowwise(torch.from_numpy(vals).to(DEV))
            g[n][b, :, :L] = c
            gs[n][b, :, :L] = s
            if batches is None or b in batches:
                oc, osc = oracle.quant_rowwise(vals)
                o[n][b, :, :L] = oc
                os_[n][b, :, :L] = osc
    return lens, g, gs, o, os_


CASES = [
    # wid, B, Hq, Hkv, d, lengths, lmax
    (3001, 6, 8, 2, 128, [1, 255, 256, 257, 700, 0], 700),
    (3002, 3, 4, 4, 64, [513, 1, 1024], 1024),
    (3003, 3, 8, 1, 256, [129, 300, 5], 300),
    (3004, 2, 16, 2, 128, [2000, 77], 2000),
    # MQA beyond 8 query heads per kv head: virtual kv heads of <= 8 query heads each
    (3005, 3, 32, 1, 128, [900, 1, 333], 900),          # G = 32: four groups of 8
    (3006, 2, 64, 4, 64, [700, 129], 700),               # G = 16: two groups of 8
    (3007, 2, 12, 1, 256, [300, 17], 300),               # G = 12: two groups of 6
    # head dim 32 (32-byte cache rows)
    (3008, 4, 8, 2, 32, [1, 300, 0, 161], 320),
    (3009, 2, 16, 1, 32, [500, 33], 500),                # G = 16 at d = 32
]


@pytest.mark.parametrize("case", CASES, ids=[f"w{c[0]}_d{c[4]}_G{c[2] // c[3]}" for c in CASES])
def test_decode_small(case):
    wid, B, Hq, Hkv, d, lens, lmax = case
    w = W.custom(wid, kind="decode", B=B, Hq=Hq, Hkv=Hkv, d=d, dtype="bf16", extra={"lengths": lens})
    lens_np, g, gs, o, os_ = build_cache(w, lmax)
    torch.cuda.synchronize()
    for n in ("k", "v"):
        np.testing.assert_array_equal(g[n].cpu().numpy(), o[n])
        np.testing.assert_array_equal(gs[n].cpu().numpy(), os_[n])
    q = W.decode_query(w)
    qd = q.to(DEV)
    seq = torch.from_numpy(lens_np.astype(np.int32)).to(DEV)
    dbg = sl8.attn_int8_decode_logits_debug(qd, g["k"], gs["k"], g["v"], gs["v"], seq)
    ref = oracle.attn_decode(q.float().numpy(), o["k"], os_["k"], o["v"], os_["v"], lens_np, num_splits=1,
                             want_logits=True)
    np.testing.assert_array_equal(dbg["q_codes"].cpu().numpy(), ref["q_codes"])
    np.testing.assert_array_equal(dbg["q_scales"].cpu().numpy(), ref["q_scales"])
    lg = dbg["logits"].cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_array_equal(lg[b, h, :lens_np[b]], ref["logits"][(b, h)])
    outs = {}
    for ns in (0, 1, 3, 7):
        o32, lse = sl8.attn_int8_decode(qd, g["k"], gs["k"], g["v"], gs["v"], seq, num_splits=ns,
                                        out_dtype=torch.float32, return_lse=True)
        ob = sl8.attn_int8_decode(qd, g["k"], gs["k"], g["v"], gs["v"], seq, num_splits=ns)
        torch.cuda.synchronize()
        outs[ns] = to_np32(o32)
        check_f32(outs[ns], ref["out"], f"w{wid} splits={ns} f32")
        check_half(ob, ref["out"], f"w{wid} splits={ns} bf16")
        ok = lens_np > 0
        np.testing.assert_allclose(to_np32(lse)[ok], ref["lse"][ok], rtol=0, atol=1e-4)
        assert np.all(np.isneginf(to_np32(lse)[~ok]))
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_OK, (st, site)


def test_decode_partials_match_oracle_splits():
    w = W.custom(3101, kind="decode", B=2, Hq=4, Hkv=2, d=128, dtype="bf16", extra={"lengths": [600, 130]})
    lens_np, g, gs, o, os_ = build_cache(w, 600)
    q = W.decode_query(w)
    seq = torch.from_numpy(lens_np.astype(np.int32)).to(DEV)
    op, lp = sl8.attn_int8_decode_splitkv(q.to(DEV), g["k"], gs["k"], g["v"], gs["v"], seq, num_splits=4)
    torch.cuda.synchronize()
    split_size = sl8.lib().sl8_attn_decode_split_size(2, 2, 600, 128, 4)   # one 160-token stage
    assert split_size == 160 and op.shape[2] == 4
    ref = oracle.attn_decode(q.float().numpy(), o["k"], os_["k"], o["v"], os_["v"], lens_np, split_size=split_size)
    lpn = to_np32(lp)
    live = np.isfinite(ref["lse_partial"])
    np.testing.assert_array_equal(np.isneginf(lpn), ~live)
    np.testing.assert_allclose(lpn[live], ref["lse_partial"][live], rtol=0, atol=1e-4)
    check_f32(to_np32(op)[live], ref["o_partial"][live], "partials")


def test_full_size_decode_workload():
    """The benchmark decode (B64 Hq32 Hkv8 d128, L ~ U[1024, 8192]) in the bench's launch
    configuration (automatic split count): every sequence and head against the oracle,
    the int8 caches byte for byte, q codes, scales and every int32 logit bit for bit."""
    w = W.get("decode")
    lens_np, g, gs, o, os_ = build_cache(w, w.lmax)
    q = W.decode_query(w)
    seq = torch.from_numpy(lens_np.astype(np.int32)).to(DEV)
    o32, lse = sl8.attn_int8_decode(q.to(DEV), g["k"], gs["k"], g["v"], gs["v"], seq, out_dtype=torch.float32,
                                    return_lse=True)
    ob = sl8.attn_int8_decode(q.to(DEV), g["k"], gs["k"], g["v"], gs["v"], seq)
    dbg = sl8.attn_int8_decode_logits_debug(q.to(DEV), g["k"], gs["k"], g["v"], gs["v"], seq)
    torch.cuda.synchronize()
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_OK, (st, site)
    for n in ("k", "v"):
        np.testing.assert_array_equal(g[n].cpu().numpy(), o[n])
        np.testing.assert_array_equal(gs[n].cpu().numpy(), os_[n])
    ref = oracle.attn_decode(q.float().numpy(), o["k"], os_["k"], o["v"], os_["v"], lens_np, want_logits=True)
    np.testing.assert_array_equal(dbg["q_codes"].cpu().numpy(), ref["q_codes"])
    np.testing.assert_array_equal(dbg["q_scales"].cpu().numpy(), ref["q_scales"])
    check_f32(to_np32(o32), ref["out"], "decode full f32, every sequence and head")
    check_half(ob, ref["out"], "decode full bf16, every sequence and head")
    np.testing.assert_allclose(to_np32(lse), ref["lse"], rtol=0, atol=1e-4)
    lg = dbg["logits"].cpu().numpy()
    for b in range(w.B):
        for h in range(w.Hq):
            np.testing.assert_array_equal(lg[b, h, :lens_np[b]], ref["logits"][(b, h)], err_msg=f"logits {(b, h)}")


# ---------------------------------------------------------------- paged (k8v8) cache

PAGED = [
    # wid, B, Hq, Hkv, d, lengths, page_size, max_blocks, shared prefix blocks
    (3201, 5, 8, 2, 128, [1, 255, 256, 700, 0], 16, 44, 0),
    (3202, 3, 4, 4, 64, [513, 17, 1024], 64, 16, 0),
    (3203, 3, 8, 1, 256, [129, 300, 5], 32, 10, 0),
    (3204, 4, 16, 2, 128, [2000, 77, 160, 161], 256, 8, 0),
    (3205, 4, 8, 2, 128, [900, 640, 1000, 700], 128, 8, 5),
    (3206, 3, 32, 2, 128, [700, 33, 1000], 64, 16, 0),   # G = 16 over a paged cache
    (3207, 3, 8, 2, 32, [100, 17, 640], 32, 20, 0),      # d = 32 over a paged cache
]


@pytest.mark.parametrize("case", PAGED, ids=[f"w{c[0]}_d{c[4]}_P{c[6]}" for c in PAGED])
def test_paged_decode(case):
    """Paged split-KV decode: parity with the oracle's paged decode, and the same bits as
    the contiguous-cache kernel on the same tokens (same Lmax, same split plan)."""
    wid, B, Hq, Hkv, d, lens, page, max_blocks, shared = case
    lmax = page * max_blocks
    w = W.custom(wid, kind="decode", B=B, Hq=Hq, Hkv=Hkv, d=d, dtype="bf16", extra={"lengths": lens})
    lens_np, g, gs, o, os_ = build_cache(w, lmax)
    if shared:
        # sequences 1.. share sequence 0's first `shared` blocks: give them the same rows
        n = shared * page
        for b in range(1, B):
            for src, dst in ((g, g), (gs, gs), (o, o), (os_, os_)):
                for key in ("k", "v"):
                    dst[key][b, :, :n] = src[key][0, :, :n]
    table, num_pages = W.page_table(w, lens_np, page, max_blocks=max_blocks, spare=3, shared_prefix=shared)
    gp, op_ = {}, {}
    for key in ("k", "v"):
        gp[key] = W.paginate(g[key], gs[key], table, lens_np, page, num_pages)
        op_[key] = W.paginate(o[key], os_[key], table, lens_np, page, num_pages)
    q = W.decode_query(w)
    qd = q.to(DEV)
    seq = torch.from_numpy(lens_np.astype(np.int32)).to(DEV)
    tab = torch.from_numpy(table).to(DEV)
    for ns in (0, 1, 3):
        ref = oracle.attn_paged_decode(q.float().numpy(), op_["k"][0], op_["k"][1], op_["v"][0], op_["v"][1],
                                       table, lens_np, split_size=sl8.lib().sl8_attn_decode_split_size(
                                           B, Hkv, lmax, d, ns))
        o32, lse = sl8.attn_int8_paged_decode(qd, gp["k"][0], gp["k"][1], gp["v"][0], gp["v"][1], tab, seq,
                                              num_splits=ns, out_dtype=torch.float32, return_lse=True)
        ob = sl8.attn_int8_paged_decode(qd, gp["k"][0], gp["k"][1], gp["v"][0], gp["v"][1], tab, seq,
                                        num_splits=ns)
        flat32 = sl8.attn_int8_decode(qd, g["k"], gs["k"], g["v"], gs["v"], seq, num_splits=ns,
                                      out_dtype=torch.float32)
        torch.cuda.synchronize()
        check_f32(to_np32(o32), ref["out"], f"w{wid} paged splits={ns} f32")
        check_half(ob, ref["out"], f"w{wid} paged splits={ns} bf16")
        ok = lens_np > 0
        np.testing.assert_allclose(to_np32(lse)[ok], ref["lse"][ok], rtol=0, atol=1e-4)
        assert np.all(np.isneginf(to_np32(lse)[~ok]))
        assert torch.equal(o32, flat32), f"w{wid} splits={ns}: paged and contiguous kernels differ"
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_OK, (st, site)


def test_paged_decode_bad_page_is_reported():
    """A block-table entry outside [0, num_pages) is reported on the device (and page 0 is
    read instead); the context stays usable."""
    w = W.custom(3206, kind="decode", B=2, Hq=4, Hkv=2, d=128, dtype="bf16", extra={"lengths": [100, 40]})
    lens_np, g, gs, o, os_ = build_cache(w, 128)
    table, num_pages = W.page_table(w, lens_np, 16, max_blocks=8)
    pk = W.paginate(g["k"], gs["k"], table, lens_np, 16, num_pages)
    pv = W.paginate(g["v"], gs["v"], table, lens_np, 16, num_pages)
    bad = table.copy()
    bad[0, 3] = num_pages + 7
    q = W.decode_query(w).to(DEV)
    seq = torch.from_numpy(lens_np.astype(np.int32)).to(DEV)
    sl8.last_device_status()
    sl8.attn_int8_paged_decode(q, pk[0], pk[1], pv[0], pv[1], torch.from_numpy(bad).to(DEV), seq)
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_ERR_DEVICE_ARG, (st, site)
    out = sl8.attn_int8_paged_decode(q, pk[0], pk[1], pv[0], pv[1], torch.from_numpy(table).to(DEV), seq)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert sl8.last_device_status()[0] == sl8.SL8_OK


# ---------------------------------------------------------------- fp16 V cache

F16V = [
    # wid, B, Hq, Hkv, d, lengths, lmax
    (3401, 6, 8, 2, 128, [1, 255, 256, 257, 700, 0], 700),
    (3402, 3, 4, 4, 64, [513, 1, 1024], 1024),
    (3403, 2, 16, 2, 128, [2000, 77], 2000),
    (3404, 3, 8, 8, 64, [160, 161, 3000], 3000),
    (3405, 2, 32, 1, 128, [1500, 200], 1500),           # G = 32 with an fp16 V cache
]


@pytest.mark.parametrize("case", F16V, ids=[f"w{c[0]}_d{c[4]}_G{c[2] // c[3]}" for c in F16V])
def test_decode_f16v(case):
    """int8 K + fp16 V decode against the oracle's fp16-V decode."""
    wid, B, Hq, Hkv, d, lens, lmax = case
    w = W.custom(wid, kind="decode", B=B, Hq=Hq, Hkv=Hkv, d=d, dtype="bf16", extra={"lengths": lens})
    lens_np, g, gs, o, os_ = build_cache(w, lmax)
    v16 = torch.zeros((B, Hkv, lmax, d), dtype=torch.float16)
    for b in range(B):
        v16[b, :, :int(lens_np[b])] = torch.from_numpy(W.decode_cache_values(w, b, "v")).to(torch.float16)
    vd = v16.to(DEV)
    q = W.decode_query(w)
    qd = q.to(DEV)
    seq = torch.from_numpy(lens_np.astype(np.int32)).to(DEV)
    for ns in (0, 1, 3):
        ref = oracle.attn_decode_f16v(q.float().numpy(), o["k"], os_["k"], v16.numpy(), lens_np,
                                      split_size=sl8.lib().sl8_attn_decode_split_size(B, Hkv, lmax, d, ns))
        o32, lse = sl8.attn_int8_decode_f16v(qd, g["k"], gs["k"], vd, seq, num_splits=ns, out_dtype=torch.float32,
                                             return_lse=True)
        ob = sl8.attn_int8_decode_f16v(qd, g["k"], gs["k"], vd, seq, num_splits=ns)
        torch.cuda.synchronize()
        check_f32(to_np32(o32), ref["out"], f"w{wid} f16v splits={ns} f32")
        check_half(ob, ref["out"], f"w{wid} f16v splits={ns} bf16")
        ok = lens_np > 0
        np.testing.assert_allclose(to_np32(lse)[ok], ref["lse"][ok], rtol=0, atol=1e-4)
        assert np.all(np.isneginf(to_np32(lse)[~ok]))
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_OK, (st, site)


@pytest.mark.parametrize("d", [32, 256])
def test_decode_f16v_rejects_d32_d256(d):
    q = torch.zeros((1, 2, d), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((1, 1, 64, d), dtype=torch.int8, device=DEV)
    ks = torch.ones((1, 1, 64), dtype=torch.float32, device=DEV)
    v = torch.zeros((1, 1, 64, d), dtype=torch.float16, device=DEV)
    seq = torch.tensor([10], dtype=torch.int32, device=DEV)
    with pytest.raises(sl8.SL8Error):
        sl8.attn_int8_decode_splitkv_f16v(q, kc, ks, v, seq)


# ---------------------------------------------------------------- speculative verify (tree mask)

VERIFY = [
    # wid, B, T, Hq, Hkv, d, lengths (draft tokens included), lmax
    (3501, 3, 4, 8, 2, 128, [300, 4, 1000], 1000),
    (3502, 2, 7, 4, 4, 64, [513, 160], 600),
    (3503, 2, 16, 8, 1, 256, [200, 2000], 2000),
    (3504, 4, 1, 8, 2, 128, [1, 17, 640, 641], 700),
    (3505, 2, 4, 8, 2, 32, [300, 64], 400),
]


@pytest.mark.parametrize("case", VERIFY, ids=[f"w{c[0]}_T{c[2]}_d{c[5]}" for c in VERIFY])
def test_decode_verify(case):
    wid, B, T, Hq, Hkv, d, lens, lmax = case
    w = W.custom(wid, kind="decode", B=B, Hq=Hq, Hkv=Hkv, d=d, dtype="bf16", extra={"lengths": lens})
    lens_np, g, gs, o, os_ = build_cache(w, lmax)
    rng = np.random.default_rng(wid)
    q = torch.from_numpy(rng.standard_normal((B, T, Hq, d)).astype(np.float32)).to(torch.bfloat16)
    # row 0: a chain; other rows: random trees (every query sees itself and some earlier drafts)
    mask = np.zeros((B, T), np.int64)
    for b in range(B):
        for t in range(T):
            if b == 0:
                mask[b, t] = (1 << (t + 1)) - 1
            else:
                anc = rng.integers(0, 2, size=t) if t else np.zeros(0, np.int64)
                mask[b, t] = (1 << t) | int(sum(int(x) << i for i, x in enumerate(anc)))
    mask32 = torch.from_numpy(mask.astype(np.uint32).view(np.int32)).to(DEV)
    qd = q.to(DEV)
    seq = torch.from_numpy(lens_np.astype(np.int32)).to(DEV)
    ref = oracle.attn_decode_verify(q.float().numpy(), o["k"], os_["k"], o["v"], os_["v"], lens_np, mask)
    for ns in (0, 3):
        o32, lse = sl8.attn_int8_decode_verify(qd, g["k"], gs["k"], g["v"], gs["v"], seq, mask32, num_splits=ns,
                                               out_dtype=torch.float32, return_lse=True)
        ob = sl8.attn_int8_decode_verify(qd, g["k"], gs["k"], g["v"], gs["v"], seq, mask32, num_splits=ns)
        torch.cuda.synchronize()
        check_f32(to_np32(o32), ref["out"], f"w{wid} verify splits={ns} f32")
        check_half(ob, ref["out"], f"w{wid} verify splits={ns} bf16")
        np.testing.assert_allclose(to_np32(lse), ref["lse"], rtol=0, atol=1e-4)
    if T == 1:
        # one draft that sees itself is plain decode.  Not bit for bit: the masked tail unit
        # may contract its arithmetic differently, and a last-bit change of p can move P'
        # by one fp16 ulp (2^-11 relative)
        plain = sl8.attn_int8_decode(qd[:, 0].contiguous(), g["k"], gs["k"], g["v"], gs["v"], seq,
                                     out_dtype=torch.float32)
        torch.cuda.synchronize()
        np.testing.assert_allclose(to_np32(o32[:, 0]), to_np32(plain), rtol=0, atol=5e-4)
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_OK, (st, site)


@pytest.mark.parametrize("qdt", ["f16", "f32"])
def test_decode_query_dtypes(qdt):
    """q in fp16 or fp32 (quantised inside the kernel like bf16): codes and logits bit-exact,
    outputs within tolerance, for plain decode and for verify."""
    B, Hq, Hkv, d, lens, lmax = 3, 8, 2, 128, [700, 33, 1], 700
    w = W.custom(3601, kind="decode", B=B, Hq=Hq, Hkv=Hkv, d=d, dtype=qdt, extra={"lengths": lens})
    lens_np, g, gs, o, os_ = build_cache(w, lmax)
    q = W.decode_query(w)
    qd = q.to(DEV)
    seq = torch.from_numpy(lens_np.astype(np.int32)).to(DEV)
    dbg = sl8.attn_int8_decode_logits_debug(qd, g["k"], gs["k"], g["v"], gs["v"], seq)
    ref = oracle.attn_decode(q.float().numpy(), o["k"], os_["k"], o["v"], os_["v"], lens_np, want_logits=True)
    np.testing.assert_array_equal(dbg["q_codes"].cpu().numpy(), ref["q_codes"])
    np.testing.assert_array_equal(dbg["q_scales"].cpu().numpy(), ref["q_scales"])
    lg = dbg["logits"].cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_array_equal(lg[b, h, :lens_np[b]], ref["logits"][(b, h)])
    o32 = sl8.attn_int8_decode(qd, g["k"], gs["k"], g["v"], gs["v"], seq, out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_f32(to_np32(o32), ref["out"], f"q {qdt} f32")
    # verify with a 2-draft chain on the same cache
    rng = np.random.default_rng(3602)
    qv = torch.from_numpy(rng.standard_normal((B, 2, Hq, d)).astype(np.float32)).to(W.torch_dtype(qdt))
    mask = np.array([[1, 3]] * B, np.int64)
    refv = oracle.attn_decode_verify(qv.float().numpy(), o["k"], os_["k"], o["v"], os_["v"], lens_np, mask)
    ov = sl8.attn_int8_decode_verify(qv.to(DEV), g["k"], gs["k"], g["v"], gs["v"], seq,
                                     torch.from_numpy(mask.astype(np.int32)).to(DEV), out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_f32(to_np32(ov), refv["out"], f"q {qdt} verify f32")
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_OK, (st, site)


CHUNK_CACHE_CASES = [
    # wid, B, Hq, Hkv, d, Nq, Nk, Lmax, causal, q dtype
    (4101, 2, 8, 2, 128, 200, 700, 760, True, "bf16"),
    (4102, 1, 4, 4, 64, 96, 96, 128, True, "f16"),       # the chunk is the whole sequence
    (4103, 1, 8, 1, 256, 130, 1000, 1000, True, "bf16"),  # MQA at d = 256
    (4104, 1, 4, 2, 128, 64, 2048, 2048, True, "bf16"),   # two items: keys split 8 ways
    (4105, 2, 4, 2, 32, 50, 300, 320, False, "f16"),      # head dim 32, not causal
    (4106, 1, 8, 2, 128, 300, 300, 300, False, "bf16"),
]


@pytest.mark.parametrize("case", CHUNK_CACHE_CASES, ids=[f"w{c[0]}_d{c[4]}_nq{c[5]}" for c in CHUNK_CACHE_CASES])
def test_chunk_onto_int8_cache(case):
    """A query chunk against an int8 cache that already holds its keys, against the
    oracle: every output row, in fp32 and in the query dtype, and the LSE."""
    wid, B, Hq, Hkv, d, nq, nk, lmax, causal, qdt = case
    w = W.custom(wid, kind="decode", B=B, Hq=Hq, Hkv=Hkv, d=d, dtype=qdt, extra={"lengths": [nk] * B})
    _, g, gs, o, os_ = build_cache(w, lmax)
    q = W.chunk_query(w, nq)
    qd = q.to(DEV)
    ref = oracle.attn_chunk_cache(q.float().numpy(), o["k"], os_["k"], o["v"], os_["v"], nk, causal=causal)
    o32, lse = sl8.attn_int8_fwd_chunk_cache(qd, g["k"], gs["k"], g["v"], gs["v"], Nk=nk, causal=causal,
                                             out_dtype=torch.float32, return_lse=True)
    oh = sl8.attn_int8_fwd_chunk_cache(qd, g["k"], gs["k"], g["v"], gs["v"], Nk=nk, causal=causal)
    torch.cuda.synchronize()
    check_f32(to_np32(o32), ref["out"], f"w{wid} f32")
    check_half(oh, ref["out"], f"w{wid} {qdt}")
    np.testing.assert_allclose(to_np32(lse), ref["lse"], rtol=0, atol=1e-4)
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_OK, (st, site)


def test_chunk_onto_int8_cache_rejects_bad_shapes():
    w = W.custom(4107, kind="decode", B=1, Hq=4, Hkv=2, d=64, dtype="bf16", extra={"lengths": [64]})
    _, g, gs, _, _ = build_cache(w, 64)
    q = W.chunk_query(w, 16).to(DEV)
    with pytest.raises(RuntimeError):  # Nk > Lmax
        sl8.attn_int8_fwd_chunk_cache(q, g["k"], gs["k"], g["v"], gs["v"], Nk=65)
    with pytest.raises(RuntimeError):  # Nq > Nk
        sl8.attn_int8_fwd_chunk_cache(q, g["k"], gs["k"], g["v"], gs["v"], Nk=8)
