"""CPU oracle for the W8A8 INT8 attention path: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) import this package.  The library in
``w8a8_int8_flashattention_gb300`` shares no code with it and never calls it.

The arithmetic lives in ``sl8_oracle.c`` (plain C, strict IEEE fp32 for the
quantiser, fp64 for everything after the int32 dot); this module only compiles
it with gcc, lays out the per-(sequence, head) slices and loops over them.

Sources: the "SuperL8" README (github.com/jajmangold/superl8) -- "Attention
kernels" table (attn_int8_fwd: W8A8 FlashAttention-2, causal, GQA/MQA, head dims
32/64/128/256; attn_varlen_fwd: ragged prefill; attn_decode: split-KV decode over
an int8 KV cache, int8-V and fp16-V variants; attn_paged_decode over a paged cache, with the
"Engine" table's k8v8 format), "Supporting kernels" table (quant_rowwise:
symmetric per-row int8), "Quantization" table (per-row int8 with K-smoothing) and
the "Quick start" section (q [B,Hq,N,d], k/v [B,Hkv,N,d], quantises internally);
the "SuperL8-serve" README's "Engine" table (chunked prefill onto the KV cache).
The readings that fill what the pages leave open are restated in ``sl8_oracle.c``
(R1-R13) and in the docstrings below (the later ones, up to R22).

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, hand-derived golden fixtures, textbook fp64 attention on
quantisation-exact inputs, invariants, brute force on tiny inputs).  The end-to-end
INT8 accuracy against unquantised attention is *parity unpinned*: the pages give
no error bound for it, so it is reported, never asserted.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sl8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_F32P = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_F64P = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_I8P = np.ctypeslib.ndpointer(dtype=np.int8, flags="C_CONTIGUOUS")
_I32P = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_I64P = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile ``sl8_oracle.c`` into ``liboracle.so`` (gcc, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_quant_rows.argtypes = [_F32P, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_int64, _I8P, _F32P]
            lib.oracle_k_mean.argtypes = [_F32P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _F32P]
            lib.oracle_quant_groups.argtypes = [_F32P, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                                ctypes.c_int64, ctypes.c_float, _I8P, _F32P, ctypes.c_void_p]
            lib.oracle_attn_prefill_head.restype = ctypes.c_int
            lib.oracle_attn_prefill_head.argtypes = [
                _I8P, _F32P, _I8P, _F32P, _F32P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, _F64P, _F64P, ctypes.c_void_p]
            lib.oracle_decode_row.restype = ctypes.c_int
            lib.oracle_decode_row.argtypes = [
                _I8P, ctypes.c_float, _I8P, _F32P, _I8P, _F32P, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int64, ctypes.c_int, _F64P, _F64P, ctypes.c_void_p]
            lib.oracle_decode_row_fv.restype = ctypes.c_int
            lib.oracle_decode_row_fv.argtypes = [
                _I8P, ctypes.c_float, _I8P, _F32P, _F32P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int, _F64P, _F64P, ctypes.c_void_p]
            lib.oracle_decode_combine.argtypes = [_F64P, _F64P, ctypes.c_int, ctypes.c_int, _F64P, _F64P]
            _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use (OMP_NUM_THREADS or all cores)."""
    return int(_load().oracle_num_threads())


def _f32(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.float32:
        raise TypeError(f"oracle wants float32 arrays (widen fp16/bf16 first), got {a.dtype}")
    return np.ascontiguousarray(a)


# ------------------------------------------------------------------ quantisation

def quant_rowwise(x, mu=None, rows_per_group=None):
    """Symmetric per-row int8 quantisation (readings R1, R3), rows along the last axis.

    x: float32 [..., d].  mu: optional float32 [groups, d] subtracted from each row
    first, row r (flattened) using group r // rows_per_group.
    Returns (codes int8 [..., d], scales float32 [...]).
    """
    x = _f32(x)
    d = x.shape[-1]
    rows = x.size // d if d else 0
    codes = np.zeros(x.shape, np.int8)
    scales = np.zeros(x.shape[:-1], np.float32)
    if rows == 0:
        return codes, scales
    mu_ptr = None
    if mu is not None:
        mu = _f32(mu)
        if rows_per_group is None:
            rows_per_group = rows
        mu_ptr = mu.ctypes.data
    _load().oracle_quant_rows(x.reshape(rows, d), rows, d, mu_ptr, int(rows_per_group or 1),
                              codes.reshape(rows, d), scales.reshape(rows))
    return codes, scales


def quant_groups(x, group, tau=0.0, mu=None):
    """Grouped symmetric int8 quantisation with outlier rows (reading R21).

    x: float32 [n, d], the rows of one sequence and head in token order; mu: optional
    float32 [d] subtracted first.  Rows form groups of ``group`` consecutive rows from
    row 0 and share the scale max|x| / 127 over the group's non-outlier rows; with
    tau > 0 a row whose max|x| exceeds tau times its group's lower median max|x| is an
    outlier and keeps its own scale.  Returns (codes int8 [n, d], scales float32 [n],
    outlier bool [n]).
    """
    x = _f32(x)
    n, d = x.shape
    if group < 1:
        raise ValueError("group must be >= 1")
    codes = np.zeros((n, d), np.int8)
    scales = np.zeros(n, np.float32)
    flags = np.zeros(n, np.uint8)
    if n == 0:
        return codes, scales, flags.astype(bool)
    mu_ptr = None
    if mu is not None:
        mu = _f32(mu).reshape(d)
        mu_ptr = mu.ctypes.data
    _load().oracle_quant_groups(x, n, d, mu_ptr, int(group), float(tau), codes, scales, flags.ctypes.data)
    return codes, scales, flags.astype(bool)


def k_channel_mean(k):
    """Per-channel mean of token rows k [n, d] in the canonical fp32 order (reading R4)."""
    k = _f32(k)
    n, d = k.shape
    mu = np.zeros(d, np.float32)
    _load().oracle_k_mean(k, n, d, d, mu)
    return mu


# ------------------------------------------------------------------ prefill

def _seq_slices(q, k, v, cu_seqlens):
    """Yield (seq index, q [Hq, n, d], k [Hkv, n, d], v [Hkv, n, d]) per sequence."""
    if cu_seqlens is None:
        for b in range(q.shape[0]):
            yield b, q[b], k[b], v[b]
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        for s in range(len(cu) - 1):
            a, e = int(cu[s]), int(cu[s + 1])
            yield s, q[a:e].transpose(1, 0, 2), k[a:e].transpose(1, 0, 2), v[a:e].transpose(1, 0, 2)


def attn_prefill(q, k, v, causal=True, smooth_k=False, cu_seqlens=None, rows=None, want_logits=False,
                 q_group=1, k_group=1, q_outlier_ratio=0.0):
    """W8A8 INT8 attention prefill, fp64 after the int32 dot.

    Dense: q [B,Hq,N,d], k/v [B,Hkv,N,d], or a chunk of Nq <= Nk queries, q [B,Hq,Nq,d]
    against k/v [B,Hkv,Nk,d]: the queries are the last Nq positions of the Nk-token
    sequence, so causal query i sees keys j <= i + Nk - Nq (bottom-right alignment,
    reading R19; the K mean runs over all Nk keys).  Varlen (cu_seqlens int [nseq+1]):
    q [T,Hq,d], k/v [T,Hkv,d] packed.  All inputs float32 (widened from fp16/bf16).
    rows: None for every query row, else an iterable of (seq, hq, i) with i the row
    index within its sequence.
    Returns a dict with
      out [like q] float64 (NaN where a row was not requested), lse [like q[..., 0]],
      q_codes/q_scales, k_codes/k_scales (the quantised Q and smoothed K, full),
      k_mean [nseq, Hkv, d] float32 (zeros when smooth_k is off),
      logits: {(seq, hq, i): int32 [n_allowed]} when want_logits.
    q_group / k_group > 1 or q_outlier_ratio > 0 select the grouped quantisation of
    attn_w8a8_fwd (reading R21, ``quant_groups``) for Q and the smoothed K; the defaults
    are the per-row quantiser.
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    lib = _load()
    varlen = cu_seqlens is not None
    d = q.shape[-1]
    hq_n, hkv_n = (q.shape[1], k.shape[1])
    if hq_n % hkv_n:
        raise ValueError("Hq must be a multiple of Hkv")
    group = hq_n // hkv_n
    nseq = (len(cu_seqlens) - 1) if varlen else q.shape[0]

    q_codes = np.zeros(q.shape, np.int8)
    q_scales = np.zeros(q.shape[:-1], np.float32)
    k_codes = np.zeros(k.shape, np.int8)
    k_scales = np.zeros(k.shape[:-1], np.float32)
    k_mean = np.zeros((nseq, hkv_n, d), np.float32)
    out = np.full(q.shape, np.nan, np.float64)
    lse = np.full(q.shape[:-1], np.nan, np.float64)
    logits = {}

    want = None
    if rows is not None:
        want = {}
        for (s, h, i) in rows:
            want.setdefault((int(s), int(h)), []).append(int(i))

    cu = np.asarray(cu_seqlens, dtype=np.int64) if varlen else None
    if not varlen and q.shape[2] > k.shape[2]:
        raise ValueError("a query chunk cannot be longer than the keys")
    for s, qs, ks, vs in _seq_slices(q, k, v, cu_seqlens):
        nq, n = qs.shape[1], ks.shape[1]
        q_off = n - nq
        # quantise this sequence's K (smoothed per kv head) and Q
        kc_seq = np.zeros((hkv_n, n, d), np.int8)
        ks_seq = np.zeros((hkv_n, n), np.float32)
        for h in range(hkv_n):
            krows = np.ascontiguousarray(ks[h])
            mu = k_channel_mean(krows) if (smooth_k and n > 0) else None
            if mu is not None:
                k_mean[s, h] = mu
            if k_group > 1:
                c, sc, _ = quant_groups(krows, k_group, 0.0, mu)
            else:
                c, sc = quant_rowwise(krows, None if mu is None else mu[None, :], n)
            kc_seq[h], ks_seq[h] = c, sc
        if q_group > 1 or q_outlier_ratio > 0:
            qc_seq = np.zeros(qs.shape, np.int8)
            qsc_seq = np.zeros(qs.shape[:-1], np.float32)
            for h in range(hq_n):
                qc_seq[h], qsc_seq[h], _ = quant_groups(np.ascontiguousarray(qs[h]), q_group, q_outlier_ratio)
        else:
            qc_seq, qsc_seq = quant_rowwise(np.ascontiguousarray(qs))
        if varlen:
            a = int(cu[s])
            k_codes[a:a + n] = kc_seq.transpose(1, 0, 2)
            k_scales[a:a + n] = ks_seq.T
            q_codes[a:a + nq] = qc_seq.transpose(1, 0, 2)
            q_scales[a:a + nq] = qsc_seq.T
        else:
            k_codes[s], k_scales[s], q_codes[s], q_scales[s] = kc_seq, ks_seq, qc_seq, qsc_seq

        for hq in range(hq_n):
            hkv = hq // group  # reading R8
            if want is not None:
                sel = want.get((s, hq))
                if not sel:
                    continue
                sel_arr = np.asarray(sel, np.int64)
                nrows = len(sel_arr)
                rows_ptr = sel_arr.ctypes.data
            else:
                sel_arr = np.arange(nq, dtype=np.int64)
                nrows = nq
                rows_ptr = None
            if nrows == 0:
                continue
            o_rows = np.zeros((nrows, d), np.float64)
            l_rows = np.zeros(nrows, np.float64)
            lg = np.zeros((nrows, n), np.int32) if want_logits else None
            vrows = np.ascontiguousarray(vs[hkv])
            ov = lib.oracle_attn_prefill_head(
                np.ascontiguousarray(qc_seq[hq]), np.ascontiguousarray(qsc_seq[hq]),
                np.ascontiguousarray(kc_seq[hkv]), np.ascontiguousarray(ks_seq[hkv]), vrows,
                nq, n, d, int(bool(causal)), q_off, rows_ptr, nrows, o_rows, l_rows,
                None if lg is None else lg.ctypes.data)
            if ov:
                raise OverflowError("int32 logit overflow")
            if varlen:
                a = int(cu[s])
                out[a + sel_arr, hq] = o_rows
                lse[a + sel_arr, hq] = l_rows
            else:
                out[s, hq, sel_arr] = o_rows
                lse[s, hq, sel_arr] = l_rows
            if want_logits:
                for r, i in enumerate(sel_arr):
                    nn = min(int(i) + 1 + q_off, n) if causal else n
                    logits[(s, hq, int(i))] = lg[r, :nn].copy()
    return dict(out=out, lse=lse, q_codes=q_codes, q_scales=q_scales, k_codes=k_codes,
                k_scales=k_scales, k_mean=k_mean, logits=logits)


# ------------------------------------------------------------------ decode

def attn_decode(q, k_codes, k_scales, v_codes, v_scales, seqlens, num_splits=1, split_size=None,
                rows=None, want_logits=False):
    """Split-KV decode over an int8 cache (readings R12, R13), fp64 after the int32 dot.

    q [B,Hq,d] float32; caches [B,Hkv,Lmax,d] int8 with scales [B,Hkv,Lmax] float32;
    seqlens [B].  The key range [0, Lmax) is cut into num_splits contiguous chunks of
    split_size = ceil(Lmax / num_splits) tokens (or the given split_size); each is a
    partial (normalised O, lse) and the partials are merged by oracle_decode_combine.
    rows: None, or an iterable of (b, hq).  Returns dict(out [B,Hq,d] f64, lse [B,Hq],
    q_codes, q_scales, o_partial [B,Hq,S,d], lse_partial [B,Hq,S], logits {(b,hq): int32 [L]}).
    """
    k_codes = np.ascontiguousarray(k_codes, np.int8)
    v_codes = np.ascontiguousarray(v_codes, np.int8)
    k_scales = _f32(k_scales)
    v_scales = _f32(v_scales)

    def rows_of(b, hkv, L):
        return k_codes[b, hkv], k_scales[b, hkv], v_codes[b, hkv], v_scales[b, hkv]

    return _decode(q, rows_of, k_codes.shape[1], k_codes.shape[2], seqlens, num_splits, split_size, rows,
                   want_logits)


def attn_paged_decode(q, k_pages, k_scale_pages, v_pages, v_scale_pages, block_table, seqlens, num_splits=1,
                      split_size=None, rows=None, want_logits=False):
    """Split-KV decode over a paged int8 (k8v8) cache, fp64 after the int32 dot.

    Source: the "SuperL8" README, "Engine" table ("Paged KV cache" row: int8, k8v3 and
    k8v8 cache formats) and "Attention kernels" table (attn_paged_decode row).  Reading
    (the pages give no layout): a page holds page_size consecutive tokens of one
    sequence for every kv head, k_pages / v_pages [num_pages, Hkv, page_size, d] int8
    codes with per-token scales [num_pages, Hkv, page_size] float32 (k8v8: both K and V
    int8, as in the int8-V decode); block_table [B, max_blocks] int32 names the page of
    the logical block i = tokens [i * page_size, (i + 1) * page_size) of sequence b, so
    token t is row t % page_size of page block_table[b, t // page_size].  The result is
    attn_decode over those rows with Lmax = max_blocks * page_size (same split plan);
    block-table entries past a sequence's last block are never read.
    """
    k_pages = np.ascontiguousarray(k_pages, np.int8)
    v_pages = np.ascontiguousarray(v_pages, np.int8)
    k_scale_pages = _f32(k_scale_pages)
    v_scale_pages = _f32(v_scale_pages)
    block_table = np.asarray(block_table, np.int64)
    page = k_pages.shape[2]
    lmax = block_table.shape[1] * page

    def rows_of(b, hkv, L):
        t = np.arange(L)
        pg, off = block_table[b, t // page], t % page
        return (np.ascontiguousarray(k_pages[pg, hkv, off]), np.ascontiguousarray(k_scale_pages[pg, hkv, off]),
                np.ascontiguousarray(v_pages[pg, hkv, off]), np.ascontiguousarray(v_scale_pages[pg, hkv, off]))

    return _decode(q, rows_of, k_pages.shape[1], lmax, seqlens, num_splits, split_size, rows, want_logits)


def attn_decode_f16v(q, k_codes, k_scales, v, seqlens, num_splits=1, split_size=None, rows=None,
                     want_logits=False):
    """Split-KV decode with an int8 K cache and an fp16 V cache, fp64 after the int32 dot.

    Source: the "SuperL8" README, "Attention kernels" table, attn_decode row (split-KV
    decode with an int8 KV cache; its "fp16 V" variant).  Reading: K is the int8 cache
    of attn_decode (codes [B,Hkv,Lmax,d] with per-token scales [B,Hkv,Lmax]); V is
    [B,Hkv,Lmax,d] fp16 with no scale, O = sum_t p_t v[t] (R12 and R13 otherwise).
    """
    k_codes = np.ascontiguousarray(k_codes, np.int8)
    k_scales = _f32(k_scales)
    v = np.asarray(v)
    if v.dtype != np.float16:
        raise ValueError("v must be float16")
    v = np.ascontiguousarray(v.astype(np.float32))   # exact widening

    def rows_of(b, hkv, L):
        return k_codes[b, hkv], k_scales[b, hkv], v[b, hkv], None

    return _decode(q, rows_of, k_codes.shape[1], k_codes.shape[2], seqlens, num_splits, split_size, rows,
                   want_logits)


def attn_decode_verify(q, k_codes, k_scales, v_codes, v_scales, seqlens, tree_mask, rows=None):
    """Speculative-decode verification over an int8 cache, fp64 after the int32 dot.

    Source: the "SuperL8" README, "Attention kernels" table, attn_decode row (its
    "verify mask" variant) and attn_tree_fwd row (tree-structured verification), with
    the "Speculative decoding" table's drafters building chain or tree masks.  Reading
    (R20): q [B, T, Hq, d] holds T draft queries per sequence; the cache (as attn_decode)
    already holds the T draft tokens at positions L_b - T .. L_b - 1; query t sees every
    position below L_b - T and draft token u (position L_b - T + u, when >= 0) iff bit u
    of tree_mask[b, t] is set (uint32, T <= 32).  Each (b, t, hq) row is the attention of
    its quantised query over exactly those positions.  Returns dict(out [B,T,Hq,d] f64,
    lse [B,T,Hq], q_codes [B,T,Hq,d], q_scales [B,T,Hq]).
    """
    q = _f32(q)
    k_codes = np.ascontiguousarray(k_codes, np.int8)
    v_codes = np.ascontiguousarray(v_codes, np.int8)
    k_scales = _f32(k_scales)
    v_scales = _f32(v_scales)
    seqlens = np.asarray(seqlens, np.int64)
    tree_mask = np.asarray(tree_mask, np.uint64)
    B, T, hq_n, d = q.shape
    hkv_n = k_codes.shape[1]
    group = hq_n // hkv_n
    lib = _load()
    q_codes, q_scales = quant_rowwise(q)
    out = np.full((B, T, hq_n, d), np.nan, np.float64)
    lse = np.full((B, T, hq_n), np.nan, np.float64)
    triples = ([(b, t, h) for b in range(B) for t in range(T) for h in range(hq_n)] if rows is None
               else [(int(b), int(t), int(h)) for b, t, h in rows])
    for b, t, hq in triples:
        hkv = hq // group
        L = int(seqlens[b])
        tail = L - T
        pos = list(range(max(tail, 0)))
        pos += [tail + u for u in range(T) if tail + u >= 0 and (int(tree_mask[b, t]) >> u) & 1]
        pos = np.asarray(pos, np.int64)
        n = len(pos)
        kc = np.ascontiguousarray(k_codes[b, hkv][pos])
        ksc = np.ascontiguousarray(k_scales[b, hkv][pos])
        vc = np.ascontiguousarray(v_codes[b, hkv][pos])
        vsc = np.ascontiguousarray(v_scales[b, hkv][pos])
        o = np.zeros(d, np.float64)
        lv = np.zeros(1, np.float64)
        lib.oracle_decode_row(q_codes[b, t, hq], float(q_scales[b, t, hq]), kc, ksc, vc, vsc, n, 0, n, d, o, lv,
                              None)
        out[b, t, hq], lse[b, t, hq] = o, lv[0]
    return dict(out=out, lse=lse, q_codes=q_codes, q_scales=q_scales)


def attn_chunk_cache(q, k_codes, k_scales, v_codes, v_scales, nk, causal=True, rows=None):
    """A query chunk against an int8 cache that holds its keys, fp64 after the int32 dot.

    Source: the "SuperL8-serve" README, "Engine" table (chunked prefill onto the KV
    cache), with the cache of the "Attention kernels" table's attn_decode row (int8 codes,
    per-token scales).  Reading (R22): q [B, Hq, Nq, d] holds the queries of positions
    nk - Nq .. nk - 1; the caches [B, Hkv, Lmax, d] hold positions 0 .. nk - 1 of every
    sequence.  Row (b, hq, i) is the decode of its quantised query over cache positions
    0 .. nk - Nq + i (causal) or 0 .. nk - 1.  Returns dict(out [B,Hq,Nq,d] f64,
    lse [B,Hq,Nq], q_codes, q_scales).
    """
    q = _f32(q)
    k_codes = np.ascontiguousarray(k_codes, np.int8)
    v_codes = np.ascontiguousarray(v_codes, np.int8)
    k_scales = _f32(k_scales)
    v_scales = _f32(v_scales)
    B, hq_n, nq, d = q.shape
    group = hq_n // k_codes.shape[1]
    lib = _load()
    q_codes, q_scales = quant_rowwise(q)
    out = np.full((B, hq_n, nq, d), np.nan, np.float64)
    lse = np.full((B, hq_n, nq), np.nan, np.float64)
    triples = ([(b, h, i) for b in range(B) for h in range(hq_n) for i in range(nq)] if rows is None
               else [(int(b), int(h), int(i)) for b, h, i in rows])
    for b, hq, i in triples:
        hkv = hq // group
        L = nk - nq + i + 1 if causal else nk
        o = np.zeros(d, np.float64)
        lv = np.zeros(1, np.float64)
        lib.oracle_decode_row(q_codes[b, hq, i], float(q_scales[b, hq, i]), k_codes[b, hkv], k_scales[b, hkv],
                              v_codes[b, hkv], v_scales[b, hkv], L, 0, L, d, o, lv, None)
        out[b, hq, i], lse[b, hq, i] = o, lv[0]
    return dict(out=out, lse=lse, q_codes=q_codes, q_scales=q_scales)


def _decode(q, rows_of, hkv_n, lmax, seqlens, num_splits, split_size, rows, want_logits):
    """The split loop shared by the decode oracles; rows_of(b, hkv, L) gives the kv head's
    cache rows (k codes, k scales, v codes, v scales) for tokens 0 .. L-1 (at least); v
    scales None means V rows of fp16 values widened to fp32, without scales."""
    q = _f32(q)
    seqlens = np.asarray(seqlens, np.int64)
    B, hq_n, d = q.shape
    group = hq_n // hkv_n
    if split_size is None:
        split_size = max(1, -(-lmax // max(1, num_splits)))
    nsplit = max(1, -(-lmax // split_size))
    lib = _load()
    q_codes, q_scales = quant_rowwise(q)
    out = np.full((B, hq_n, d), np.nan, np.float64)
    lse = np.full((B, hq_n), np.nan, np.float64)
    o_part = np.full((B, hq_n, nsplit, d), np.nan, np.float64)
    l_part = np.full((B, hq_n, nsplit), np.nan, np.float64)
    logits = {}
    pairs = [(b, h) for b in range(B) for h in range(hq_n)] if rows is None else [(int(b), int(h)) for b, h in rows]
    cached = {}
    for b, hq in pairs:
        hkv = hq // group
        L = int(seqlens[b])
        if (b, hkv) not in cached:
            cached.clear()
            cached[(b, hkv)] = rows_of(b, hkv, L)
        kc, ksc, vc, vsc = cached[(b, hkv)]

        def row(t0, t1, o, lv, lg):
            if vsc is None:
                lib.oracle_decode_row_fv(q_codes[b, hq], float(q_scales[b, hq]), kc, ksc, vc, L, t0, t1, d, o, lv, lg)
            else:
                lib.oracle_decode_row(q_codes[b, hq], float(q_scales[b, hq]), kc, ksc, vc, vsc, L, t0, t1, d, o, lv,
                                      lg)

        for s in range(nsplit):
            o = np.zeros(d, np.float64)
            lv = np.zeros(1, np.float64)
            row(s * split_size, (s + 1) * split_size, o, lv, None)
            o_part[b, hq, s], l_part[b, hq, s] = o, lv[0]
        o = np.zeros(d, np.float64)
        lv = np.zeros(1, np.float64)
        lib.oracle_decode_combine(np.ascontiguousarray(o_part[b, hq]), np.ascontiguousarray(l_part[b, hq]),
                                  nsplit, d, o, lv)
        out[b, hq], lse[b, hq] = o, lv[0]
        if want_logits:
            lg = np.zeros(max(L, 1), np.int32)
            o2 = np.zeros(d, np.float64)
            l2 = np.zeros(1, np.float64)
            row(0, L, o2, l2, lg.ctypes.data)
            logits[(b, hq)] = lg[:L].copy()
    return dict(out=out, lse=lse, q_codes=q_codes, q_scales=q_scales, o_partial=o_part,
                lse_partial=l_part, logits=logits)


def decode_combine(o_partial, lse_partial):
    """Merge split partials o [..., S, d] / lse [..., S] (reading R13), fp64."""
    o_partial = np.ascontiguousarray(o_partial, np.float64)
    lse_partial = np.ascontiguousarray(lse_partial, np.float64)
    lead = o_partial.shape[:-2]
    S, d = o_partial.shape[-2:]
    flat_o = o_partial.reshape(-1, S, d)
    flat_l = lse_partial.reshape(-1, S)
    out = np.zeros((flat_o.shape[0], d), np.float64)
    lse = np.zeros(flat_o.shape[0], np.float64)
    lib = _load()
    for r in range(flat_o.shape[0]):
        o = np.zeros(d, np.float64)
        lv = np.zeros(1, np.float64)
        lib.oracle_decode_combine(np.ascontiguousarray(flat_o[r]), np.ascontiguousarray(flat_l[r]), S, d, o, lv)
        out[r], lse[r] = o, lv[0]
    return out.reshape(*lead, d), lse.reshape(lead)
