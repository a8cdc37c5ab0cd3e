"""Seeded synthetic inputs for the five attention workloads.

This module only draws random numbers and casts them to the input dtypes; it
holds none of the attention or quantisation arithmetic.  Both the CPU oracle
(``oracle/``) and the CUDA library's tests and benchmark take their inputs from
here, so both sides see identical bytes.

Every tensor is drawn per slice from its own PCG64 stream, keyed by
``(0x5EED0000 + workload id, tensor tag, slice indices...)``, so a single head
or sequence can be regenerated without drawing the rest.  Normals are numpy
``standard_normal`` in float32, cast to fp16/bf16 by torch (round to nearest
even).  Shapes and distributions follow the workload list:

  1 tiny       B1 Hq4 Hkv2 N256 d64, fp16 N(0,1); in each kv head one K channel
               (max(1, round(1% of d))) is scaled x20 before the cast.
  2 qwen3_8b   B1 Hq32 Hkv8 N4096 d128, bf16 N(0,1); K gets a per-(kv head, channel)
               bias drawn N(0, std 2), the same for every token.
  3 decode     B64, one query token, Hq32 Hkv8 d128; context lengths uniform on
               the integers [1024, 8192]; cache values fp32 N(0,1) (quantised per
               token row by whoever consumes them); q bf16 N(0,1).
  4 gemma3_d256  B2 Hq16 Hkv8 N8192 d256, bf16 N(0,1).
  5 varlen     32 sequences, lengths uniform on the integers [17, 3000], packed
               [T, H, d] with cu_seqlens, Hq64 Hkv8 d128, bf16 N(0,1).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np
import torch

SEED_BASE = 0x5EED0000

# tensor tags (stream keys)
TAG_Q, TAG_K, TAG_V, TAG_KBIAS, TAG_OUTLIER, TAG_LENS, TAG_PAGES = 1, 2, 3, 4, 5, 6, 7


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    kind: str  # "prefill" | "varlen" | "decode"
    B: int
    Hq: int
    Hkv: int
    d: int
    N: int = 0            # prefill sequence length (dense)
    dtype: str = "bf16"   # Q/K/V dtype (prefill) or q dtype (decode)
    causal: bool = True
    smooth_k: bool = True
    k_outlier_frac: float = 0.0
    k_bias_std: float = 0.0
    len_lo: int = 0       # varlen / decode lengths, inclusive range
    len_hi: int = 0
    lmax: int = 0         # decode cache capacity
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny": Workload(1, "tiny", "prefill", B=1, Hq=4, Hkv=2, d=64, N=256, dtype="f16",
                     k_outlier_frac=0.01, smooth_k=True),
    "qwen3_8b": Workload(2, "qwen3_8b", "prefill", B=1, Hq=32, Hkv=8, d=128, N=4096, dtype="bf16",
                         k_bias_std=2.0, smooth_k=True),
    "decode": Workload(3, "decode", "decode", B=64, Hq=32, Hkv=8, d=128, dtype="bf16",
                       len_lo=1024, len_hi=8192, lmax=8192, smooth_k=False),
    "gemma3_d256": Workload(4, "gemma3_d256", "prefill", B=2, Hq=16, Hkv=8, d=256, N=8192, dtype="bf16",
                            smooth_k=True),
    "varlen": Workload(5, "varlen", "varlen", B=32, Hq=64, Hkv=8, d=128, dtype="bf16",
                       len_lo=17, len_hi=3000, smooth_k=True),
}


def get(name: str, **overrides) -> Workload:
    """A named workload, optionally with fields replaced (smaller test sizes)."""
    return replace(WORKLOADS[name], **overrides)


def _rng(w: Workload, tag: int, *idx: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([SEED_BASE + w.wid, tag, *idx])))


def torch_dtype(name: str) -> torch.dtype:
    return {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[name]


def _cast(x: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(x).to(torch_dtype(dtype))


def _outlier_channels(w: Workload, hkv: int) -> np.ndarray:
    if w.k_outlier_frac <= 0:
        return np.zeros(0, np.int64)
    n = max(1, int(round(w.k_outlier_frac * w.d)))
    return np.sort(_rng(w, TAG_OUTLIER, hkv).choice(w.d, size=n, replace=False))


def _k_bias(w: Workload) -> np.ndarray | None:
    if w.k_bias_std <= 0:
        return None
    return (_rng(w, TAG_KBIAS).standard_normal((w.Hkv, w.d), dtype=np.float32) * np.float32(w.k_bias_std))


def _k_rows(w: Workload, rows: np.ndarray, hkv: int, bias: np.ndarray | None) -> np.ndarray:
    """Apply the K bias / outlier scaling (fp32, before the cast) to one kv head's rows."""
    if bias is not None:
        rows = rows + bias[hkv][None, :]
    ch = _outlier_channels(w, hkv)
    if len(ch):
        rows = rows.copy()
        rows[:, ch] *= np.float32(20.0)
    return rows


def prefill_dense(w: Workload):
    """q [B,Hq,N,d], k/v [B,Hkv,N,d] as torch CPU tensors of the workload dtype."""
    B, N, d = w.B, w.N, w.d
    q = np.empty((B, w.Hq, N, d), np.float32)
    k = np.empty((B, w.Hkv, N, d), np.float32)
    v = np.empty((B, w.Hkv, N, d), np.float32)
    bias = _k_bias(w)
    for b in range(B):
        for h in range(w.Hq):
            q[b, h] = _rng(w, TAG_Q, b, h).standard_normal((N, d), dtype=np.float32)
        for h in range(w.Hkv):
            k[b, h] = _k_rows(w, _rng(w, TAG_K, b, h).standard_normal((N, d), dtype=np.float32), h, bias)
            v[b, h] = _rng(w, TAG_V, b, h).standard_normal((N, d), dtype=np.float32)
    return _cast(q, w.dtype), _cast(k, w.dtype), _cast(v, w.dtype)


def seq_lengths(w: Workload) -> np.ndarray:
    """Sequence lengths (varlen) or context lengths (decode), uniform on [len_lo, len_hi]."""
    if "lengths" in w.extra:
        return np.asarray(w.extra["lengths"], np.int64)
    return _rng(w, TAG_LENS).integers(w.len_lo, w.len_hi, size=w.B, endpoint=True).astype(np.int64)


def prefill_varlen(w: Workload):
    """Packed q [T,Hq,d], k/v [T,Hkv,d] (torch CPU) and cu_seqlens int32 [nseq+1]."""
    lens = seq_lengths(w)
    cu = np.zeros(len(lens) + 1, np.int64)
    cu[1:] = np.cumsum(lens)
    T, d = int(cu[-1]), w.d
    q = np.empty((T, w.Hq, d), np.float32)
    k = np.empty((T, w.Hkv, d), np.float32)
    v = np.empty((T, w.Hkv, d), np.float32)
    bias = _k_bias(w)
    for s, L in enumerate(lens):
        a, e = int(cu[s]), int(cu[s + 1])
        q[a:e] = _rng(w, TAG_Q, s).standard_normal((int(L), w.Hq, d), dtype=np.float32)
        kk = _rng(w, TAG_K, s).standard_normal((int(L), w.Hkv, d), dtype=np.float32)
        for h in range(w.Hkv):
            kk[:, h] = _k_rows(w, kk[:, h], h, bias)
        k[a:e] = kk
        v[a:e] = _rng(w, TAG_V, s).standard_normal((int(L), w.Hkv, d), dtype=np.float32)
    return (_cast(q, w.dtype), _cast(k, w.dtype), _cast(v, w.dtype), torch.from_numpy(cu.astype(np.int32)))


def decode_query(w: Workload) -> torch.Tensor:
    """q [B, Hq, d] of the workload dtype (one query token per sequence)."""
    q = np.empty((w.B, w.Hq, w.d), np.float32)
    for b in range(w.B):
        q[b] = _rng(w, TAG_Q, b).standard_normal((w.Hq, w.d), dtype=np.float32)
    return _cast(q, w.dtype)


def chunk_query(w: Workload, nq: int) -> torch.Tensor:
    """q [B, Hq, nq, d] of the workload dtype: the queries of a chunk of nq positions per
    sequence (prefill onto a cache), N(0,1)."""
    q = np.empty((w.B, w.Hq, nq, w.d), np.float32)
    for b in range(w.B):
        q[b] = _rng(w, TAG_Q, b, nq).standard_normal((w.Hq, nq, w.d), dtype=np.float32)
    return _cast(q, w.dtype)


def decode_cache_values(w: Workload, b: int, which: str) -> np.ndarray:
    """fp32 cache values [Hkv, L_b, d] for sequence b (which = "k" or "v"), N(0,1).

    Rows at t >= L_b are never drawn: a cache holds nothing there."""
    L = int(seq_lengths(w)[b])
    tag = TAG_K if which == "k" else TAG_V
    return _rng(w, tag, b).standard_normal((w.Hkv, L, w.d), dtype=np.float32)


def page_table(w: Workload, lens, page_size: int, max_blocks: int | None = None, spare: int = 0,
               shared_prefix: int = 0):
    """A block table for a paged cache of the decode workload w.

    Sequence b needs ceil(L_b / page_size) logical blocks.  The pages are a seeded
    random permutation of 0 .. num_pages-1, where num_pages counts every block in use
    plus `spare` pages nobody uses; entries past a sequence's last block are -1.  With
    shared_prefix = n > 0, every sequence's first n blocks point at the pages of
    sequence 0 (a shared prompt prefix).  Returns (block_table [B, max_blocks] int32,
    num_pages)."""
    lens = np.asarray(lens, np.int64)
    need = (lens + page_size - 1) // page_size
    if max_blocks is None:
        max_blocks = int(max(1, need.max() if len(need) else 1))
    own = [int(n) if b == 0 else max(0, int(n) - min(shared_prefix, int(need[0]), int(n)))
           for b, n in enumerate(need)]
    num_pages = int(sum(own)) + spare
    perm = _rng(w, TAG_PAGES, page_size).permutation(max(num_pages, 1))
    table = np.full((len(lens), max_blocks), -1, np.int32)
    nxt = 0
    for b, n in enumerate(need):
        n = int(n)
        share = 0 if b == 0 else min(shared_prefix, int(need[0]), n)
        table[b, :share] = table[0, :share]
        table[b, share:n] = perm[nxt:nxt + n - share]
        nxt += n - share
    return table, max(num_pages, 1)


def paginate(cache, scales, block_table, lens, page_size: int, num_pages: int):
    """Copy a contiguous cache [B, Hkv, Lmax, d] (+ scales [B, Hkv, Lmax]) into pages
    [num_pages, Hkv, page_size, d] (+ [num_pages, Hkv, page_size]) following block_table:
    logical block i of sequence b (tokens [i * page_size, (i + 1) * page_size)) becomes
    page block_table[b, i], for the blocks that hold tokens t < L_b.  Works on numpy
    arrays or torch tensors (of any device); pages no block uses stay zero.  A page shared
    by several sequences receives each one's block (callers share pages only between
    identical prefixes)."""
    is_torch = isinstance(cache, torch.Tensor)
    B, H, lmax, d = cache.shape
    nb = block_table.shape[1]
    lens = np.asarray(lens, np.int64)
    need = (lens + page_size - 1) // page_size
    table = np.asarray(block_table.cpu() if isinstance(block_table, torch.Tensor) else block_table, np.int64)
    sel_b, sel_i = np.nonzero(np.arange(nb)[None, :] < need[:, None])
    dst = table[sel_b, sel_i]
    if is_torch:
        pad = nb * page_size - lmax
        c = torch.nn.functional.pad(cache, (0, 0, 0, max(pad, 0)))[:, :, :nb * page_size]
        sc = torch.nn.functional.pad(scales, (0, max(pad, 0)))[:, :, :nb * page_size]
        blocks = c.reshape(B, H, nb, page_size, d).permute(0, 2, 1, 3, 4)
        sblocks = sc.reshape(B, H, nb, page_size).permute(0, 2, 1, 3)
        pages = torch.zeros((num_pages, H, page_size, d), dtype=cache.dtype, device=cache.device)
        spages = torch.zeros((num_pages, H, page_size), dtype=scales.dtype, device=scales.device)
        ib = torch.from_numpy(sel_b).to(cache.device)
        ii = torch.from_numpy(sel_i).to(cache.device)
        it = torch.from_numpy(dst).to(cache.device)
        pages[it] = blocks[ib, ii]
        spages[it] = sblocks[ib, ii]
    else:
        pad = max(nb * page_size - lmax, 0)
        c = np.pad(cache, ((0, 0), (0, 0), (0, pad), (0, 0)))[:, :, :nb * page_size]
        sc = np.pad(scales, ((0, 0), (0, 0), (0, pad)))[:, :, :nb * page_size]
        blocks = c.reshape(B, H, nb, page_size, d).transpose(0, 2, 1, 3, 4)
        sblocks = sc.reshape(B, H, nb, page_size).transpose(0, 2, 1, 3)
        pages = np.zeros((num_pages, H, page_size, d), cache.dtype)
        spages = np.zeros((num_pages, H, page_size), scales.dtype)
        pages[dst] = blocks[sel_b, sel_i]
        spages[dst] = sblocks[sel_b, sel_i]
    return pages, spages


def custom(wid: int, kind: str = "prefill", **fields) -> Workload:
    """A workload of any shape with its own seed id (test cases beyond the five above)."""
    base = dict(name=f"custom{wid}", kind=kind, B=1, Hq=1, Hkv=1, d=128)
    base.update(fields)
    return Workload(wid=wid, **base)
