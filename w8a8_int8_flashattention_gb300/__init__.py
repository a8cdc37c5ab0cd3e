"""sl8 -- W8A8 INT8 attention for NVIDIA GB300 (sm_103a).

A thin Python binding over the C ABI of ``libsl8.so`` (declared in
``include/sl8.h``).  This module only marshals arguments: it takes torch CUDA
tensors, allocates outputs and workspaces with torch, and calls the library on
torch's current stream.  Every step of the computation runs in the library's
CUDA kernels; there is no CPU or PyTorch fallback, and a missing library is an
error.

Operations (the "SuperL8" README, github.com/jajmangold/superl8): symmetric
per-row int8 quantisation ("Supporting kernels" table, quant_rowwise; "Quantization"
table, per-row int8 with K-smoothing), W8A8 INT8 FlashAttention prefill, dense and
varlen ("Attention kernels" table, attn_int8_fwd / attn_varlen_fwd; "Quick start"
layouts) and split-KV decode over an int8 KV cache ("Attention kernels" table,
attn_decode, int8-V variant).
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsl8.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "sl8.h")

SL8_F16, SL8_BF16, SL8_F32, SL8_I8 = 0, 1, 2, 3
SL8_OK, SL8_ERR_INVALID_ARG, SL8_ERR_UNSUPPORTED, SL8_ERR_WORKSPACE, SL8_ERR_CUDA, SL8_ERR_TIMEOUT, \
    SL8_ERR_DEVICE_ARG = range(7)

_DTYPES = {torch.float16: SL8_F16, torch.bfloat16: SL8_BF16, torch.float32: SL8_F32, torch.int8: SL8_I8}
_TORCH_DTYPES = {v: k for k, v in _DTYPES.items()}


class SL8Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {status_string(status)} (status {status})"
        if status == SL8_ERR_CUDA:
            try:
                msg += ": " + lib().sl8_last_cuda_error_string().decode()
            except Exception:  # noqa: BLE001 - used while formatting another error
                pass
        super().__init__(msg)


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_SZ = ctypes.c_size_t
_U64 = ctypes.c_uint64

_SIGNATURES = {
    "sl8_status_string": (ctypes.c_char_p, [_INT]),
    "sl8_last_cuda_error_string": (ctypes.c_char_p, []),
    "sl8_version": (_INT, []),
    "sl8_quant_rowwise": (_INT, [_P, _INT, _I64, _I32, _I64, _P, _I64, _P, _P, _P]),
    "sl8_k_channel_mean_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "sl8_k_channel_mean": (_INT, [_P, _INT, _I32, _I32, _I32, _I32, _P, _I64, _P, _P, _SZ, _P]),
    "sl8_attn_int8_fwd_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I64]),
    "sl8_attn_int8_fwd": (_INT, [_P, _P, _P, _INT, _INT, _I32, _I32, _I32, _I32, _I32, _P, _I64, _INT, _INT, _P,
                                 _INT, _P, _P, _SZ, _P]),
    "sl8_attn_int8_fwd_chunk_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32]),
    "sl8_attn_int8_fwd_chunk": (_INT, [_P, _P, _P, _INT, _INT, _I32, _I32, _I32, _I32, _I32, _I32, _INT, _INT, _P,
                                       _INT, _P, _P, _SZ, _P]),
    "sl8_attn_int8_fwd_chunk_cache": (_INT, [_P, _INT, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _INT,
                                             _P, _INT, _P, _P, _SZ, _P]),
    "sl8_attn_int8_qk_logits_debug": (_INT, [_P, _P, _INT, _I32, _I32, _I32, _I32, _I32, _P, _I64, _INT, _I32, _I32,
                                             _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "sl8_attn_w8a8_fwd": (_INT, [_P, _P, _P, _INT, _INT, _I32, _I32, _I32, _I32, _I32, _P, _I64, _INT, _INT, _I32,
                                 _I32, ctypes.c_float, _P, _INT, _P, _P, _SZ, _P]),
    "sl8_attn_w8a8_qk_logits_debug": (_INT, [_P, _P, _INT, _I32, _I32, _I32, _I32, _I32, _P, _I64, _INT, _I32,
                                             _I32, ctypes.c_float, _I32, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "sl8_attn_decode_num_splits": (_I32, [_I32, _I32, _I32, _I32, _I32]),
    "sl8_attn_decode_split_size": (_I32, [_I32, _I32, _I32, _I32, _I32]),
    "sl8_attn_decode_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32]),
    "sl8_attn_decode_lse_offset": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32]),
    "sl8_attn_int8_decode_splitkv": (_INT, [_P, _INT, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P,
                                            _P, _P]),
    "sl8_attn_decode_verify_num_splits": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _I32]),
    "sl8_attn_int8_decode_verify": (_INT, [_P, _INT, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                                           _I32, _P, _P, _P, _INT, _P, _P]),
    "sl8_attn_int8_decode_splitkv_f16v": (_INT, [_P, _INT, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P,
                                                 _P, _P]),
    "sl8_attn_int8_paged_decode_splitkv": (_INT, [_P, _INT, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _I32, _I32,
                                                  _I32, _I32, _I32, _P, _P, _P]),
    "sl8_attn_decode_combine": (_INT, [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _INT, _P, _P]),
    "sl8_attn_int8_decode_logits_debug": (_INT, [_P, _INT, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P,
                                                 _P, _P, _P, _P]),
    "sl8_attn_int8_decode_noalloc": (_INT, [_P, _INT, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _INT,
                                            _P]),
    "sl8_last_device_status": (_INT, [_P, ctypes.POINTER(_INT)]),
    "sl8_set_spin_limit_ns": (None, [_U64]),
    "sl8_get_spin_limit_ns": (_U64, []),
    "sl8_selftest_timeout": (_INT, [_U64, _P]),
    "sl8_trace_enable": (None, [_INT]),
    "sl8_trace_collect": (_INT, [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(_I64),
                                 ctypes.POINTER(ctypes.c_double), _INT]),
}


def lib() -> ctypes.CDLL:
    """The loaded libsl8 (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libsl8.so not found at {LIB_PATH}: build it first "
                                   "(python -c 'import __graft_entry__ as g; g.build()'); there is no fallback")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                f = getattr(l, name)
                f.restype = res
                f.argtypes = args
            _lib = l
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/sl8.h declares."""
    src = open(HEADER_PATH).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sl8_[a-z0-9_]+)\s*\(", src)))


def status_string(status: int) -> str:
    try:
        return lib().sl8_status_string(status).decode()
    except Exception:  # noqa: BLE001 - used while formatting another error
        return f"status {status}"


def _check(status: int, what: str) -> None:
    if status != SL8_OK:
        raise SL8Error(status, what)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _dt(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _DTYPES[t.dtype]


def _need_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("sl8 takes CUDA tensors only (no CPU fallback)")
            if not t.is_contiguous():
                raise ValueError("sl8 takes contiguous tensors")


# ------------------------------------------------------------------ quantisation

def quant_rowwise(x: torch.Tensor, sub_mean: torch.Tensor | None = None, rows_per_group: int | None = None):
    """Symmetric per-row int8 quantisation of the last axis of x (f16/bf16/f32).

    Returns (codes int8 like x, scales fp32 x.shape[:-1]).  sub_mean [groups, cols]
    fp32 is subtracted from row r (flattened) with group r // rows_per_group."""
    _need_cuda(x, sub_mean)
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    codes = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    scales = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    rpg = 0
    if sub_mean is not None:
        rpg = rows_per_group or rows
    _check(lib().sl8_quant_rowwise(_ptr(x), _dt(x), rows, cols, cols, _ptr(sub_mean), rpg, _ptr(codes),
                                   _ptr(scales), _stream(x.device)), "sl8_quant_rowwise")
    return codes, scales


def k_channel_mean(k: torch.Tensor, cu_seqlens: torch.Tensor | None = None, max_seqlen: int | None = None):
    """Per-(sequence, kv head, channel) mean of K.  Dense k [B,Hkv,N,d] or packed
    k [T,Hkv,d] with cu_seqlens.  Returns fp32 [B, Hkv, d]."""
    _need_cuda(k, cu_seqlens)
    if cu_seqlens is None:
        B, Hkv, N, d = k.shape
        T = 0
    else:
        T, Hkv, d = k.shape
        B = cu_seqlens.numel() - 1
        N = int(max_seqlen) if max_seqlen is not None else T
    mean = torch.empty((B, Hkv, d), dtype=torch.float32, device=k.device)
    ws_bytes = lib().sl8_k_channel_mean_workspace_size(B, Hkv, N, d)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=k.device)
    _check(lib().sl8_k_channel_mean(_ptr(k), _dt(k), B, Hkv, N, d, _ptr(cu_seqlens), T, _ptr(mean), _ptr(ws),
                                    ws.numel(), _stream(k.device)), "sl8_k_channel_mean")
    return mean


# ------------------------------------------------------------------ prefill

def prefill_workspace_bytes(B, Hq, Hkv, N, d, total_tokens=0) -> int:
    return int(lib().sl8_attn_int8_fwd_workspace_size(B, Hq, Hkv, N, d, total_tokens))


def attn_int8_fwd(q, k, v, causal=True, smooth_k=True, cu_seqlens=None, max_seqlen=None, out_dtype=None,
                  return_lse=False, workspace=None, out=None, lse=None):
    """W8A8 INT8 attention prefill.

    Dense: q [B,Hq,N,d], k/v [B,Hkv,N,d].  Varlen: q [T,Hq,d], k/v [T,Hkv,d] with
    cu_seqlens int32 [B+1] (CUDA) and max_seqlen (host int >= every length).
    Returns out (q's layout, dtype v.dtype or out_dtype=float32) and, with
    return_lse, the fp32 log-sum-exp per query row."""
    return _prefill("sl8_attn_int8_fwd", (), q, k, v, causal, smooth_k, cu_seqlens, max_seqlen, out_dtype,
                    return_lse, workspace, out, lse)


def attn_w8a8_fwd(q, k, v, causal=True, smooth_k=True, q_group=32, k_group=32, q_outlier_ratio=4.0,
                  cu_seqlens=None, max_seqlen=None, out_dtype=None, return_lse=False, workspace=None, out=None,
                  lse=None):
    """W8A8 prefill with grouped scales: rows of a (sequence, head) share one scale per
    group of q_group (Q) / k_group (K) consecutive positions; a Q row above
    q_outlier_ratio times its group's lower median row maximum keeps its own scale
    (0 turns that off).  Groups are powers of two up to 64; q_group = k_group = 1 is
    attn_int8_fwd.  Layouts and the rest as attn_int8_fwd."""
    return _prefill("sl8_attn_w8a8_fwd", (int(q_group), int(k_group), float(q_outlier_ratio)), q, k, v, causal,
                    smooth_k, cu_seqlens, max_seqlen, out_dtype, return_lse, workspace, out, lse)


def _prefill(fn, extra, q, k, v, causal, smooth_k, cu_seqlens, max_seqlen, out_dtype, return_lse, workspace, out,
             lse):
    _need_cuda(q, k, v, cu_seqlens, workspace)
    if cu_seqlens is None:
        B, Hq, N, d = q.shape
        Hkv = k.shape[1]
        T = 0
    else:
        T, Hq, d = q.shape
        Hkv = k.shape[1]
        B = cu_seqlens.numel() - 1
        if max_seqlen is None:
            raise ValueError("varlen prefill needs max_seqlen")
        N = int(max_seqlen)
        if cu_seqlens.dtype != torch.int32:
            raise TypeError("cu_seqlens must be int32")
    out_dtype = out_dtype or v.dtype
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if return_lse and lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    ws_bytes = prefill_workspace_bytes(B, Hq, Hkv, N, d, T)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    _check(getattr(lib(), fn)(_ptr(q), _ptr(k), _ptr(v), _dt(q), _dt(v), B, Hq, Hkv, N, d, _ptr(cu_seqlens), T,
                              int(bool(causal)), int(bool(smooth_k)), *extra, _ptr(out), _dt(out),
                              _ptr(lse) if return_lse else None, _ptr(workspace), workspace.numel(),
                              _stream(q.device)), fn)
    return (out, lse) if return_lse else out


def attn_int8_fwd_chunk(q, k, v, causal=True, smooth_k=True, out_dtype=None, return_lse=False, workspace=None,
                        out=None, lse=None):
    """Prefill of a query chunk: q [B,Hq,Nq,d] holds the last Nq positions of sequences
    whose keys/values k, v [B,Hkv,Nk,d] cover all Nk >= Nq positions (bottom-right causal
    alignment).  Returns out [B,Hq,Nq,d] (and the fp32 LSE with return_lse)."""
    _need_cuda(q, k, v, workspace)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    out_dtype = out_dtype or v.dtype
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if return_lse and lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    if workspace is None:
        # room for the key-split partials, which the library uses when the chunk is small
        ws_bytes = int(lib().sl8_attn_int8_fwd_chunk_workspace_size(B, Hq, Hkv, Nq, Nk, d))
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    _check(lib().sl8_attn_int8_fwd_chunk(_ptr(q), _ptr(k), _ptr(v), _dt(q), _dt(v), B, Hq, Hkv, Nq, Nk, d,
                                         int(bool(causal)), int(bool(smooth_k)), _ptr(out), _dt(out),
                                         _ptr(lse) if return_lse else None, _ptr(workspace), workspace.numel(),
                                         _stream(q.device)), "sl8_attn_int8_fwd_chunk")
    return (out, lse) if return_lse else out


def attn_int8_fwd_chunk_cache(q, k_cache, k_scale, v_cache, v_scale, Nk=None, causal=True, out_dtype=None,
                              return_lse=False, workspace=None, out=None, lse=None):
    """Prefill of a query chunk onto an int8 KV cache: q [B,Hq,Nq,d] (fp16/bf16) holds
    positions Nk-Nq .. Nk-1; the caches k_cache, v_cache [B,Hkv,Lmax,d] int8 with scales
    [B,Hkv,Lmax] fp32 hold Nk (default Lmax) positions of every sequence.  Returns out
    [B,Hq,Nq,d] (and the fp32 LSE with return_lse)."""
    _need_cuda(q, k_cache, k_scale, v_cache, v_scale, workspace)
    B, Hq, Nq, d = q.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    Nk = Lmax if Nk is None else int(Nk)
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if return_lse and lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    if workspace is None:
        ws_bytes = int(lib().sl8_attn_int8_fwd_chunk_workspace_size(B, Hq, Hkv, Nq, Nk, d))
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    _check(lib().sl8_attn_int8_fwd_chunk_cache(_ptr(q), _dt(q), _ptr(k_cache), _ptr(k_scale), _ptr(v_cache),
                                               _ptr(v_scale), B, Hq, Hkv, Nq, Nk, Lmax, d, int(bool(causal)),
                                               _ptr(out), _dt(out), _ptr(lse) if return_lse else None,
                                               _ptr(workspace), workspace.numel(), _stream(q.device)),
           "sl8_attn_int8_fwd_chunk_cache")
    return (out, lse) if return_lse else out


def attn_int8_qk_logits_debug(q, k, smooth_k=True, row_begin=0, row_end=None, want_codes=True, groups=None,
                              cu_seqlens=None, max_seqlen=None, want_logits=True, workspace=None):
    """Exact int32 logits of the prefill tensor-core path for query rows
    [row_begin, row_end) of every sequence against every key of that sequence, plus the
    int8 codes and fp32 scales of Q and (smoothed) K.  Dense q [B,Hq,N,d], k [B,Hkv,N,d],
    or varlen q [T,Hq,d], k [T,Hkv,d] with cu_seqlens and max_seqlen; logits are
    [B,Hq,row_end-row_begin,N] (entries past a sequence's length stay 0).
    groups = (q_group, k_group, q_outlier_ratio) selects the grouped quantisation of
    attn_w8a8_fwd.  Returns a dict."""
    _need_cuda(q, k, cu_seqlens, workspace)
    if cu_seqlens is None:
        B, Hq, N, d = q.shape
        T = 0
        code_shape = lambda H: (B, H, N)  # noqa: E731
    else:
        T, Hq, d = q.shape
        B = cu_seqlens.numel() - 1
        if max_seqlen is None:
            raise ValueError("varlen logits need max_seqlen")
        N = int(max_seqlen)
        code_shape = lambda H: (T, H)  # noqa: E731
    Hkv = k.shape[-2] if cu_seqlens is not None else k.shape[1]
    row_end = N if row_end is None else row_end
    dev = q.device
    logits = (torch.zeros((B, Hq, row_end - row_begin, N), dtype=torch.int32, device=dev) if want_logits else None)
    res = dict(logits=logits)
    if want_codes:
        res.update(q_codes=torch.empty((*code_shape(Hq), d), dtype=torch.int8, device=dev),
                   q_scales=torch.empty(code_shape(Hq), dtype=torch.float32, device=dev),
                   k_codes=torch.empty((*code_shape(Hkv), d), dtype=torch.int8, device=dev),
                   k_scales=torch.empty(code_shape(Hkv), dtype=torch.float32, device=dev))
    ws_bytes = prefill_workspace_bytes(B, Hq, Hkv, N, d, T)
    ws = workspace if workspace is not None else torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    head = (_ptr(q), _ptr(k), _dt(q), B, Hq, Hkv, N, d, _ptr(cu_seqlens), T, int(bool(smooth_k)))
    tail = (row_begin, row_end, _ptr(logits), _ptr(res.get("q_codes")), _ptr(res.get("q_scales")),
            _ptr(res.get("k_codes")), _ptr(res.get("k_scales")), _ptr(ws), ws.numel(), _stream(dev))
    if groups is None:
        _check(lib().sl8_attn_int8_qk_logits_debug(*head, *tail), "sl8_attn_int8_qk_logits_debug")
    else:
        g = (int(groups[0]), int(groups[1]), float(groups[2]))
        _check(lib().sl8_attn_w8a8_qk_logits_debug(*head, *g, *tail), "sl8_attn_w8a8_qk_logits_debug")
    return res


# ------------------------------------------------------------------ decode

def decode_num_splits(B: int, Hkv: int, Lmax: int, d: int, num_splits: int = 0) -> int:
    """Effective split count of the decode for this shape (0 = automatic)."""
    return int(lib().sl8_attn_decode_num_splits(B, Hkv, Lmax, d, num_splits))


def decode_workspace(B: int, Hq: int, Hkv: int, Lmax: int, d: int, num_splits: int = 0, device=None):
    """The decode's split partials carved from one buffer of
    sl8_attn_decode_workspace_size bytes: (o_partial [B,Hq,S,d], lse_partial [B,Hq,S])
    fp32 views, at the offsets the header states."""
    S = decode_num_splits(B, Hkv, Lmax, d, num_splits)
    nbytes = int(lib().sl8_attn_decode_workspace_size(B, Hq, Hkv, Lmax, d, num_splits))
    off = int(lib().sl8_attn_decode_lse_offset(B, Hq, Hkv, Lmax, d, num_splits))
    if S <= 0 or nbytes == 0:
        raise SL8Error(SL8_ERR_UNSUPPORTED, "sl8_attn_decode_workspace_size")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    o_partial = ws[:B * Hq * S * d * 4].view(torch.float32).view(B, Hq, S, d)
    lse_partial = ws[off:off + B * Hq * S * 4].view(torch.float32).view(B, Hq, S)
    return o_partial, lse_partial


def attn_int8_decode_splitkv(q, k_cache, k_scale, v_cache, v_scale, seqlens, num_splits=0, o_partial=None,
                             lse_partial=None):
    """Split-KV partials (normalised O [B,Hq,S,d] fp32, lse [B,Hq,S] fp32)."""
    _need_cuda(q, k_cache, k_scale, v_cache, v_scale, seqlens)
    B, Hq, d = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    S = decode_num_splits(B, Hkv, Lmax, d, num_splits)
    if o_partial is None and lse_partial is None and S > 0:
        o_partial, lse_partial = decode_workspace(B, Hq, Hkv, Lmax, d, num_splits, q.device)
    if o_partial is None:
        o_partial = torch.empty((B, Hq, max(S, 1), d), dtype=torch.float32, device=q.device)
    if lse_partial is None:
        lse_partial = torch.empty((B, Hq, max(S, 1)), dtype=torch.float32, device=q.device)
    _check(lib().sl8_attn_int8_decode_splitkv(_ptr(q), _dt(q), _ptr(k_cache), _ptr(k_scale), _ptr(v_cache),
                                              _ptr(v_scale), _ptr(seqlens), B, Hq, Hkv, Lmax, d, num_splits,
                                              _ptr(o_partial), _ptr(lse_partial), _stream(q.device)),
           "sl8_attn_int8_decode_splitkv")
    return o_partial, lse_partial


def attn_decode_combine(o_partial, lse_partial, seqlens, Lmax, out_dtype=torch.bfloat16, return_lse=False, out=None):
    _need_cuda(o_partial, lse_partial, seqlens)
    B, Hq, S, d = o_partial.shape
    if out is None:
        out = torch.empty((B, Hq, d), dtype=out_dtype, device=o_partial.device)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=o_partial.device) if return_lse else None
    _check(lib().sl8_attn_decode_combine(_ptr(o_partial), _ptr(lse_partial), _ptr(seqlens), B, Hq, Lmax, d, S,
                                         _ptr(out), _dt(out), _ptr(lse), _stream(o_partial.device)),
           "sl8_attn_decode_combine")
    return (out, lse) if return_lse else out


def attn_int8_decode(q, k_cache, k_scale, v_cache, v_scale, seqlens, num_splits=0, out_dtype=None, return_lse=False,
                     o_partial=None, lse_partial=None, out=None):
    """Split-KV decode plus combine: out [B, Hq, d] (dtype q.dtype unless given)."""
    o_p, l_p = attn_int8_decode_splitkv(q, k_cache, k_scale, v_cache, v_scale, seqlens, num_splits, o_partial,
                                        lse_partial)
    return attn_decode_combine(o_p, l_p, seqlens, k_cache.shape[2], out_dtype or q.dtype, return_lse, out)


def attn_int8_decode_verify(q, k_cache, k_scale, v_cache, v_scale, seqlens, tree_mask, num_splits=0, out_dtype=None,
                            return_lse=False, o_partial=None, lse_partial=None, out=None):
    """Speculative-decode verification: q [B, T, Hq, d] draft queries, tree_mask [B, T] int32
    (bit u of row (b, t): query t sees draft token u, which sits at position L_b - T + u of
    the cache).  Returns out [B, T, Hq, d] (and the LSE [B, T, Hq] with return_lse)."""
    _need_cuda(q, k_cache, k_scale, v_cache, v_scale, seqlens, tree_mask)
    if tree_mask.dtype != torch.int32:
        raise TypeError("tree_mask must be int32 (bit u: draft token u is visible)")
    B, T, Hq, d = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    S = int(lib().sl8_attn_decode_verify_num_splits(B, T, Hq, Hkv, Lmax, d, num_splits))
    if o_partial is None:
        o_partial = torch.empty((B * T, Hq, max(S, 1), d), dtype=torch.float32, device=q.device)
    if lse_partial is None:
        lse_partial = torch.empty((B * T, Hq, max(S, 1)), dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty((B, T, Hq, d), dtype=out_dtype or q.dtype, device=q.device)
    lse = torch.empty((B, T, Hq), dtype=torch.float32, device=q.device) if return_lse else None
    _check(lib().sl8_attn_int8_decode_verify(_ptr(q), _dt(q), _ptr(k_cache), _ptr(k_scale), _ptr(v_cache),
                                             _ptr(v_scale), _ptr(seqlens), _ptr(tree_mask), T, B, Hq, Hkv, Lmax, d,
                                             num_splits, _ptr(o_partial), _ptr(lse_partial), _ptr(out), _dt(out),
                                             _ptr(lse), _stream(q.device)), "sl8_attn_int8_decode_verify")
    return (out, lse) if return_lse else out


def attn_int8_decode_splitkv_f16v(q, k_cache, k_scale, v_cache, seqlens, num_splits=0, o_partial=None,
                                  lse_partial=None):
    """Split-KV partials with an int8 K cache and an fp16 V cache [B, Hkv, Lmax, d]."""
    _need_cuda(q, k_cache, k_scale, v_cache, seqlens)
    if v_cache.dtype != torch.float16:
        raise ValueError("v_cache must be float16")
    B, Hq, d = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    S = decode_num_splits(B, Hkv, Lmax, d, num_splits)
    if o_partial is None:
        o_partial = torch.empty((B, Hq, max(S, 1), d), dtype=torch.float32, device=q.device)
    if lse_partial is None:
        lse_partial = torch.empty((B, Hq, max(S, 1)), dtype=torch.float32, device=q.device)
    _check(lib().sl8_attn_int8_decode_splitkv_f16v(_ptr(q), _dt(q), _ptr(k_cache), _ptr(k_scale), _ptr(v_cache),
                                                   _ptr(seqlens), B, Hq, Hkv, Lmax, d, num_splits, _ptr(o_partial),
                                                   _ptr(lse_partial), _stream(q.device)),
           "sl8_attn_int8_decode_splitkv_f16v")
    return o_partial, lse_partial


def attn_int8_decode_f16v(q, k_cache, k_scale, v_cache, seqlens, num_splits=0, out_dtype=None, return_lse=False,
                          o_partial=None, lse_partial=None, out=None):
    """Split-KV decode (int8 K, fp16 V) plus combine: out [B, Hq, d] (dtype q.dtype unless given)."""
    o_p, l_p = attn_int8_decode_splitkv_f16v(q, k_cache, k_scale, v_cache, seqlens, num_splits, o_partial,
                                             lse_partial)
    return attn_decode_combine(o_p, l_p, seqlens, k_cache.shape[2], out_dtype or q.dtype, return_lse, out)


def attn_int8_paged_decode_splitkv(q, k_pages, k_scale_pages, v_pages, v_scale_pages, block_table, seqlens,
                                   num_splits=0, o_partial=None, lse_partial=None):
    """Split-KV partials over a paged k8v8 cache: pages [num_pages, Hkv, page_size, d] int8,
    scales [num_pages, Hkv, page_size] fp32, block_table [B, max_blocks] int32."""
    _need_cuda(q, k_pages, k_scale_pages, v_pages, v_scale_pages, block_table, seqlens)
    B, Hq, d = q.shape
    num_pages, Hkv, page_size, _ = k_pages.shape
    max_blocks = block_table.shape[1]
    S = decode_num_splits(B, Hkv, max_blocks * page_size, d, num_splits)
    if o_partial is None:
        o_partial = torch.empty((B, Hq, max(S, 1), d), dtype=torch.float32, device=q.device)
    if lse_partial is None:
        lse_partial = torch.empty((B, Hq, max(S, 1)), dtype=torch.float32, device=q.device)
    _check(lib().sl8_attn_int8_paged_decode_splitkv(_ptr(q), _dt(q), _ptr(k_pages), _ptr(k_scale_pages),
                                                    _ptr(v_pages), _ptr(v_scale_pages), _ptr(block_table),
                                                    max_blocks, page_size, num_pages, _ptr(seqlens), B, Hq, Hkv, d,
                                                    num_splits, _ptr(o_partial), _ptr(lse_partial),
                                                    _stream(q.device)),
           "sl8_attn_int8_paged_decode_splitkv")
    return o_partial, lse_partial


def attn_int8_paged_decode(q, k_pages, k_scale_pages, v_pages, v_scale_pages, block_table, seqlens, num_splits=0,
                           out_dtype=None, return_lse=False, o_partial=None, lse_partial=None, out=None):
    """Paged split-KV decode plus combine: out [B, Hq, d] (dtype q.dtype unless given)."""
    o_p, l_p = attn_int8_paged_decode_splitkv(q, k_pages, k_scale_pages, v_pages, v_scale_pages, block_table,
                                              seqlens, num_splits, o_partial, lse_partial)
    lmax = block_table.shape[1] * k_pages.shape[2]
    return attn_decode_combine(o_p, l_p, seqlens, lmax, out_dtype or q.dtype, return_lse, out)


def attn_int8_decode_logits_debug(q, k_cache, k_scale, v_cache, v_scale, seqlens):
    """Exact int32 decode logits [B, Hq, Lmax] (entries t >= L_b stay 0) and q codes/scales."""
    _need_cuda(q, k_cache, k_scale, v_cache, v_scale, seqlens)
    B, Hq, d = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    dev = q.device
    S = decode_num_splits(B, Hkv, Lmax, d, 0)
    logits = torch.zeros((B, Hq, Lmax), dtype=torch.int32, device=dev)
    q_codes = torch.empty((B, Hq, d), dtype=torch.int8, device=dev)
    q_scales = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    o_p = torch.empty((B, Hq, max(S, 1), d), dtype=torch.float32, device=dev)
    l_p = torch.empty((B, Hq, max(S, 1)), dtype=torch.float32, device=dev)
    _check(lib().sl8_attn_int8_decode_logits_debug(_ptr(q), _dt(q), _ptr(k_cache), _ptr(k_scale), _ptr(v_cache),
                                                   _ptr(v_scale), _ptr(seqlens), B, Hq, Hkv, Lmax, d, _ptr(logits),
                                                   _ptr(q_codes), _ptr(q_scales), _ptr(o_p), _ptr(l_p),
                                                   _stream(dev)), "sl8_attn_int8_decode_logits_debug")
    return dict(logits=logits, q_codes=q_codes, q_scales=q_scales)


# ------------------------------------------------------------------ status / tracing

def last_device_status(device=None) -> tuple[int, int]:
    """(status, site) of the device's status word after synchronising the current stream; clears it."""
    site = _INT(0)
    dev = torch.device("cuda") if device is None else torch.device(device)
    st = lib().sl8_last_device_status(_stream(dev), ctypes.byref(site))
    return int(st), int(site.value)


def set_spin_limit_ns(ns: int) -> None:
    lib().sl8_set_spin_limit_ns(int(ns))


def get_spin_limit_ns() -> int:
    return int(lib().sl8_get_spin_limit_ns())


def selftest_timeout(limit_ns: int, device=None) -> None:
    dev = torch.device("cuda") if device is None else torch.device(device)
    _check(lib().sl8_selftest_timeout(int(limit_ns), _stream(dev)), "sl8_selftest_timeout")


def trace_enable(on: bool = True) -> None:
    lib().sl8_trace_enable(int(bool(on)))


def trace_collect(max_names: int = 64) -> dict[str, tuple[int, float]]:
    """{kernel name: (launches, total ms)} since the last collect (synchronises the traced events)."""
    names = (ctypes.c_char_p * max_names)()
    launches = (_I64 * max_names)()
    ms = (ctypes.c_double * max_names)()
    n = lib().sl8_trace_collect(names, launches, ms, max_names)
    return {names[i].decode(): (int(launches[i]), float(ms[i])) for i in range(n)}
