"""Failure detection on the GPU without a fault: bounded waits give up and report,
and device-side argument checks report instead of reading out of bounds.  Nothing
here traps, faults or hangs the GPU: the timeout case waits on a barrier that
nothing arrives on, with a 1 ms limit."""
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


def test_bounded_wait_times_out_and_context_survives():
    assert sl8.last_device_status() == (sl8.SL8_OK, 0)
    sl8.selftest_timeout(1_000_000)  # 1 ms
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_ERR_TIMEOUT and site == 999
    # the status is cleared by the read, and the context still runs work
    assert sl8.last_device_status() == (sl8.SL8_OK, 0)
    w = W.custom(4001, B=1, Hq=2, Hkv=1, N=64, d=64, dtype="bf16")
    q, k, v = (t.to(DEV) for t in W.prefill_dense(w))
    out = sl8.attn_int8_fwd(q, k, v)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert sl8.last_device_status() == (sl8.SL8_OK, 0)


def test_bad_cu_seqlens_reported_not_faulted():
    w = W.custom(4002, kind="varlen", B=2, Hq=2, Hkv=1, d=64, dtype="bf16", extra={"lengths": [40, 50]})
    q, k, v, cu = W.prefill_varlen(w)
    # second sequence claims more tokens than max_seqlen allows
    out = sl8.attn_int8_fwd(q.to(DEV), k.to(DEV), v.to(DEV), cu_seqlens=cu.to(DEV), max_seqlen=45)
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_ERR_DEVICE_ARG and site == 900
    assert torch.isfinite(out[:40].float()).all()


def test_bad_decode_seqlen_reported():
    B, Hq, Hkv, L, d = 1, 2, 1, 64, 64
    q = torch.zeros((B, Hq, d), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((B, Hkv, L, d), dtype=torch.int8, device=DEV)
    ks = torch.ones((B, Hkv, L), dtype=torch.float32, device=DEV)
    seq = torch.tensor([L + 5], dtype=torch.int32, device=DEV)
    sl8.attn_int8_decode(q, kc, ks, kc, ks, seq)
    st, site = sl8.last_device_status()
    assert st == sl8.SL8_ERR_DEVICE_ARG and site == 700


def test_trace_records_kernels():
    sl8.trace_enable(True)
    try:
        w = W.custom(4003, B=1, Hq=4, Hkv=2, N=256, d=128, dtype="bf16")
        q, k, v = (t.to(DEV) for t in W.prefill_dense(w))
        sl8.attn_int8_fwd(q, k, v)
        rec = sl8.trace_collect()
    finally:
        sl8.trace_enable(False)
    for name in ("kv_partials", "quant_qk", "prefill_attn"):
        assert name in rec and rec[name][0] == 1 and rec[name][1] > 0
