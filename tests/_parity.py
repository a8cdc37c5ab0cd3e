"""Shared helpers for the GPU parity tests (not collected by pytest).

Tolerances (the oracle is fp64 after the int32 dot):
  * int8 codes, fp32 scales, K means and int32 logits: bit-exact.
  * fp32 output (same kernel, only the final store differs): max-abs <= 2e-3 and
    mean-abs <= 2e-4 against the oracle.
  * bf16/fp16 output: a bf16 value cannot be closer to the fp64 oracle than half of
    its own spacing (3.9e-3 for |o| in [1, 2)), so each element must lie within
    max(2e-3, one output ulp at the oracle value) of the oracle, and the mean
    absolute distance to the correctly rounded oracle must stay <= 2e-4.
"""
import numpy as np
import torch

MAX_ABS = 2e-3
MEAN_ABS = 2e-4


def to_np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    mant = {torch.bfloat16: 7, torch.float16: 10}[dtype]
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    return 2.0 ** (np.floor(np.log2(ax)) - mant)


def check_f32(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    mask = ~np.isnan(ref)
    g, r = gpu[mask].astype(np.float64), ref[mask]
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - r)
    assert err.max() <= MAX_ABS, f"{what}: max-abs {err.max():.3e} > {MAX_ABS}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean-abs {err.mean():.3e} > {MEAN_ABS}"
    return float(err.max()), float(err.mean())


def check_half(gpu: torch.Tensor, ref: np.ndarray, what: str = ""):
    dt = gpu.dtype
    g = to_np32(gpu).astype(np.float64)
    mask = ~np.isnan(ref)
    g, r = g[mask], ref[mask]
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - r)
    bound = np.maximum(MAX_ABS, ulp(r, dt))
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond max(2e-3, 1 ulp); worst {err.max():.3e}"
    rounded = torch.from_numpy(r).to(dt).double().numpy()
    mean_rounded = np.abs(g - rounded).mean()
    assert mean_rounded <= MEAN_ABS, f"{what}: mean-abs vs rounded oracle {mean_rounded:.3e}"
    return float(err.max()), float(mean_rounded)


def sample_rows(rng, nseq_lens, Hq, per_head=16, edge=True):
    """(seq, hq, i) rows: the first and last rows, rows around tile edges and random ones."""
    rows = []
    for s, L in enumerate(nseq_lens):
        for h in range(Hq):
            cand = set()
            if edge:
                cand.update(i for i in (0, 1, 2, 63, 127, 128, 129, L - 2, L - 1) if 0 <= i < L)
            cand.update(int(i) for i in rng.integers(0, L, size=min(per_head, L)))
            rows.extend((s, h, i) for i in sorted(cand))
    return rows
