"""Shared helpers of the parity tests: conversions and the tolerance rules.

Tolerances (floating point, GPU bf16 path with fp32 accumulation against the
fp64 oracle that never rounds):
  layer output / per-stage h, y:  max|got-ref| <= 2e-2 * max|ref|  and
                                  ||got-ref||_F / ||ref||_F <= 5e-3
  routing weights (same fp32 logits on both sides): |got-ref| <= 2e-6
  router logits: |got-ref| <= 2 * gamma_D * sum_d |x_d w_d| + |bias| * 2^-23,
                 gamma_D = D * 2^-24 (worst-case bound of a length-D fp32 sum)
Integer outputs (ids, offsets, permutation indices, permuted rows) are exact.
"""
import numpy as np
import torch

from oracle import oracle as O

MAX_ABS_FRAC = 2e-2
REL_FROB = 5e-3
WEIGHT_ATOL = 2e-6
NEAR_TIE = 1e-5


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return O.bf16_to_f64(bits(t))
    return t.detach().cpu().numpy().astype(np.float64)


def close_metrics(got, ref) -> dict:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = got - ref
    return dict(max_abs=float(np.max(np.abs(d))) if d.size else 0.0,
                max_ref=float(np.max(np.abs(ref))) if ref.size else 0.0,
                rel_frob=float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-300)) if d.size else 0.0)


def assert_close(got, ref, name="", max_abs_frac=MAX_ABS_FRAC, rel_frob=REL_FROB) -> dict:
    m = close_metrics(got, ref)
    assert np.all(np.isfinite(np.asarray(got, np.float64))), f"{name}: non-finite output"
    assert m["max_abs"] <= max_abs_frac * m["max_ref"] + 1e-30, f"{name}: {m}"
    assert m["rel_frob"] <= rel_frob, f"{name}: {m}"
    return m


def near_tie_mask(L: np.ndarray, K: int) -> np.ndarray:
    """Tokens whose K-th and (K+1)-th largest logits are closer than 1e-5."""
    E = L.shape[1]
    if K >= E:
        return np.zeros(L.shape[0], bool)
    s = -np.sort(-L, axis=1)
    return (s[:, K - 1] - s[:, K]) < NEAR_TIE


def logits_bound(x64, wg64, bias64=None) -> np.ndarray:
    D = x64.shape[1]
    gamma = D * 2.0 ** -24
    b = 2 * gamma * (np.abs(x64) @ np.abs(wg64).T)
    if bias64 is not None:
        b = b + np.abs(bias64)[None, :] * 2.0 ** -23
    return b + 1e-30


def random_ids(N, E, K, gen: torch.Generator, skew=None) -> torch.Tensor:
    """[N,K] int32, K distinct experts per token.  With skew, low expert
    indices are favoured (Gumbel top-K over skewed scores)."""
    scores = torch.rand((N, E), generator=gen, dtype=torch.float64)
    if skew:
        scores = torch.log(scores) / (torch.arange(1, E + 1, dtype=torch.float64) ** -skew)
    return torch.topk(scores, K, dim=1).indices.to(torch.int32)
