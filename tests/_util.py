"""Shared helpers for the GPU parity tests (test code only)."""

import math

import numpy as np
import torch

import oracle as O
from sparse_kv_cache_page_gb300 import synth

# Attention tolerances for bf16 inputs with fp32 accumulation, and for fp32 inputs.
BF16_MAX_ABS, BF16_MEAN_ABS = 1e-2, 1e-3
F32_MAX_ABS = 1e-5
# LSE is fp32 from fp32-accumulated logits of exact bf16 inputs: error ~1e-5.
LSE_ABS = 2e-3

U32 = 2.0 ** -24      # unit roundoff of fp32
LAMBDA = 4.0          # probabilistic rounding-error bound constant (Higham & Mary, 2019)


def np_of(t: torch.Tensor) -> np.ndarray:
    return synth.to_oracle(t)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def assert_attn_close(o_gpu: torch.Tensor, o_ref: np.ndarray, dtype, what=""):
    err = np.abs(f64(o_gpu) - o_ref)
    if dtype == torch.bfloat16:
        assert err.max() <= BF16_MAX_ABS and err.mean() <= BF16_MEAN_ABS, \
            f"{what}: max|err|={err.max():.3e} mean|err|={err.mean():.3e}"
    else:
        assert err.max() <= F32_MAX_ABS, f"{what}: max|err|={err.max():.3e}"
    return err


def mean_error_bound(x64: np.ndarray) -> np.ndarray:
    """Probabilistic bound, per element, on the fp32 rounding error of the
    mean over axis 0 of x64 ([n][...] fp64): lambda*u*||s||_2 / n + u*|mean|,
    with s_k the partial sums in row order.  The error of a floating-point sum
    is sum_k delta_k s_k with independent |delta_k| <= u, which is below
    lambda*u*||s||_2 with probability >= 1 - 2 exp(-lambda^2 / 2) (Higham &
    Mary, 2019, the lemma behind their sqrt(n) * u * sum|x_i| bound; that
    simplification bounds ||s||_2 for any order but ignores the cancellation
    of zero-mean data, by a factor of about sqrt(n)).  Blocked or tree orders,
    as the kernels use, have partial sums no larger than the row-order ones
    for such data."""
    n = x64.shape[0]
    s = np.cumsum(x64, axis=0)
    return LAMBDA * U32 * np.sqrt(np.einsum("i...,i...->...", s, s)) / n + U32 * np.abs(s[-1]) / n


def score_error_bound(dq: np.ndarray, dk: np.ndarray, qbar: np.ndarray, kbar: np.ndarray,
                      head_dim: int) -> np.ndarray:
    """Bound on |alpha_gpu - alpha_exact| per page from the error bounds of
    the mean query (dq [H][d]) and of the page means (dk [n_pages][H][d],
    see mean_error_bound), plus the fp32 dot product of H*d terms and the
    final scaling (Higham & Mary's lambda*sqrt(n)*u*sum|terms| form)."""
    c = qbar.size
    rd = LAMBDA * math.sqrt(c) * U32 + U32
    terms = np.abs(qbar)[None] * np.abs(kbar)
    return (np.sum(dq[None] * np.abs(kbar), axis=(1, 2)) + np.sum(np.abs(qbar)[None] * dk, axis=(1, 2))
            + rd * terms.sum(axis=(1, 2))) / math.sqrt(head_dim)


def page_mean_error_bounds(k_pages) -> np.ndarray:
    """mean_error_bound of every page of a bank [n_pages][P][H][d] (bf16 bits
    or float), one page at a time: [n_pages][H][d]."""
    import oracle as O
    return np.stack([mean_error_bound(O.as_f64(k_pages[j])) for j in range(len(k_pages))])


def assert_selection_margin(alpha_all: np.ndarray, cand, k_p: int, bound: np.ndarray):
    """The oracle's gap between the k_p-th and (k_p+1)-th candidate scores must
    exceed the rounding bound of both; otherwise the case is a tie within
    rounding and the seed must change (the kernel is not loosened)."""
    cand = list(cand)
    if k_p >= len(cand):
        return
    order = sorted(range(len(cand)), key=lambda i: (-alpha_all[i], cand[i]))
    a, b = order[k_p - 1], order[k_p]
    gap = alpha_all[a] - alpha_all[b]
    need = bound[cand[a]] + bound[cand[b]]
    assert gap > need, f"tie within rounding: gap {gap:.3e} <= bound {need:.3e}; change the seed"
