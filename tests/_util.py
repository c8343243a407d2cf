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


def score_error_bound(q64: np.ndarray, k_pages64_abs_means: np.ndarray, qbar: np.ndarray,
                      kbar: np.ndarray, n_q: int, page_tokens: int, head_dim: int) -> np.ndarray:
    """Probabilistic bound on |alpha_gpu - alpha_exact| per page for fp32
    sums of n terms (error <= lambda*sqrt(n)*u*sum|terms|, Higham & Mary):
    the mean query, the page means, and the final dot product.

    q64: [n_q][H][d] fp64 queries; k_pages64_abs_means: [n_pages][H][d] mean |k|.
    """
    rq = LAMBDA * math.sqrt(n_q) * U32 + U32
    rk = LAMBDA * math.sqrt(page_tokens) * U32 + U32
    dq = rq * np.abs(q64).mean(axis=0)                 # |dQbar| per element
    dk = rk * k_pages64_abs_means                      # |dKbar| per page element
    c = q64.shape[1] * q64.shape[2]
    rd = LAMBDA * math.sqrt(c) * U32 + U32
    terms = np.abs(qbar)[None] * np.abs(kbar)
    bound = (np.sum(dq[None] * np.abs(kbar), axis=(1, 2)) + np.sum(np.abs(qbar)[None] * dk,
                                                                   axis=(1, 2))
             + rd * terms.sum(axis=(1, 2))) / math.sqrt(head_dim)
    return bound


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
