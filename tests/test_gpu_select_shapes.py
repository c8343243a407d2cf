"""GPU parity of the two-stage retrieval on shapes that take the selection
kernel's less common paths, against the fp64 oracle (WorldAttention review
page, HKV section: prompt-stage top-1 chunk by cosine, page-stage
alpha = Qbar^T Kbar / sqrt(d_k), top-K_p with ties to the lower page):

* one column block for all heads (a head row under 32 values, or not whole
  16-byte vectors), and several heads per column block;
* head rows that are not a multiple of 4 values (scalar dot products);
* a prompt dimension that is not a multiple of 4 (scalar prompt loop) and many
  past chunks;
* more than 32 candidates (block bitonic sort), and more partial scores than
  the last CTA stages in shared memory;
* a page set per head with more than 32 candidates;
* very few and odd query counts.

Indices and the chunk pick are compared bit for bit behind the margin guard
(a boundary within fp32 rounding would be a tie and the seed must change);
scores within fp32 rounding of the oracle's."""

import numpy as np
import pytest
import torch

import oracle as O
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
from tests._util import (assert_selection_margin, mean_error_bound, np_of,
                         page_mean_error_bounds, score_error_bound)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(c, per_head, use_prompt=True):
    kp = c.k_pages.to(DEV)
    kbar = torch.empty((c.n_pages, c.n_heads, c.head_dim), dtype=torch.float32, device=DEV)
    wa.wa_page_summarize(kp, kbar)
    shape = (c.n_heads, c.k_p) if per_head else (c.k_p,)
    idx = torch.full(shape, -1, dtype=torch.int32, device=DEV)
    sc = torch.empty(shape, dtype=torch.float32, device=DEV)
    ch = torch.full((1,), -9, dtype=torch.int32, device=DEV)
    pc = c.prompt_chunks.to(DEV) if use_prompt and c.prompt_chunks is not None else None
    cur = c.prompt_cur.to(DEV) if pc is not None else None
    fn = wa.wa_select_pages_per_head if per_head else wa.wa_select_pages
    fn(c.q.to(DEV), kbar, cur, pc, c.pages_per_chunk, c.k_p, idx, sc, ch)
    wa.wa_check()
    return kbar, idx.cpu().numpy(), sc.cpu().numpy(), int(ch.item())


def _check(c, per_head=False, use_prompt=True):
    kbar_dev, g_idx, g_sc, g_ch = _run(c, per_head, use_prompt)
    okp, oq = np_of(c.k_pages), np_of(c.q)
    kbar = O.page_summarize(okp)
    pc = np_of(c.prompt_chunks) if use_prompt and c.prompt_chunks is not None else None
    cur = np_of(c.prompt_cur) if pc is not None else None
    sel = O.select_pages_per_head if per_head else O.select_pages
    idx, sc, ch = sel(oq, kbar, cur, pc, c.pages_per_chunk, c.k_p)
    assert g_ch == ch
    cand = O.candidate_pages(c.n_pages, ch, c.pages_per_chunk)
    qbar = O.mean_query(oq)
    dq, dk = mean_error_bound(O.as_f64(oq)), page_mean_error_bounds(okp)
    if per_head:
        alpha = O.page_scores_per_head(qbar, kbar, cand, c.head_dim)
        for h in range(c.n_heads):
            bound = score_error_bound(dq[h:h + 1], dk[:, h:h + 1], qbar[h:h + 1],
                                      kbar[:, h:h + 1], c.head_dim)
            assert_selection_margin(alpha[h], cand, c.k_p, bound)
            assert g_idx[h].tolist() == idx[h].tolist()
            assert np.all(np.abs(g_sc[h] - sc[h]) <= bound[idx[h]])
    else:
        alpha = O.page_scores(qbar, kbar, cand, c.head_dim)
        bound = score_error_bound(dq, dk, qbar, kbar, c.head_dim)
        assert_selection_margin(np.array(alpha), cand, c.k_p, bound)
        assert g_idx.tolist() == idx.tolist()
        # every returned score within the rounding bound of its page's score
        assert np.all(np.abs(g_sc - sc) <= bound[idx])


def _case(tag, H, d, n_pages, ppc, n_chunks, prompt_dim, k_p, n_q, dtype, P=24, recall=None,
          plant=None, strength=0.0):
    return synth.make_chunk_case(f"selshape_{tag}", n_heads=H, head_dim=d, page_tokens=P,
                                 n_pages=n_pages, pages_per_chunk=ppc, n_chunks=n_chunks,
                                 prompt_dim=prompt_dim, k_p=k_p, n_q=n_q, n_loc=1, dtype=dtype,
                                 recall_chunk=recall, plant_pages=plant,
                                 plant_strength=strength)


@pytest.mark.parametrize("tag,H,d,dtype", [
    ("onecb_fp32_d12", 3, 12, torch.float32),     # head rows under 32 values: one column block
    ("scalar_fp32_d6", 2, 6, torch.float32),      # head rows not a multiple of 4: scalar dots
    ("grouped_bf16_d40", 8, 40, torch.bfloat16),  # 5 vectors a head: 8 heads per block
    ("grouped_bf16_d64", 6, 64, torch.bfloat16),  # 8 vectors a head: 2 heads per block (6 % 4)
    ("wide_fp32_d256", 4, 256, torch.float32),    # 64 vectors a head: one head per block
])
def test_column_block_layouts(tag, H, d, dtype):
    c = _case(tag, H, d, n_pages=20, ppc=4, n_chunks=5, prompt_dim=64, k_p=2, n_q=333,
              dtype=dtype, recall=2)
    _check(c)


@pytest.mark.parametrize("n_q", [1, 5, 17, 4679])
def test_query_counts(n_q):
    c = _case(f"nq{n_q}", 12, 128, n_pages=16, ppc=8, n_chunks=2, prompt_dim=256, k_p=4,
              n_q=n_q, dtype=torch.bfloat16, recall=1)
    _check(c)


def test_many_chunks_and_a_ragged_prompt():
    """20 past chunks of 3 pages, prompt embeddings of dim 37 (scalar loop)."""
    c = _case("chunks", 4, 64, n_pages=60, ppc=3, n_chunks=20, prompt_dim=37, k_p=2, n_q=200,
              dtype=torch.bfloat16, recall=13)
    _check(c)


def test_many_candidates_sorted_in_blocks():
    """No prompt stage, 200 candidates (> 32: the block bitonic sort)."""
    c = _case("cand200", 4, 64, n_pages=200, ppc=1, n_chunks=0, prompt_dim=0, k_p=7, n_q=150,
              dtype=torch.bfloat16, plant=[3, 77, 150, 199], strength=0.3)
    _check(c, use_prompt=False)


def test_partial_scores_beyond_the_staging_area():
    """4 heads x 1,100 candidate pages = 4,400 partial scores, more than the
    last CTA stages in shared memory (4,096): they are summed from scratch."""
    c = _case("cand1100", 4, 32, n_pages=1100, ppc=1, n_chunks=0, prompt_dim=0, k_p=5, n_q=64,
              dtype=torch.bfloat16, P=4, plant=[10, 500, 1099], strength=0.6)
    _check(c, use_prompt=False)


def test_per_head_sets_with_many_candidates():
    """A page set per head with 48 candidates (> 32: a block sort per head)."""
    c = _case("ph48", 3, 64, n_pages=96, ppc=48, n_chunks=2, prompt_dim=32, k_p=3, n_q=120,
              dtype=torch.bfloat16, recall=1)
    _check(c, per_head=True)
