"""GPU parity of page summaries, two-stage retrieval and the gather, through
the C ABI, against the fp64 oracle.  Indices and gathered bytes must match
bit for bit; summaries and scores within fp32 rounding."""

import numpy as np
import pytest
import torch

import oracle as O
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
from tests._util import (assert_selection_margin, f64, mean_error_bound, np_of,
                         page_mean_error_bounds, score_error_bound)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _summarize(kp):
    n, p, h, d = kp.shape
    out = torch.empty((n, h, d), dtype=torch.float32, device=DEV)
    wa.wa_page_summarize(kp, out)
    wa.wa_check()
    return out


@pytest.mark.parametrize("dtype,n_pages,P,H,d", [
    (torch.float32, 8, 32, 1, 64),        # tiny fp32 workload shape
    (torch.bfloat16, 5, 1000, 12, 128),   # ragged split of rows
    (torch.bfloat16, 3, 77, 32, 128),     # 4096-wide rows: two vectors per thread
    (torch.float32, 2, 50, 64, 128),      # 8192-wide fp32 rows
    (torch.bfloat16, 700, 3, 2, 8),       # many tiny pages: one CTA per page
    (torch.bfloat16, 1, 12480, 12, 128),  # one full page
])
def test_page_summarize(dtype, n_pages, P, H, d):
    kp = synth.normal((n_pages, P, H, d), synth.seed_of("sum", n_pages, P, H, d), dtype=dtype)
    got = _summarize(kp.to(DEV))
    ref = O.page_summarize(np_of(kp))
    scale = O.as_f64(np_of(kp)).__abs__().mean()
    err = np.abs(f64(got) - ref).max()
    assert err <= 1e-6 * max(1.0, scale) * 8, err


def test_page_summarize_deterministic():
    kp = synth.normal((6, 2000, 12, 128), 7, dtype=torch.bfloat16).to(DEV)
    a, b = _summarize(kp), _summarize(kp)
    assert torch.equal(a, b)


def _select(c, kbar_dev, k_p=None, use_prompt=True):
    k_p = c.k_p if k_p is None else k_p
    idx = torch.full((k_p,), -7, dtype=torch.int32, device=DEV)
    sc = torch.empty(k_p, dtype=torch.float32, device=DEV)
    ch = torch.full((1,), -9, dtype=torch.int32, device=DEV)
    pc = c.prompt_chunks.to(DEV) if (use_prompt and c.prompt_chunks is not None) else None
    cur = c.prompt_cur.to(DEV) if pc is not None else None
    wa.wa_select_pages(c.q.to(DEV), kbar_dev, cur, pc, c.pages_per_chunk, k_p, idx, sc, ch)
    wa.wa_check()
    return idx.cpu().numpy(), sc.cpu().numpy(), int(ch.item())


def _oracle_select(c, k_p=None, use_prompt=True):
    k_p = c.k_p if k_p is None else k_p
    kbar = O.page_summarize(np_of(c.k_pages))
    pc = np_of(c.prompt_chunks) if (use_prompt and c.prompt_chunks is not None) else None
    cur = np_of(c.prompt_cur) if pc is not None else None
    return O.select_pages(np_of(c.q), kbar, cur, pc, c.pages_per_chunk, k_p), kbar


@pytest.mark.parametrize("recall", [0, 1])
def test_select_tiny_fp32_with_prompt(recall):
    c = synth.tiny_fp32_case(recall_chunk=recall)
    (idx, sc, ch), kbar = _oracle_select(c)
    g_idx, g_sc, g_ch = _select(c, _summarize(c.k_pages.to(DEV)))
    assert g_ch == ch == recall
    assert g_idx.tolist() == idx.tolist()
    assert np.abs(g_sc - sc).max() < 1e-6


def test_select_all_pages_bypasses_prompt():
    c = synth.tiny_fp32_case()
    (idx, sc, ch), _ = _oracle_select(c, k_p=8, use_prompt=False)
    g_idx, g_sc, g_ch = _select(c, _summarize(c.k_pages.to(DEV)), k_p=8, use_prompt=False)
    assert ch == g_ch == -1
    assert g_idx.tolist() == idx.tolist() == list(range(8))


@pytest.mark.parametrize("k_p", [1, 3, 5, 16])
def test_select_random_no_prompt(k_p):
    c = synth.make_chunk_case("sel_rand", n_heads=4, head_dim=64, page_tokens=64, n_pages=37,
                              pages_per_chunk=1, n_chunks=0, prompt_dim=0, k_p=k_p, n_q=200,
                              n_loc=1, dtype=torch.bfloat16)
    (idx, sc, ch), kbar = _oracle_select(c)
    cand = range(c.n_pages)
    alpha = O.page_scores(O.mean_query(np_of(c.q)), kbar, cand, c.head_dim)
    bound = score_error_bound(mean_error_bound(O.as_f64(np_of(c.q))),
                              page_mean_error_bounds(np_of(c.k_pages)), O.mean_query(np_of(c.q)),
                              kbar, c.head_dim)
    assert_selection_margin(alpha, cand, k_p, bound)
    g_idx, g_sc, _ = _select(c, _summarize(c.k_pages.to(DEV)))
    assert g_idx.tolist() == idx.tolist()
    assert np.abs(g_sc - sc).max() < 1e-5


def test_select_exact_ties_go_to_lowest_index():
    c = synth.make_chunk_case("sel_ties", n_heads=2, head_dim=64, page_tokens=16, n_pages=12,
                              pages_per_chunk=4, n_chunks=3, prompt_dim=32, k_p=3, n_q=16,
                              n_loc=1, dtype=torch.float32, recall_chunk=1)
    # duplicate pages 4 == 6 and 5 == 7 (chunk 1 owns pages 4..7); queries favour them
    c.k_pages[6] = c.k_pages[4]
    c.k_pages[7] = c.k_pages[5]
    c.q = (c.k_pages[4] * 2.0 + c.k_pages[5]).contiguous()
    (idx, sc, ch), _ = _oracle_select(c)
    g_idx, g_sc, g_ch = _select(c, _summarize(c.k_pages.to(DEV)))
    assert ch == g_ch == 1
    assert idx.tolist() == [4, 5, 6]          # {4, 6} tie, {5, 7} tie: lowest index wins
    assert g_idx.tolist() == idx.tolist()
    # duplicate prompt embeddings: the lower chunk wins
    c.prompt_chunks[2] = c.prompt_chunks[1]
    (idx, _, ch), _ = _oracle_select(c)
    g_idx, _, g_ch = _select(c, _summarize(c.k_pages.to(DEV)))
    assert ch == g_ch == 1 and g_idx.tolist() == idx.tolist()


def test_select_large_candidate_set():
    """A long history without prompts: top-4 of 1,500 single-frame pages."""
    c = synth.make_chunk_case("sel_many", n_heads=2, head_dim=64, page_tokens=8, n_pages=1500,
                              pages_per_chunk=1, n_chunks=0, prompt_dim=0, k_p=4, n_q=64,
                              n_loc=1, dtype=torch.bfloat16, plant_pages=[3, 777, 1499],
                              plant_strength=0.7)
    (idx, _, _), _ = _oracle_select(c)
    g_idx, _, _ = _select(c, _summarize(c.k_pages.to(DEV)))
    assert g_idx.tolist() == idx.tolist()
    assert {3, 777, 1499} <= set(idx.tolist())


def test_select_worldattention_shape_full():
    """Full one-layer WorldAttention shape: 40 pages of 12,480 tokens, 12 heads,
    prompt dim 4096, top-1 chunk of 5, top-4 of its 8 pages."""
    c = synth.worldattention_case(device=DEV, recall_chunk=3, plant_pages=[26, 29],
                                  plant_strength=0.05)
    kbar_dev = _summarize(c.k_pages)
    g_idx, g_sc, g_ch = _select(c, kbar_dev)
    okp = np_of(c.k_pages)
    kbar = O.page_summarize(okp)
    assert np.abs(f64(kbar_dev) - kbar).max() < 1e-6
    oq = np_of(c.q)
    idx, sc, ch = O.select_pages(oq, kbar, np_of(c.prompt_cur), np_of(c.prompt_chunks),
                                 c.pages_per_chunk, c.k_p)
    cand = O.candidate_pages(c.n_pages, ch, c.pages_per_chunk)
    alpha = O.page_scores(O.mean_query(oq), kbar, cand, c.head_dim)
    bound = score_error_bound(mean_error_bound(O.as_f64(oq)), page_mean_error_bounds(okp),
                              O.mean_query(oq), kbar, c.head_dim)
    assert_selection_margin(np.array(alpha), cand, c.k_p, bound)
    assert g_ch == ch == 3
    assert g_idx.tolist() == idx.tolist()
    assert {26, 29} <= set(idx.tolist())
    assert np.abs(g_sc - sc).max() < 1e-6


# ----------------------------------------------------------------------------
# gather
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n_pages,P,H,d,idx", [
    (9, 50, 2, 64, [7, 0, 3]),
    (6, 12480, 12, 128, [5, 1, 2, 4]),       # full pages, span count not a power of two
    (4, 3, 1, 8, [3, 3, 0, 1, 2]),           # tiny pages, repeated index
])
def test_gather_device_bitexact(n_pages, P, H, d, idx):
    kp = synth.normal((n_pages, P, H, d), 11, dtype=torch.bfloat16).to(DEV)
    vp = synth.normal((n_pages, P, H, d), 12, dtype=torch.bfloat16).to(DEV)
    idx_t = torch.tensor(idx, dtype=torch.int32, device=DEV)
    kb = torch.empty((len(idx) * P, H, d), dtype=torch.bfloat16, device=DEV)
    vb = torch.empty_like(kb)
    wa.wa_gather_pages(kp, vp, idx_t, None, kb, vb)
    wa.wa_check()
    ref_k = O.gather_pages(np_of(kp), idx)
    ref_v = O.gather_pages(np_of(vp), idx)
    assert np.array_equal(np_of(kb), ref_k)
    assert np.array_equal(np_of(vb), ref_v)
    assert torch.equal(kb, torch.index_select(kp, 0, idx_t.long()).reshape(kb.shape))


def test_gather_keys_only_fp32():
    kp = synth.normal((5, 33, 1, 64), 13).to(DEV)
    idx_t = torch.tensor([4, 2], dtype=torch.int32, device=DEV)
    kb = torch.empty((66, 1, 64), dtype=torch.float32, device=DEV)
    wa.wa_gather_pages(kp, None, idx_t, None, kb, None)
    wa.wa_check()
    assert np.array_equal(np_of(kb), O.gather_pages(np_of(kp), [4, 2]))


def test_gather_bad_device_index_reported():
    kp = synth.normal((3, 40, 1, 64), 14, dtype=torch.bfloat16).to(DEV)
    idx_t = torch.tensor([1, 3], dtype=torch.int32, device=DEV)   # 3 is out of range
    kb = torch.full((80, 1, 64), 5.0, dtype=torch.bfloat16, device=DEV)
    wa.wa_gather_pages(kp, None, idx_t, None, kb, None)
    with pytest.raises(wa.WaError) as e:
        wa.wa_check()
    assert e.value.status == 5
    assert torch.equal(kb[:40], kp[1])
    assert torch.count_nonzero(kb[40:]) == 0
    wa.wa_check()   # the status word was cleared


def test_gather_host_pinned_tier():
    kp = synth.normal((7, 300, 4, 128), 15, dtype=torch.bfloat16).pin_memory()
    vp = synth.normal((7, 300, 4, 128), 16, dtype=torch.bfloat16).pin_memory()
    idx = [6, 2, 3]
    idx_h = torch.tensor(idx, dtype=torch.int32)
    kb = torch.empty((900, 4, 128), dtype=torch.bfloat16, device=DEV)
    vb = torch.empty_like(kb)
    wa.wa_gather_pages(kp, vp, None, idx_h, kb, vb)
    wa.wa_check()
    assert np.array_equal(np_of(kb), O.gather_pages(np_of(kp), idx))
    assert np.array_equal(np_of(vb), O.gather_pages(np_of(vp), idx))
    with pytest.raises(wa.WaError) as e:
        wa.wa_gather_pages(kp, vp, None, torch.tensor([0, 7, 1], dtype=torch.int32), kb, vb)
    assert e.value.status == 5
    # device indices: the kernel reads the pinned pages over the CPU-GPU link
    kb2, vb2 = torch.zeros_like(kb), torch.zeros_like(vb)
    wa.wa_gather_pages(kp, vp, torch.tensor(idx, dtype=torch.int32, device=DEV), None, kb2, vb2)
    wa.wa_check()
    assert torch.equal(kb2, kb) and torch.equal(vb2, vb)
