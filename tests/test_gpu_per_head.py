"""GPU parity of per-head page sets (the per-head variant of the page stage)
through the C ABI against the fp64 oracle: per-head top-K_p indices bit-exact
(with a margin check that no head's boundary is a tie within fp32 rounding),
the per-head gather byte-exact (and its bad-index path), and attention over the
per-head buffer, on small cases and at the one-layer WorldAttention shape."""

import numpy as np
import pytest
import torch

import oracle as O
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
from tests._util import (assert_attn_close, f64, mean_error_bound, np_of, page_mean_error_bounds,
                         score_error_bound)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _plant_per_head(c, seed, strength, chunk):
    """Head h: k_p pages of the recalled chunk share a direction with the
    head's queries, at falling strengths and different pages for different
    heads, so each head's top-k_p set is clear of rounding."""
    kp, q = c.k_pages.float(), c.q.float()
    ppc = c.pages_per_chunk
    for h in range(c.n_heads):
        u = synth.normal((c.head_dim,), synth.seed_of("perhead", seed, h)).to(kp.device)
        for r in range(c.k_p):
            j = chunk * ppc + (3 * h + 5 * r) % ppc
            kp[j, :, h, :] += strength * (1.0 - 0.1 * r) * u
        q[:, h, :] += strength * u
    c.k_pages, c.q = kp.to(c.dtype), q.to(c.dtype)
    return c


def _case(seed, H=6, P=256, n_pages=16, ppc=8, k_p=3, strength=0.5):
    c = synth.make_chunk_case(f"perhead{seed}", n_heads=H, head_dim=128, page_tokens=P,
                              n_pages=n_pages, pages_per_chunk=ppc, n_chunks=n_pages // ppc,
                              prompt_dim=64, k_p=k_p, n_q=300, n_loc=100, recall_chunk=1)
    return _plant_per_head(c, seed, strength, 1)


def _gpu_select(c, kbar):
    idx = torch.full((c.n_heads, c.k_p), -7, dtype=torch.int32, device=DEV)
    sc = torch.empty((c.n_heads, c.k_p), dtype=torch.float32, device=DEV)
    ch = torch.full((1,), -9, dtype=torch.int32, device=DEV)
    wa.wa_select_pages_per_head(c.q.to(DEV), kbar, c.prompt_cur.to(DEV), c.prompt_chunks.to(DEV),
                                c.pages_per_chunk, c.k_p, idx, sc, ch)
    wa.wa_check()
    return idx, sc.cpu().numpy(), int(ch.item())


def _check_margins(q, k_pages, kbar64, chunk, ppc, k_p):
    """Each head's gap between its k_p-th and (k_p+1)-th candidate must exceed
    the probabilistic fp32 rounding bound of both scores (the retrieval tests'
    bound, applied to the head's slice); else the case is a tie within
    rounding and the seed must change."""
    q64 = O.as_f64(q)
    cand = O.candidate_pages(kbar64.shape[0], chunk, ppc)
    qbar = O.mean_query(q)
    a = O.page_scores_per_head(qbar, kbar64, cand, kbar64.shape[2])
    dq = mean_error_bound(q64)
    dk = page_mean_error_bounds(k_pages)
    for h in range(a.shape[0]):
        bound = score_error_bound(dq[h:h + 1], dk[:, h:h + 1], qbar[h:h + 1],
                                  kbar64[:, h:h + 1], kbar64.shape[2])
        order = sorted(range(len(cand)), key=lambda i: (-a[h][i], cand[i]))
        if k_p < len(order):
            i0, i1 = order[k_p - 1], order[k_p]
            gap = a[h][i0] - a[h][i1]
            assert gap > bound[cand[i0]] + bound[cand[i1]], \
                f"head {h}: tie within rounding ({gap:.3e}); change the seed"


@pytest.mark.parametrize("seed", [1, 2])
def test_per_head_select_small(seed):
    c = _case(seed)
    kbar = torch.empty((c.n_pages, c.n_heads, 128), dtype=torch.float32, device=DEV)
    wa.wa_page_summarize(c.k_pages.to(DEV), kbar)
    idx, sc, ch = _gpu_select(c, kbar)
    kb64 = O.page_summarize(np_of(c.k_pages))
    ref_idx, ref_sc, ref_ch = O.select_pages_per_head(np_of(c.q), kb64, np_of(c.prompt_cur),
                                                      np_of(c.prompt_chunks), c.pages_per_chunk,
                                                      c.k_p)
    _check_margins(np_of(c.q), np_of(c.k_pages), kb64, ref_ch, c.pages_per_chunk, c.k_p)
    assert ch == ref_ch == 1
    assert idx.cpu().numpy().tolist() == ref_idx.tolist()
    assert np.abs(sc - ref_sc).max() < 1e-5
    assert len({tuple(r) for r in ref_idx.tolist()}) > 1     # heads chose different sets


@pytest.mark.parametrize("n_pages,k_p", [(32, 1), (32, 5), (32, 31), (32, 32), (33, 5), (64, 16)])
def test_per_head_select_no_prompt(n_pages, k_p):
    """No prompt stage: every page is a candidate.  Up to 32 candidates are
    scored and sorted by one warp per head (the boundary case 32 included, with
    k_p up to all of them); 33 and more take the block-wide path.  Indices
    bit-exact and scores against the oracle on both paths."""
    c = synth.make_chunk_case("phnp1", n_heads=5, head_dim=64, page_tokens=32, n_pages=n_pages,
                              pages_per_chunk=1, n_chunks=0, prompt_dim=0, k_p=k_p, n_q=64,
                              n_loc=1, dtype=torch.bfloat16)
    kbar = torch.empty((n_pages, c.n_heads, 64), dtype=torch.float32, device=DEV)
    wa.wa_page_summarize(c.k_pages.to(DEV), kbar)
    idx = torch.full((c.n_heads, k_p), -7, dtype=torch.int32, device=DEV)
    sc = torch.empty((c.n_heads, k_p), dtype=torch.float32, device=DEV)
    ch = torch.full((1,), -9, dtype=torch.int32, device=DEV)
    wa.wa_select_pages_per_head(c.q.to(DEV), kbar, None, None, 1, k_p, idx, sc, ch)
    wa.wa_check()
    kb64 = O.page_summarize(np_of(c.k_pages))
    ref_idx, ref_sc, ref_ch = O.select_pages_per_head(np_of(c.q), kb64, None, None, 1, k_p)
    _check_margins(np_of(c.q), np_of(c.k_pages), kb64, ref_ch, 1, k_p)
    assert int(ch.item()) == ref_ch == -1
    assert idx.cpu().numpy().tolist() == ref_idx.tolist()
    assert np.abs(sc.cpu().numpy() - ref_sc).max() < 1e-5


def test_per_head_gather_and_attention():
    c = _case(3)
    idx = torch.tensor(O.select_pages_per_head(np_of(c.q), O.page_summarize(np_of(c.k_pages)),
                                               np_of(c.prompt_cur), np_of(c.prompt_chunks),
                                               c.pages_per_chunk, c.k_p)[0], device=DEV)
    kb = torch.empty((c.k_p * c.page_tokens, c.n_heads, 128), dtype=torch.bfloat16, device=DEV)
    vb = torch.empty_like(kb)
    wa.wa_gather_pages_per_head(c.k_pages.to(DEV), c.v_pages.to(DEV), idx, kb, vb)
    wa.wa_check()
    ref_k = O.gather_pages_per_head(np_of(c.k_pages), idx.cpu().numpy())
    ref_v = O.gather_pages_per_head(np_of(c.v_pages), idx.cpu().numpy())
    assert np.array_equal(np_of(kb), ref_k) and np.array_equal(np_of(vb), ref_v)
    o = torch.empty(c.q.shape, dtype=torch.float32, device=DEV)
    wa.wa_block_attn(c.q.to(DEV), kb, vb, c.k_loc.to(DEV), c.v_loc.to(DEV), o)
    wa.wa_check()
    ref, _ = O.block_attn(np_of(c.q), ref_k, ref_v, np_of(c.k_loc), np_of(c.v_loc))
    assert_attn_close(o, ref, torch.bfloat16, "per-head buffer")


def test_per_head_gather_bad_index_reported():
    kp = synth.normal((3, 40, 2, 128), 21, dtype=torch.bfloat16).to(DEV)
    idx = torch.tensor([[1, 2], [0, 3]], dtype=torch.int32, device=DEV)   # head 1, slot 1: bad
    kb = torch.full((80, 2, 128), 5.0, dtype=torch.bfloat16, device=DEV)
    wa.wa_gather_pages_per_head(kp, None, idx, kb, None)
    with pytest.raises(wa.WaError) as e:
        wa.wa_check()
    assert e.value.status == 5
    assert torch.equal(kb[:40, 0], kp[1, :, 0]) and torch.equal(kb[40:, 0], kp[2, :, 0])
    assert torch.equal(kb[:40, 1], kp[0, :, 1])
    assert torch.count_nonzero(kb[40:, 1]) == 0
    wa.wa_check()


def test_per_head_worldattention_shape():
    """One layer at the WorldAttention shape (40 pages x 12,480 tokens, 12
    heads, top-4 of the recalled chunk's 8 pages per head): indices, the
    gathered buffer on sampled token rows, attention on sampled query rows."""
    c = synth.worldattention_case(device=DEV, recall_chunk=3)
    c = _plant_per_head(c, 7, 0.25, 3)
    kbar = torch.empty((c.n_pages, c.n_heads, 128), dtype=torch.float32, device=DEV)
    wa.wa_page_summarize(c.k_pages, kbar)
    idx, _, ch = _gpu_select(c, kbar)
    kb64 = O.page_summarize(np_of(c.k_pages))
    ref_idx, _, ref_ch = O.select_pages_per_head(np_of(c.q), kb64, np_of(c.prompt_cur),
                                                 np_of(c.prompt_chunks), c.pages_per_chunk, c.k_p)
    _check_margins(np_of(c.q), kp_np := np_of(c.k_pages), kb64, ref_ch, c.pages_per_chunk, c.k_p)
    assert ch == ref_ch == 3 and idx.cpu().numpy().tolist() == ref_idx.tolist()
    P = c.page_tokens
    kb = torch.empty((c.k_p * P, c.n_heads, 128), dtype=torch.bfloat16, device=DEV)
    vb = torch.empty_like(kb)
    wa.wa_gather_pages_per_head(c.k_pages, c.v_pages, idx, kb, vb)
    wa.wa_check()
    vp_np = np_of(c.v_pages)
    rows = np.random.default_rng(7).choice(c.k_p * P, 64, replace=False)
    kb_np, vb_np = np_of(kb), np_of(vb)
    for r in rows:
        s_, t = divmod(int(r), P)
        for h in range(c.n_heads):
            assert np.array_equal(kb_np[r, h], kp_np[ref_idx[h, s_], t, h])
            assert np.array_equal(vb_np[r, h], vp_np[ref_idx[h, s_], t, h])
    o = torch.empty(c.q.shape, dtype=torch.float32, device=DEV)
    wa.wa_block_attn(c.q, kb, vb, c.k_loc, c.v_loc, o)
    wa.wa_check()
    qrows = np.random.default_rng(8).choice(c.n_q, 24, replace=False)
    ref, _ = O.block_attn(np_of(c.q), kb_np, vb_np, np_of(c.k_loc), np_of(c.v_loc), rows=qrows)
    assert_attn_close(o[torch.as_tensor(qrows, device=DEV)], ref, torch.bfloat16, "sampled rows")
