"""The workloads end to end on the GPU, each as one chain of C-ABI calls,
against the fp64 oracle at the shapes the workloads name.

* Tiny fp32 workload (1 head, d_k = 64, 16-token frames, 2-frame pages, 8 pages
  in 2 chunks, prompts of dim 32, K_p = 2, a 1-frame query chunk + its local
  KV): summaries -> two-stage retrieval -> gather -> fp32 attention, within
  1e-5; with K_p = all pages (no prompt stage) the chain must equal dense
  attention over [all pages ascending ; local].  WorldAttention review page,
  HKV section (two-stage retrieval, K_p) and "How It Works" step 3.
* The one-layer WorldAttention chunk exactly as the benchmark draws it (no
  planted pages): chunk pick, page indices and gathered bytes bit-exact,
  attention on sampled rows within the bf16 tolerance.
* The minute-long stress workload at full size: 30 layers, top-4 of 120 pages
  of 12,480 tokens whose bodies sit in pinned host memory, fetched by the
  double-buffered side-stream pipeline; every layer's indices and every
  layer's gathered buffer (as the attention read it) bit-exact, attention on
  sampled rows of three layers.  WorldAttention review page, HKV tiers L1/L2
  (Fig. 2); Inferix summary page, KV Cache Manager (offloading to main memory).
"""

import numpy as np
import pytest
import torch

import oracle as O
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
from sparse_kv_cache_page_gb300.tiered import TieredPipeline, TierLayer
from tests._util import (LSE_ABS, assert_attn_close, assert_selection_margin, f64,
                         mean_error_bound, np_of, page_mean_error_bounds, score_error_bound)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _chain(c, k_p, use_prompt, o_dtype=torch.float32, fused=False):
    """summarize -> select -> gather -> attention through the C ABI (with
    `fused`, the gather and the attention as one launch, as benchmarked)."""
    H, d = c.n_heads, c.head_dim
    kp, vp, q = c.k_pages.to(DEV), c.v_pages.to(DEV), c.q.to(DEV)
    kbar = torch.empty((c.n_pages, H, d), dtype=torch.float32, device=DEV)
    wa.wa_page_summarize(kp, kbar)
    idx = torch.full((k_p,), -1, dtype=torch.int32, device=DEV)
    sc = torch.empty(k_p, dtype=torch.float32, device=DEV)
    ch = torch.full((1,), -9, dtype=torch.int32, device=DEV)
    pc = c.prompt_chunks.to(DEV) if use_prompt else None
    cur = c.prompt_cur.to(DEV) if use_prompt else None
    wa.wa_select_pages(q, kbar, cur, pc, c.pages_per_chunk, k_p, idx, sc, ch)
    kb = torch.empty((k_p * c.page_tokens, H, d), dtype=c.dtype, device=DEV)
    vb = torch.empty_like(kb)
    o = torch.empty(q.shape, dtype=o_dtype, device=DEV)
    lse = torch.empty((H, c.n_q), dtype=torch.float32, device=DEV)
    if fused:
        wa.wa_gather_attn(q, kp, vp, idx, c.k_loc.to(DEV), c.v_loc.to(DEV), o, kb, vb, lse)
    else:
        wa.wa_gather_pages(kp, vp, idx, None, kb, vb)
        wa.wa_block_attn(q, kb, vb, c.k_loc.to(DEV), c.v_loc.to(DEV), o, lse)
    wa.wa_check()
    return dict(kbar=kbar, idx=idx.cpu().numpy(), sc=sc.cpu().numpy(), chunk=int(ch.item()),
                kb=kb, vb=vb, o=o, lse=lse)


@pytest.mark.parametrize("recall", [0, 1])
@pytest.mark.parametrize("peaked", [False, True])
def test_tiny_fp32_chain(recall, peaked):
    """The tiny fp32 workload as one chain, K_p = 2 after the prompt stage."""
    c = synth.tiny_fp32_case(recall_chunk=recall)
    if peaked:
        # each query points at one key of the recalled chunk's pages, so the
        # softmax rows are far from uniform and attention errors show
        own = c.k_pages[recall * c.pages_per_chunk:(recall + 1) * c.pages_per_chunk]
        c.q, _ = synth.peaked_queries(own.reshape(-1, 1, c.head_dim), c.n_q,
                                      synth.seed_of("tiny_peak", recall), gain=4.0)
    g = _chain(c, c.k_p, True)
    okp, ovp, oq = np_of(c.k_pages), np_of(c.v_pages), np_of(c.q)
    kbar = O.page_summarize(okp)
    idx, sc, ch = O.select_pages(oq, kbar, np_of(c.prompt_cur), np_of(c.prompt_chunks),
                                 c.pages_per_chunk, c.k_p)
    cand = O.candidate_pages(c.n_pages, ch, c.pages_per_chunk)
    qbar = O.mean_query(oq)
    bound = score_error_bound(mean_error_bound(O.as_f64(oq)), page_mean_error_bounds(okp), qbar,
                              kbar, c.head_dim)
    assert_selection_margin(O.page_scores(qbar, kbar, cand, c.head_dim), cand, c.k_p, bound)
    assert g["chunk"] == ch == recall
    assert g["idx"].tolist() == idx.tolist()
    assert np.abs(f64(g["kbar"]) - kbar).max() <= 1e-6
    assert np.abs(g["sc"] - sc).max() <= 1e-6
    kbuf, vbuf = O.gather_pages(okp, idx), O.gather_pages(ovp, idx)
    assert np.array_equal(np_of(g["kb"]), kbuf) and np.array_equal(np_of(g["vb"]), vbuf)
    ref, ref_lse = O.block_attn(oq, kbuf, vbuf, np_of(c.k_loc), np_of(c.v_loc))
    assert_attn_close(g["o"], ref, torch.float32, "tiny chain")
    assert np.abs(f64(g["lse"]) - ref_lse).max() <= 1e-5


@pytest.mark.parametrize("peaked", [False, True])
def test_tiny_fp32_all_pages_equals_dense(peaked):
    """K_p = all 8 pages (prompt stage bypassed): the chain selects every page
    in ascending order, and its attention equals dense attention over
    [all pages ascending ; local] computed by the oracle without retrieval."""
    c = synth.tiny_fp32_case()
    if peaked:
        c.q, _ = synth.peaked_queries(c.k_pages.reshape(-1, 1, c.head_dim), c.n_q,
                                      synth.seed_of("tiny_peak_all"), gain=4.0)
    g = _chain(c, c.n_pages, False)
    assert g["chunk"] == -1
    assert g["idx"].tolist() == list(range(c.n_pages))
    okp, ovp = np_of(c.k_pages), np_of(c.v_pages)
    H, d = c.n_heads, c.head_dim
    dense_k = okp.reshape(c.n_pages * c.page_tokens, H, d)
    dense_v = ovp.reshape(c.n_pages * c.page_tokens, H, d)
    assert np.array_equal(np_of(g["kb"]), dense_k) and np.array_equal(np_of(g["vb"]), dense_v)
    ref, ref_lse = O.block_attn(np_of(c.q), dense_k, dense_v, np_of(c.k_loc), np_of(c.v_loc))
    assert_attn_close(g["o"], ref, torch.float32, "all pages vs dense")
    assert np.abs(f64(g["lse"]) - ref_lse).max() <= 1e-5


def test_headline_chunk_as_benchmarked():
    """The benchmark's one-layer chunk, unplanted: 40 pages of 12,480 tokens
    in 5 chunks, the current prompt recalling chunk 3, top-4 of its 8 pages;
    the gather and the attention in one launch, as the benchmark runs them."""
    c = synth.worldattention_case(device=DEV, recall_chunk=3)
    g = _chain(c, c.k_p, True, o_dtype=torch.float32, fused=True)
    okp, oq = np_of(c.k_pages), np_of(c.q)
    kbar = O.page_summarize(okp)
    assert np.abs(f64(g["kbar"]) - kbar).max() < 1e-6
    idx, sc, ch = O.select_pages(oq, kbar, np_of(c.prompt_cur), np_of(c.prompt_chunks),
                                 c.pages_per_chunk, c.k_p)
    cand = O.candidate_pages(c.n_pages, ch, c.pages_per_chunk)
    alpha = O.page_scores(O.mean_query(oq), kbar, cand, c.head_dim)
    bound = score_error_bound(mean_error_bound(O.as_f64(oq)), page_mean_error_bounds(okp),
                              O.mean_query(oq), kbar, c.head_dim)
    assert_selection_margin(np.array(alpha), cand, c.k_p, bound)
    assert g["chunk"] == ch == 3
    assert g["idx"].tolist() == idx.tolist()
    assert np.abs(g["sc"] - sc).max() < 1e-6
    kbuf = O.gather_pages(okp, idx)
    vbuf = O.gather_pages(np_of(c.v_pages), idx)
    assert np.array_equal(np_of(g["kb"]), kbuf) and np.array_equal(np_of(g["vb"]), vbuf)
    rows = np.array([0, 1, 127, 128, 2047, 2303, 4095, 4607, 4608, 4679])
    ref, ref_lse = O.block_attn(oq, kbuf, vbuf, np_of(c.k_loc), np_of(c.v_loc), rows=rows)
    rt = torch.from_numpy(rows).to(DEV)
    assert_attn_close(g["o"][rt], ref, torch.bfloat16, "headline chunk")
    assert np.abs(f64(g["lse"][:, rt]) - ref_lse).max() <= LSE_ABS


def test_stress_workload_full_size_every_layer():
    """30 layers, top-4 of 120 pinned-host pages each, through the layer
    pipeline that the benchmark times (copy-engine fetches on a side stream,
    double-buffered, overlapped with the previous layer's attention)."""
    NPG, NL, P, H, D = synth.STRESS_PAGES, synth.STRESS_LAYERS, synth.PAGE_TOKENS, 12, 128
    NQ = NLOC = 3 * synth.TOKENS_PER_FRAME
    hk = torch.empty((NPG, P, H, D), dtype=torch.bfloat16, pin_memory=True)
    hv = torch.empty((NPG, P, H, D), dtype=torch.bfloat16, pin_memory=True)
    kbar = torch.empty((NPG, H, D), dtype=torch.float32, device=DEV)
    for j in range(NPG):
        kj, vj = synth.stress_page(j, DEV)
        wa.wa_page_summarize(kj[None], kbar[j:j + 1])
        hk[j].copy_(kj)
        hv[j].copy_(vj)
    torch.cuda.synchronize()
    wa.wa_check()
    okp, ovp = np_of(hk), np_of(hv)          # views of the pinned store, no copy
    ref_kbar = np.empty((NPG, H, D))
    dk = np.empty((NPG, H, D))
    for j in range(NPG):
        ref_kbar[j] = O.page_summarize(okp[j:j + 1])[0]
        dk[j] = mean_error_bound(O.as_f64(okp[j]))
    assert np.abs(f64(kbar) - ref_kbar).max() < 1e-6

    layers, ref_idx = [], []
    for l in range(NL):
        q, kl, vl = synth.stress_layer(l, DEV)
        out = torch.empty((NQ, H, D), dtype=torch.float32, device=DEV)
        layers.append(TierLayer(q, kl, vl, kbar, hk, hv, out))
        oq = np_of(q)
        idx, _, ch = O.select_pages(oq, ref_kbar, None, None, 1, 4)
        assert ch == -1
        qbar = O.mean_query(oq)
        alpha = O.page_scores(qbar, ref_kbar, range(NPG), D)
        bound = score_error_bound(mean_error_bound(O.as_f64(oq)), dk, qbar, ref_kbar, D)
        assert_selection_margin(alpha, range(NPG), 4, bound)
        ref_idx.append(idx)

    # the oracle's gathered buffers of every layer, compared on the device with
    # the buffers the pipeline's attention read, without holding the pipeline
    expect = [(torch.from_numpy(O.gather_pages(okp, ix).view(np.int16)).to(DEV),
               torch.from_numpy(O.gather_pages(ovp, ix).view(np.int16)).to(DEV))
              for ix in ref_idx]
    same = torch.zeros(NL, dtype=torch.int32, device=DEV)

    def on_layer(l, kb, vb):
        ek, ev = expect[l]
        same[l] = ((kb.view(torch.int16) == ek).all() & (vb.view(torch.int16) == ev).all()).int()

    pipe = TieredPipeline(4, P, H, D)
    idx_h = pipe.run(layers, "pipeline", on_layer=on_layer)
    torch.cuda.synchronize()
    wa.wa_check()
    got = [idx_h[l].tolist() for l in range(NL)]
    assert got == [ix.tolist() for ix in ref_idx]
    assert same.cpu().tolist() == [1] * NL
    del expect

    rows = np.array([0, 777, 2500, 4679])
    for l in (0, 15, NL - 1):
        ly = layers[l]
        ref, _ = O.block_attn(np_of(ly.q), O.gather_pages(okp, ref_idx[l]),
                              O.gather_pages(ovp, ref_idx[l]), np_of(ly.k_loc), np_of(ly.v_loc),
                              rows=rows)
        assert_attn_close(ly.out[torch.from_numpy(rows).to(DEV)], ref, torch.bfloat16,
                          f"stress layer {l}")
