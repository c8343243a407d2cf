"""GPU checks of the KV cache manager (libwa wa_cache_*): chunks appended
into a small HBM tier with the rest offloaded to pinned DRAM; retrieval picks
the oracle's pages (two-stage selection over the whole cached sequence) and
copies their bytes exactly from either tier; promoted and re-offloaded pages
keep their bytes; window access returns the sequence's last tokens."""

import numpy as np
import pytest
import torch

import oracle as O
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
from tests._util import np_of

pytestmark = pytest.mark.gpu
DEV = "cuda"
H, D, P, PPC, PDIM = 4, 128, 256, 4, 32


def _chunk(m, plant=None, u=None):
    s = lambda t: synth.seed_of("cache", m, t)  # noqa: E731
    k = synth.normal((PPC * P, H, D), s("k"), DEV)
    v = synth.normal((PPC * P, H, D), s("v"), DEV, torch.bfloat16)
    if plant is not None:
        for j in plant:
            k[j * P:(j + 1) * P] += u
    return k.to(torch.bfloat16), v, synth.normal((PDIM,), s("prompt"), DEV)


def _setup(n_chunks=5, hbm=6, host=24):
    u = synth.normal((H, D), synth.seed_of("cache", "dir"), DEV) * 0.6
    cache = wa.WaCache(H, D, P, PPC, hbm_pages=hbm, host_pages=host, max_chunks=8, prompt_dim=PDIM)
    ks, vs, ps = [], [], []
    for m in range(n_chunks):
        k, v, pr = _chunk(m, plant=(1, 3) if m == 2 else None, u=u)
        cache.append(k, v, pr)
        ks.append(k)
        vs.append(v)
        ps.append(pr)
    wa.wa_check()
    q = (synth.normal((200, H, D), synth.seed_of("cache", "q"), DEV) + u).to(torch.bfloat16)
    cur = ps[2] + 0.5 * synth.normal((PDIM,), synth.seed_of("cache", "cur"), DEV)
    return cache, ks, vs, ps, q, cur


def _bank(ts):
    return torch.cat(ts).reshape(-1, P, H, D)


def test_retrieve_from_both_tiers_and_promote():
    cache, ks, vs, ps, q, cur = _setup()
    st0 = cache.stats()
    assert st0["n_pages"] == 20 and st0["in_hbm"] == 6 and st0["offloads"] == 14
    kb = torch.empty((2 * P, H, D), dtype=torch.bfloat16, device=DEV)
    vb = torch.empty_like(kb)
    idx = cache.retrieve(q, cur, 2, kb, vb)
    wa.wa_check()
    kbank, vbank = _bank(ks), _bank(vs)
    kbar = O.page_summarize(np_of(kbank))
    ref_idx, _, ref_chunk = O.select_pages(np_of(q), kbar, np_of(cur), np_of(torch.stack(ps)), PPC, 2)
    assert ref_chunk == 2 and idx == ref_idx.tolist() == [9, 11]
    assert np.array_equal(np_of(kb), O.gather_pages(np_of(kbank), idx))
    assert np.array_equal(np_of(vb), O.gather_pages(np_of(vbank), idx))
    # both pages lived in DRAM (chunk 2 is old): now promoted
    st1 = cache.stats()
    assert st1["promotions"] == 2 and all(cache.location(p)[0] == 0 for p in idx)
    # more appends push them out again; a later retrieval still returns their bytes
    for m in (5, 6):
        k, v, pr = _chunk(m)
        cache.append(k, v, pr)
        ks.append(k)
        vs.append(v)
        ps.append(pr)
    assert cache.location(9)[0] == 1
    idx2 = cache.retrieve(q, cur, 2, kb, vb)
    wa.wa_check()
    kbank, vbank = _bank(ks), _bank(vs)
    assert idx2 == [9, 11]
    assert np.array_equal(np_of(kb), O.gather_pages(np_of(kbank), idx2))
    assert np.array_equal(np_of(vb), O.gather_pages(np_of(vbank), idx2))
    cache.close()


def test_retrieve_without_prompt_stage():
    cache, ks, vs, ps, q, cur = _setup(n_chunks=4, hbm=5, host=16)
    kb = torch.empty((3 * P, H, D), dtype=torch.bfloat16, device=DEV)
    vb = torch.empty_like(kb)
    idx = cache.retrieve(q, None, 3, kb, vb)
    wa.wa_check()
    kbank = _bank(ks)
    ref_idx, _, ch = O.select_pages(np_of(q), O.page_summarize(np_of(kbank)), None, None, PPC, 3)
    assert ch == -1 and idx == ref_idx.tolist()
    assert 9 in idx and 11 in idx
    assert np.array_equal(np_of(kb), O.gather_pages(np_of(kbank), idx))
    cache.close()


@pytest.mark.parametrize("n_tok", [600, 256, 1, 20 * P])
def test_window(n_tok):
    cache, ks, vs, _, _, _ = _setup()
    ko = torch.empty((n_tok, H, D), dtype=torch.bfloat16, device=DEV)
    vo = torch.empty_like(ko)
    cache.window(n_tok, ko, vo)
    wa.wa_check()
    assert torch.equal(ko, torch.cat(ks)[-n_tok:]) and torch.equal(vo, torch.cat(vs)[-n_tok:])
    cache.close()
