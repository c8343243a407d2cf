"""GPU checks of the KV cache manager (libwa wa_cache_*): chunks appended
into a small HBM tier with the rest offloaded to pinned DRAM (on the cache's
own copy stream, overlapping later calls); retrieval picks the oracle's pages
(two-stage selection over the whole cached sequence) and copies their bytes
exactly from either tier; promoted and re-evicted pages keep their bytes;
window access returns the sequence's last tokens.  With a compressed DRAM
tier (FP8 or NVFP4) a page that has been offloaded reads back as the oracle
codec's decode(encode(page)), bit for bit, from either tier."""

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


def _setup(n_chunks=5, hbm=6, host=24, fmt="native"):
    u = synth.normal((H, D), synth.seed_of("cache", "dir"), DEV) * 0.6
    cache = wa.WaCache(H, D, P, PPC, hbm_pages=hbm, host_pages=host, max_chunks=8, prompt_dim=PDIM,
                       dram_format=fmt)
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


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _expected(cache, ts, fmt):
    """bf16 bits of every cached page as a read should return it: the page
    itself, or (compressed tier) decode(encode(page)) once it has a DRAM copy.
    Valid while no DRAM copy has been reclaimed."""
    assert cache.stats()["reclaims"] == 0
    bank = _bank(ts)
    out = _bits(bank).copy()
    if fmt != "native":
        for p in range(bank.shape[0]):
            if cache.slots(p)[1] >= 0:
                x = np_of(bank[p])
                dec = (O.fp8_decode_rows(*O.fp8_encode_rows(x)) if fmt == "fp8"
                       else O.nvfp4_decode_rows(*O.nvfp4_encode_rows(x)))
                out[p] = O.bf16_bits(dec)
    return out


@pytest.mark.parametrize("fmt", ["native", "fp8", "nvfp4"])
def test_retrieve_from_both_tiers_and_promote(fmt):
    cache, ks, vs, ps, q, cur = _setup(fmt=fmt)
    st0 = cache.stats()
    assert st0["n_pages"] == 20 and st0["in_hbm"] == 6 and st0["offloads"] == 14
    kb = torch.empty((2 * P, H, D), dtype=torch.bfloat16, device=DEV)
    vb = torch.empty_like(kb)
    idx = cache.retrieve(q, cur, 2, kb, vb)
    wa.wa_check()
    kbank = _bank(ks)
    kbar = O.page_summarize(np_of(kbank))
    ref_idx, _, ref_chunk = O.select_pages(np_of(q), kbar, np_of(cur), np_of(torch.stack(ps)), PPC, 2)
    assert ref_chunk == 2 and idx == ref_idx.tolist() == [9, 11]
    ek, ev = _expected(cache, ks, fmt), _expected(cache, vs, fmt)
    assert np.array_equal(_bits(kb), np.concatenate([ek[i] for i in idx]))
    assert np.array_equal(_bits(vb), np.concatenate([ev[i] for i in idx]))
    # both pages lived in DRAM (chunk 2 is old): now promoted, DRAM copies kept
    st1 = cache.stats()
    assert st1["promotions"] == 2 and all(cache.location(p)[0] == 0 for p in idx)
    assert all(cache.slots(p)[1] >= 0 for p in idx)
    # more appends push them out again (no copy: DRAM already holds them); a later
    # retrieval still returns the same bytes
    for m in (5, 6):
        k, v, pr = _chunk(m)
        cache.append(k, v, pr)
        ks.append(k)
        vs.append(v)
        ps.append(pr)
    assert cache.location(9)[0] == 1 and cache.stats()["evictions"] >= 2
    idx2 = cache.retrieve(q, cur, 2, kb, vb)
    wa.wa_check()
    assert idx2 == [9, 11]
    ek, ev = _expected(cache, ks, fmt), _expected(cache, vs, fmt)
    assert np.array_equal(_bits(kb), np.concatenate([ek[i] for i in idx2]))
    assert np.array_equal(_bits(vb), np.concatenate([ev[i] for i in idx2]))
    cache.close()


@pytest.mark.parametrize("fmt", ["native", "fp8", "nvfp4"])
def test_offloads_in_flight_are_waited_for(fmt):
    """Ten chunks appended back to back into an HBM tier of one chunk (every
    append offloads the previous chunk, 36 offloads through a staging ring of
    8 pages), then, with no synchronisation, a retrieval of the planted pages
    of chunk 8 -- offloaded by the last append, their copies possibly still in
    flight -- and a window over the whole sequence."""
    u = synth.normal((H, D), synth.seed_of("cache", "dir"), DEV) * 0.6
    cache = wa.WaCache(H, D, P, PPC, hbm_pages=PPC, host_pages=40, max_chunks=10,
                       prompt_dim=PDIM, dram_format=fmt)
    ks, vs, ps = [], [], []
    for m in range(10):
        k, v, pr = _chunk(m, plant=(0, 2) if m == 8 else None, u=u)
        cache.append(k, v, pr)
        ks.append(k)
        vs.append(v)
        ps.append(pr)
    q = (synth.normal((200, H, D), synth.seed_of("cache", "q"), DEV) + u).to(torch.bfloat16)
    cur = ps[8] + 0.5 * synth.normal((PDIM,), synth.seed_of("cache", "cur"), DEV)
    kb = torch.empty((2 * P, H, D), dtype=torch.bfloat16, device=DEV)
    vb = torch.empty_like(kb)
    idx = cache.retrieve(q, cur, 2, kb, vb)
    ko = torch.empty((40 * P, H, D), dtype=torch.bfloat16, device=DEV)
    vo = torch.empty_like(ko)
    cache.window(40 * P, ko, vo)
    cache.wait_copies()
    wa.wa_check()
    st = cache.stats()
    # 36 by the appends, 2 by the promotion of pages 32 and 34 (chunk 9's 36, 37)
    assert st["offloads"] == 38 and st["reclaims"] == 0
    assert idx == [32, 34]
    ek, ev = _expected(cache, ks, fmt), _expected(cache, vs, fmt)
    assert np.array_equal(_bits(kb), np.concatenate([ek[i] for i in idx]))
    assert np.array_equal(_bits(vb), np.concatenate([ev[i] for i in idx]))
    assert np.array_equal(_bits(ko), ek.reshape(40 * P, H, D))
    assert np.array_equal(_bits(vo), ev.reshape(40 * P, H, D))
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


@pytest.mark.parametrize("fmt", ["native", "fp8", "nvfp4"])
@pytest.mark.parametrize("n_tok", [600, 256, 1, 17 * P + 100, 20 * P])
def test_window(n_tok, fmt):
    cache, ks, vs, _, _, _ = _setup(fmt=fmt)
    ko = torch.empty((n_tok, H, D), dtype=torch.bfloat16, device=DEV)
    vo = torch.empty_like(ko)
    cache.window(n_tok, ko, vo)
    wa.wa_check()
    ek = _expected(cache, ks, fmt).reshape(-1, H, D)
    ev = _expected(cache, vs, fmt).reshape(-1, H, D)
    assert np.array_equal(_bits(ko), ek[-n_tok:]) and np.array_equal(_bits(vo), ev[-n_tok:])
    cache.close()


@pytest.mark.parametrize("fmt", ["native", "fp8", "nvfp4"])
def test_full_size_pages(fmt):
    """Pages at the workload's full size (12,480 tokens x 12 heads x 128): three
    chunks of 4 pages through a 4-page HBM tier, then a retrieval whose prompt
    recalls the offloaded first chunk; the selection equals the oracle's and a
    sample of 400 token rows of both retrieved pages (K and V) reads back as the
    page, or the oracle codec's round trip of it."""
    P, H, D, PPC, PDIM = 12480, 12, 128, 4, 64
    u = synth.normal((H, D), synth.seed_of("cachefull", "dir"), DEV) * 0.6
    cache = wa.WaCache(H, D, P, PPC, hbm_pages=PPC, host_pages=12, max_chunks=3, prompt_dim=PDIM,
                       dram_format=fmt)
    ks, vs, ps = [], [], []
    for m in range(3):
        s = lambda t: synth.seed_of("cachefull", m, t)  # noqa: E731
        k = synth.normal((PPC * P, H, D), s("k"), DEV)
        if m == 0:
            for j in (1, 2):
                k[j * P:(j + 1) * P] += u
        k = k.to(torch.bfloat16)
        v = synth.normal((PPC * P, H, D), s("v"), DEV, torch.bfloat16)
        pr = synth.normal((PDIM,), s("prompt"), DEV)
        cache.append(k, v, pr)
        ks.append(k)
        vs.append(v)
        ps.append(pr)
    q = (synth.normal((512, H, D), synth.seed_of("cachefull", "q"), DEV) + u).to(torch.bfloat16)
    cur = ps[0] + 0.5 * synth.normal((PDIM,), synth.seed_of("cachefull", "cur"), DEV)
    kb = torch.empty((2 * P, H, D), dtype=torch.bfloat16, device=DEV)
    vb = torch.empty_like(kb)
    idx = cache.retrieve(q, cur, 2, kb, vb)
    cache.wait_copies()
    wa.wa_check()
    kbar = O.page_summarize(np_of(torch.cat(ks)).reshape(-1, P, H, D))
    ref_idx, _, ref_chunk = O.select_pages(np_of(q), kbar, np_of(cur), np_of(torch.stack(ps)),
                                           PPC, 2)
    assert ref_chunk == 0 and idx == ref_idx.tolist() == [1, 2]
    assert cache.stats()["promotions"] == 2
    rows = np.random.default_rng(8).integers(0, P, 400)
    for buf, src in ((kb, ks[0]), (vb, vs[0])):
        for slot, page in enumerate(idx):
            got = _bits(buf[torch.from_numpy(slot * P + rows).to(DEV)])
            x = np_of(src[torch.from_numpy(page * P + rows).to(DEV)])
            if fmt == "fp8":
                x = O.bf16_bits(O.fp8_decode_rows(*O.fp8_encode_rows(x)))
            elif fmt == "nvfp4":
                x = O.bf16_bits(O.nvfp4_decode_rows(*O.nvfp4_encode_rows(x)))
            assert np.array_equal(got, x), (fmt, page)
    cache.close()
