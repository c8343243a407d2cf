"""Host logic of the KV cache manager (libwa wa_cache_*), on CPU with dry-run
caches (no device memory, no CUDA calls): page placement across the HBM and
DRAM tiers under appends and retrievals, checked against a reference model
written here from the stated policy -- pages to free HBM slots (lowest slot
first); when HBM is full the least recently used resident page (ties: lower
page) leaves it, pages of the current append or retrieval never; a leaving
page with a DRAM copy moves nothing (the DRAM tier is inclusive: pages never
change once appended), one without is offloaded to the lowest free DRAM slot,
else to the slot of the most recently used page holding both copies (ties:
lower page), else, in a promotion, to the promoted page's own; a page used
from DRAM only is promoted back to HBM and keeps its DRAM copy; one clock
tick per append and per retrieval."""

import random

import pytest
import torch

import sparse_kv_cache_page_gb300 as wa


class Model:
    def __init__(self, hbm, host, ppc):
        self.hbm, self.host, self.ppc = [None] * hbm, [None] * host, ppc
        self.tab, self.clock, self.n = {}, 0, 0      # page -> [hbm slot, host slot, last use]
        self.off = self.pro = self.evi = self.rec = 0

    @staticmethod
    def _free(arr):
        return next((i for i, x in enumerate(arr) if x is None), None)

    def _host_slot(self, self_page):
        x = self._free(self.host)
        if x is not None:
            return x
        both = [p for p, (h, hx, _) in self.tab.items() if h is not None and hx is not None]
        w = min(both, key=lambda p: (-self.tab[p][2], p)) if both else None
        if w is None and self_page is not None and self.tab[self_page][1] is not None:
            w = self_page
        assert w is not None
        x = self.tab[w][1]
        self.tab[w][1], self.host[x] = None, None
        self.rec += 1
        return x

    def _hbm_slot(self, keep, self_page=None):
        s = self._free(self.hbm)
        if s is None:
            res = [p for p, (h, _, _) in self.tab.items() if h is not None and p not in keep]
            v = min(res, key=lambda p: (self.tab[p][2], p))
            s = self.tab[v][0]
            if self.tab[v][1] is not None:
                self.evi += 1
            else:
                x = self._host_slot(self_page)
                self.host[x], self.tab[v][1] = v, x
                self.off += 1
            self.hbm[s], self.tab[v][0] = None, None
        return s

    def append(self):
        self.clock += 1
        keep = set()
        for _ in range(self.ppc):
            p = self.n
            self.n += 1
            self.tab[p] = [None, None, self.clock]
            keep.add(p)
            s = self._hbm_slot(keep)
            self.hbm[s], self.tab[p][0] = p, s

    def touch(self, pages):
        self.clock += 1
        keep = set(pages)
        for p in pages:
            self.tab[p][2] = self.clock
            if self.tab[p][0] is None:
                s = self._hbm_slot(keep, self_page=p)
                self.hbm[s], self.tab[p][0] = p, s
                self.pro += 1

    def location(self, p):
        h, x, _ = self.tab[p]
        return (0, h) if h is not None else (1, x)

    def slots(self, p):
        h, x, _ = self.tab[p]
        return (-1 if h is None else h, -1 if x is None else x)


def _cache(hbm, host, ppc, max_chunks=64, page_tokens=16):
    return wa.WaCache(4, 64, page_tokens, ppc, hbm_pages=hbm, host_pages=host,
                      max_chunks=max_chunks, dry_run=True)


@pytest.mark.parametrize("hbm,host,ppc,seed", [(4, 8, 2, 1), (6, 20, 3, 2), (8, 8, 4, 3),
                                               (5, 30, 1, 4)])
def test_placement_matches_reference_model(hbm, host, ppc, seed):
    rng = random.Random(seed)
    c, m = _cache(hbm, host, ppc), Model(hbm, host, ppc)
    chunks = (hbm + host) // ppc
    for step in range(60):
        if m.n + ppc <= hbm + host and m.n // ppc < chunks and (m.n == 0 or rng.random() < 0.4):
            c.append(None, None)
            m.append()
        elif m.n > 0:
            k = rng.randint(1, min(hbm, m.n))
            pages = sorted(rng.sample(range(m.n), k))
            c.touch(pages)
            m.touch(pages)
        for p in range(m.n):
            assert c.location(p) == m.location(p), f"step {step}, page {p}"
            assert c.slots(p) == m.slots(p), f"step {step}, page {p}"
        st = c.stats()
        assert st["n_pages"] == m.n and st["offloads"] == m.off and st["promotions"] == m.pro
        assert st["evictions"] == m.evi and st["reclaims"] == m.rec
        assert st["in_hbm"] == sum(x is not None for x in m.hbm) <= hbm
        assert st["in_host"] == sum(x is not None for x in m.host) <= host
        # every page has at least one copy
        assert all(c.slots(p) != (-1, -1) for p in range(m.n))


@pytest.mark.parametrize("fmt", ["native", "fp8", "nvfp4"])
def test_bytes_planned(fmt):
    c = wa.WaCache(4, 64, 16, 2, hbm_pages=2, host_pages=4, max_chunks=64, dry_run=True,
                   dram_format=fmt)
    rows = 16 * 4                                           # (token, head) rows of a page
    page = rows * 64 * 2                                    # bf16 K (or V) of one page
    host_page = {"native": page,
                 "fp8": rows * 64 + rows * 4,               # FP8 codes + fp32 scales
                 "nvfp4": rows * 32 + rows * 4 + rows * 4}[fmt]   # E2M1 + E4M3 blocks + fp32
    c.append(None, None)
    c.append(None, None)            # pages 0, 1 offloaded
    c.touch([0])                    # page 0 back (keeps its DRAM copy), page 2 out
    st = c.stats()
    assert st["bytes_d2d"] == 4 * 2 * page + 2 * page    # appends + the promotion
    assert st["bytes_d2h"] == 3 * 2 * host_page          # three offloads
    assert (st["offloads"], st["promotions"], st["evictions"]) == (3, 1, 0)
    assert c.location(0) == (0, 0) and c.slots(0) == (0, 0) and c.location(2) == (1, 2)
    c.touch([2])                    # page 2 back, page 3 (HBM only) offloaded
    c.touch([3])                    # page 3 back, page 0 leaves HBM with no copy
    st = c.stats()
    assert (st["offloads"], st["promotions"], st["evictions"]) == (4, 3, 1)
    assert st["bytes_d2h"] == 4 * 2 * host_page
    assert c.slots(0) == (-1, 0) and c.slots(3) == (0, 3)
    assert (st["in_hbm"], st["in_host"]) == (2, 4)


def test_reclaim_and_own_slot_fallback():
    # DRAM full of DRAM-only pages: a promotion's victim takes the promoted page's slot
    c, m = _cache(2, 2, 1), Model(2, 2, 1)
    for _ in range(4):
        c.append(None, None)
        m.append()
    c.touch([0])
    m.touch([0])
    assert c.slots(0) == m.slots(0) == (0, -1) and c.slots(2) == m.slots(2) == (-1, 0)
    assert c.stats()["reclaims"] == 1
    # a spare DRAM slot makes a page with both copies, whose DRAM copy is reclaimed next
    c, m = _cache(3, 4, 1), Model(3, 4, 1)
    for _ in range(6):
        c.append(None, None)
        m.append()
    c.touch([0])
    m.touch([0])
    assert c.slots(0) == (0, 0) and c.slots(3) == (-1, 3)
    c.touch([1])
    m.touch([1])
    assert c.slots(0) == (0, -1) and c.slots(4) == (-1, 0) and c.slots(1) == (1, 1)
    st = c.stats()
    assert (st["reclaims"], st["offloads"]) == (m.rec, m.off) == (1, 5)


def test_capacity_and_argument_errors():
    c = _cache(2, 2, 2, max_chunks=8)
    c.append(None, None)
    c.append(None, None)
    with pytest.raises(wa.WaError) as e:
        c.append(None, None)        # both tiers full
    assert e.value.status == 6
    with pytest.raises(wa.WaError) as e:
        c.touch([0, 9])             # unknown page
    assert e.value.status == 5
    with pytest.raises(wa.WaError) as e:
        c.location(4)
    assert e.value.status == 5
    c2 = _cache(2, 2, 1, max_chunks=1)
    c2.append(None, None)
    with pytest.raises(wa.WaError) as e:
        c2.append(None, None)       # max_chunks
    assert e.value.status == 6
    with pytest.raises(wa.WaError) as e:
        wa.WaCache(4, 64, 16, 2, hbm_pages=0, host_pages=2, max_chunks=4, dry_run=True)
    assert e.value.status == 1
    with pytest.raises(wa.WaError) as e:
        wa.WaCache(3, 3, 16, 2, hbm_pages=2, host_pages=2, max_chunks=4, dry_run=True)
    assert e.value.status == 2      # head rows not whole 16-byte vectors
    with pytest.raises(wa.WaError) as e:
        wa.WaCache(4, 96, 16, 2, hbm_pages=2, host_pages=2, max_chunks=4, dry_run=True,
                   dram_format="nvfp4")
    assert e.value.status == 2      # compressed tier: head_dim 64, 128 or 256
    with pytest.raises(wa.WaError) as e:
        wa.WaCache(4, 64, 16, 2, hbm_pages=2, host_pages=2, max_chunks=4, dry_run=True,
                   dtype=torch.float32, dram_format="fp8")
    assert e.value.status == 3      # compressed tier: bf16 caches only


def test_current_pages_never_evicted():
    """A retrieval that uses as many pages as HBM holds keeps all of them."""
    c, m = _cache(3, 9, 3), Model(3, 9, 3)
    for _ in range(4):
        c.append(None, None)
        m.append()
    c.touch([0, 4, 8])
    m.touch([0, 4, 8])
    assert sorted(p for p in range(12) if c.location(p)[0] == 0) == [0, 4, 8]
