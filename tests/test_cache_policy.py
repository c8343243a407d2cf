"""Host logic of the KV cache manager (libwa wa_cache_*), on CPU with dry-run
caches (no device memory, no CUDA calls): page placement across the HBM and
DRAM tiers under appends and retrievals, checked against a reference model
written here from the stated policy -- pages to free HBM slots (lowest slot
first), the least recently used resident page (ties: lower page) offloaded to
the lowest free DRAM slot when HBM is full, pages of the current append or
retrieval never evicted, a page used from DRAM promoted back to HBM after
releasing its DRAM slot, one clock tick per append and per retrieval."""

import random

import pytest

import sparse_kv_cache_page_gb300 as wa


class Model:
    def __init__(self, hbm, host, ppc):
        self.hbm, self.host, self.ppc = [None] * hbm, [None] * host, ppc
        self.tab, self.clock, self.n, self.off, self.pro = {}, 0, 0, 0, 0

    @staticmethod
    def _free(arr):
        return next((i for i, x in enumerate(arr) if x is None), None)

    def _lru(self, tier, keep):
        c = [p for p, (t, _, _) in self.tab.items() if t == tier and p not in keep]
        return min(c, key=lambda p: (self.tab[p][2], p)) if c else None

    def _offload(self, p):
        hs = self._free(self.host)
        assert hs is not None
        _, s, u = self.tab[p]
        self.hbm[s], self.host[hs] = None, p
        self.tab[p] = (1, hs, u)
        self.off += 1

    def _hbm_slot(self, keep):
        s = self._free(self.hbm)
        if s is None:
            v = self._lru(0, keep)
            s = self.tab[v][1]
            self._offload(v)
        return s

    def append(self):
        self.clock += 1
        keep = set()
        for _ in range(self.ppc):
            p = self.n
            self.n += 1
            self.tab[p] = (-1, -1, self.clock)
            keep.add(p)
            s = self._hbm_slot(keep)
            self.hbm[s] = p
            self.tab[p] = (0, s, self.clock)

    def touch(self, pages):
        self.clock += 1
        keep = set(pages)
        for p in pages:
            t, s, _ = self.tab[p]
            self.tab[p] = (t, s, self.clock)
            if t == 1:
                self.host[s] = None
                hs = self._hbm_slot(keep)
                self.hbm[hs] = p
                self.tab[p] = (0, hs, self.clock)
                self.pro += 1


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
            assert c.location(p) == m.tab[p][:2], f"step {step}, page {p}"
        st = c.stats()
        assert st["n_pages"] == m.n and st["offloads"] == m.off and st["promotions"] == m.pro
        assert st["in_hbm"] == sum(x is not None for x in m.hbm) <= hbm
        assert st["in_hbm"] + st["in_host"] == m.n


def test_bytes_planned():
    c = _cache(2, 4, 2, page_tokens=16)
    page = 16 * 4 * 64 * 2
    c.append(None, None)
    c.append(None, None)            # pages 0, 1 offloaded
    c.touch([0])                    # page 0 back, page 2 (oldest of chunk 1) out
    st = c.stats()
    assert st["bytes_d2d"] == 4 * 2 * page + 2 * page    # appends + the promotion
    assert st["bytes_d2h"] == 3 * 2 * page               # three offloads
    assert (st["offloads"], st["promotions"]) == (3, 1)
    assert c.location(0) == (0, 0) and c.location(2)[0] == 1


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


def test_current_pages_never_evicted():
    """A retrieval that uses as many pages as HBM holds keeps all of them."""
    c, m = _cache(3, 9, 3), Model(3, 9, 3)
    for _ in range(4):
        c.append(None, None)
        m.append()
    c.touch([0, 4, 8])
    m.touch([0, 4, 8])
    assert sorted(p for p in range(12) if c.location(p)[0] == 0) == [0, 4, 8]
