"""GPU parity of gather and attention in one launch (wa_gather_attn).

The gathered buffer must equal the oracle's gather bit for bit (WorldAttention
review page, Fig. 1 and the HKV section: the selected pages copied, in slot
order, into one contiguous buffer). The attention must be within the bf16
tolerance of the oracle's attention over [buffer ; local] (Inferix summary
page, §3 Step 3). Both must also be bit-identical to the two-launch path
(wa_gather_pages, then wa_block_attn), which the fused launch reproduces.

The cases cover:

* pages of 64 rows, where a key tile spans two pages;
* pages of 192 and 320 rows, where a tile straddles a page boundary;
* pages that are not whole 64-row boxes (24, 200, 1,560 rows: 8-row boxes);
* an odd number of 64-row boxes, where the last tile is half past the buffer;
* repeated and unsorted indices;
* a page set per head, small and at the full WorldAttention size;
* no buffer output; a bf16 output without LSE;
* forced split counts, which move the buffer stores between CTAs;
* bad indices;
* the one-layer WorldAttention chunk at full size, with the pages the
  selection picks;
* fp32 inputs (the CUDA-core kernel's paged form), pages of any size, and the
  tiny fp32 workload's chain through the one launch, within 1e-5.
"""

import numpy as np
import pytest
import torch

import oracle as O
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
from tests._util import LSE_ABS, assert_attn_close, f64, np_of

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128


@pytest.fixture
def split(monkeypatch):
    def _set(n):
        if n is None:
            monkeypatch.delenv("WA_ATTN_SPLIT", raising=False)
        else:
            monkeypatch.setenv("WA_ATTN_SPLIT", str(n))
    yield _set
    monkeypatch.delenv("WA_ATTN_SPLIT", raising=False)


def _bank(tag, n_pages, P, H, n_q, n_loc):
    g = lambda shape, t: synth.normal(shape, synth.seed_of("gattn", tag, t), DEV,  # noqa: E731
                                      torch.bfloat16, std=D ** -0.25)
    kp, vp = g((n_pages, P, H, D), "kp"), g((n_pages, P, H, D), "vp")
    q = g((n_q, H, D), "q")
    kl = g((n_loc, H, D), "kl") if n_loc else None
    vl = g((n_loc, H, D), "vl") if n_loc else None
    return kp, vp, q, kl, vl


def _bufs(idx, P, H):
    n = idx.shape[-1] * P
    return (torch.full((n, H, D), 7.0, dtype=torch.bfloat16, device=DEV),
            torch.full((n, H, D), 7.0, dtype=torch.bfloat16, device=DEV))


def _two_launch(q, kp, vp, idx, kl, vl, check=True):
    P, H = kp.shape[1], kp.shape[2]
    kb, vb = _bufs(idx, P, H)
    if idx.dim() == 2:
        wa.wa_gather_pages_per_head(kp, vp, idx, kb, vb)
    else:
        wa.wa_gather_pages(kp, vp, idx, None, kb, vb)
    o = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    lse = torch.empty((H, q.shape[0]), dtype=torch.float32, device=DEV)
    wa.wa_block_attn(q, kb, vb, kl, vl, o, lse)
    if check:
        wa.wa_check()
    return kb, vb, o, lse


def _fused(q, kp, vp, idx, kl, vl, with_buf=True, check=True):
    P, H = kp.shape[1], kp.shape[2]
    kb, vb = _bufs(idx, P, H) if with_buf else (None, None)
    o = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    lse = torch.empty((H, q.shape[0]), dtype=torch.float32, device=DEV)
    wa.wa_gather_attn(q, kp, vp, idx, kl, vl, o, kb, vb, lse)
    if check:
        wa.wa_check()
    return kb, vb, o, lse


def _oracle_check(q, kp, vp, idx, kl, vl, kb, vb, o, lse, what):
    okp, ovp = np_of(kp), np_of(vp)
    ix = idx.cpu().numpy()
    gather = O.gather_pages_per_head if ix.ndim == 2 else O.gather_pages
    rk, rv = gather(okp, ix), gather(ovp, ix)
    assert np.array_equal(np_of(kb), rk), f"{what}: gathered keys"
    assert np.array_equal(np_of(vb), rv), f"{what}: gathered values"
    n = lambda t: None if t is None else np_of(t)  # noqa: E731
    ref_o, ref_lse = O.block_attn(np_of(q), rk, rv, n(kl), n(vl))
    assert_attn_close(o, ref_o, torch.bfloat16, what)
    assert np.abs(f64(lse) - ref_lse).max() <= LSE_ABS, what


@pytest.mark.parametrize("tag,n_pages,P,idx,H,n_q,n_loc", [
    ("p192", 6, 192, [5, 0, 3], 2, 300, 100),      # tiles straddle page boundaries
    ("p64odd", 5, 64, [4, 1, 1], 3, 520, 0),       # 3 boxes: the last tile half past the buffer
    ("p128one", 4, 128, [2], 1, 17, 33),           # one page, one tile, few queries
    ("p320", 3, 320, [2, 0], 2, 1000, 250),        # 5 boxes per page, ragged local tail
    ("p200", 5, 200, [4, 1, 3], 2, 300, 60),       # not whole 64-row boxes: 8-row boxes
    ("p24", 6, 24, [5, 0, 2, 2, 1], 1, 150, 40),   # pages smaller than a tile
    ("p1560", 4, 1560, [3, 1], 2, 700, 100),       # one 1,560-token frame per page
])
def test_fused_equals_two_launch_and_oracle(tag, n_pages, P, idx, H, n_q, n_loc):
    kp, vp, q, kl, vl = _bank(tag, n_pages, P, H, n_q, n_loc)
    ix = torch.tensor(idx, dtype=torch.int32, device=DEV)
    kb, vb, o, lse = _fused(q, kp, vp, ix, kl, vl)
    kb2, vb2, o2, lse2 = _two_launch(q, kp, vp, ix, kl, vl)
    assert torch.equal(kb, kb2) and torch.equal(vb, vb2)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    _oracle_check(q, kp, vp, ix, kl, vl, kb, vb, o, lse, tag)


@pytest.mark.parametrize("n_split", [1, 2, 3, 5])
def test_every_split_writes_every_buffer_tile_once(split, n_split):
    """Three query pairs over 9 key tiles of 64-row pages: the storing CTA
    of a tile depends on the split; every tile is written, and the result
    equals the two-launch path under the same split."""
    split(n_split)
    kp, vp, q, kl, vl = _bank(f"split{n_split}", 12, 64, 2, 700, 130)
    ix = torch.tensor([11, 3, 7, 0, 9, 2, 5, 8, 1, 4, 6, 10, 3, 3], dtype=torch.int32, device=DEV)
    kb, vb, o, lse = _fused(q, kp, vp, ix, kl, vl)
    kb2, vb2, o2, lse2 = _two_launch(q, kp, vp, ix, kl, vl)
    assert torch.equal(kb, kb2) and torch.equal(vb, vb2)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    _oracle_check(q, kp, vp, ix, kl, vl, kb, vb, o, lse, f"split {n_split}")


def test_page_set_per_head():
    H, P = 4, 128
    kp, vp, q, kl, vl = _bank("perhead", 9, P, H, 400, 64)
    ix = torch.tensor([[0, 4, 8], [1, 2, 3], [8, 7, 6], [5, 5, 0]], dtype=torch.int32, device=DEV)
    kb, vb, o, lse = _fused(q, kp, vp, ix, kl, vl)
    kb2, vb2, o2, lse2 = _two_launch(q, kp, vp, ix, kl, vl)
    assert torch.equal(kb, kb2) and torch.equal(vb, vb2)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    _oracle_check(q, kp, vp, ix, kl, vl, kb, vb, o, lse, "per head")


def test_attention_only_without_a_buffer():
    kp, vp, q, kl, vl = _bank("nobuf", 5, 192, 2, 260, 90)
    ix = torch.tensor([4, 2], dtype=torch.int32, device=DEV)
    _, _, o, lse = _fused(q, kp, vp, ix, kl, vl, with_buf=False)
    _, _, o2, lse2 = _two_launch(q, kp, vp, ix, kl, vl)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_bf16_output_and_no_lse():
    """The bf16 output (rounded once, as wa_block_attn rounds it) and a call
    without LSE give the two-launch path's bits."""
    kp, vp, q, kl, vl = _bank("bf16out", 6, 128, 3, 333, 77)
    ix = torch.tensor([5, 1, 2], dtype=torch.int32, device=DEV)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=DEV)
    wa.wa_gather_attn(q, kp, vp, ix, kl, vl, o)
    kb, vb = _bufs(ix, 128, 3)
    wa.wa_gather_pages(kp, vp, ix, None, kb, vb)
    o2 = torch.empty_like(o)
    wa.wa_block_attn(q, kb, vb, kl, vl, o2)
    wa.wa_check()
    assert torch.equal(o, o2)
    ref, _ = O.block_attn(np_of(q), np_of(kb), np_of(vb), np_of(kl), np_of(vl))
    err = np.abs(f64(o) - ref)
    # the fp32 tolerance plus half a bf16 ulp of rounding of the output
    assert err.max() <= 1e-2 + np.abs(ref).max() * 2.0 ** -9


def test_page_set_per_head_at_full_size():
    """The per-head workload: the WorldAttention bank with a top-4 page set
    per head from the per-head selection; the one launch equals the per-head
    gather then attention bit for bit, and the buffer equals each head's
    pages indexed on the device."""
    c = synth.worldattention_case(device=DEV, recall_chunk=3)
    kbar = torch.empty((c.n_pages, c.n_heads, D), dtype=torch.float32, device=DEV)
    wa.wa_page_summarize(c.k_pages, kbar)
    ix = torch.empty((c.n_heads, c.k_p), dtype=torch.int32, device=DEV)
    wa.wa_select_pages_per_head(c.q, kbar, c.prompt_cur, c.prompt_chunks, c.pages_per_chunk,
                                c.k_p, ix)
    kb, vb, o, lse = _fused(c.q, c.k_pages, c.v_pages, ix, c.k_loc, c.v_loc)
    kb2, vb2, o2, lse2 = _two_launch(c.q, c.k_pages, c.v_pages, ix, c.k_loc, c.v_loc)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert torch.equal(kb, kb2) and torch.equal(vb, vb2)
    P = c.page_tokens
    for h in (0, 5, 11):
        for s_ in range(c.k_p):
            page = int(ix[h, s_])
            assert torch.equal(kb[s_ * P:(s_ + 1) * P, h], c.k_pages[page, :, h])
            assert torch.equal(vb[s_ * P:(s_ + 1) * P, h], c.v_pages[page, :, h])


def test_bad_index_reads_zeros_and_is_recorded():
    """An index outside [0, n_pages) gives a slot of zeros, as the gather
    does, and WA_ERR_INDEX from wa_check; the launch is otherwise complete."""
    kp, vp, q, kl, vl = _bank("bad", 4, 64, 2, 200, 50)
    ix = torch.tensor([1, 4, -2], dtype=torch.int32, device=DEV)
    wa.wa_check()
    kb, vb, o, lse = _fused(q, kp, vp, ix, kl, vl, check=False)
    with pytest.raises(wa.WaError) as e:
        wa.wa_check()
    assert e.value.status == 5
    kb2, vb2, o2, lse2 = _two_launch(q, kp, vp, ix, kl, vl, check=False)
    with pytest.raises(wa.WaError):
        wa.wa_check()
    assert torch.all(kb[64:] == 0) and torch.all(vb[64:] == 0)
    assert torch.equal(kb, kb2) and torch.equal(vb, vb2)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_worldattention_chunk_at_full_size():
    """The one-layer WorldAttention chunk (40 pages of 12,480 tokens, 12
    heads; 4,680 queries and 4,680 local tokens), with the four pages the
    selection picks: the fused launch equals the two-launch path bit for bit,
    the buffer equals the pages indexed on the device, and sampled rows match
    the oracle."""
    c = synth.worldattention_case(device=DEV, recall_chunk=3)
    kbar = torch.empty((c.n_pages, c.n_heads, D), dtype=torch.float32, device=DEV)
    wa.wa_page_summarize(c.k_pages, kbar)
    ix = torch.empty(c.k_p, dtype=torch.int32, device=DEV)
    wa.wa_select_pages(c.q, kbar, c.prompt_cur, c.prompt_chunks, c.pages_per_chunk, c.k_p, ix)
    kb, vb, o, lse = _fused(c.q, c.k_pages, c.v_pages, ix, c.k_loc, c.v_loc)
    kb2, vb2, o2, lse2 = _two_launch(c.q, c.k_pages, c.v_pages, ix, c.k_loc, c.v_loc)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert torch.equal(kb, kb2) and torch.equal(vb, vb2)
    il = ix.long()
    assert torch.equal(kb, c.k_pages[il].reshape(kb.shape))
    assert torch.equal(vb, c.v_pages[il].reshape(vb.shape))
    rows = list(range(0, c.q.shape[0], 389)) + [c.q.shape[0] - 1]
    ref_o, ref_lse = O.block_attn(np_of(c.q), np_of(kb), np_of(vb), np_of(c.k_loc),
                                  np_of(c.v_loc), rows=rows)
    assert_attn_close(o[rows], ref_o, torch.bfloat16, "WorldAttention chunk")
    assert np.abs(f64(lse[:, rows]) - ref_lse).max() <= LSE_ABS


@pytest.mark.parametrize("seed", range(16))
def test_random_shapes_equal_two_launches(seed):
    """Seeded random shapes: pages of 40..448 rows (multiples of 8), 1..6
    slots with repeats, 1..5 heads, 1..700 queries, 0..300 local tokens, a
    shared or a per-head page set; the one launch equals the two launches bit
    for bit, and the buffer equals the pages indexed on the device."""
    rng = np.random.default_rng(1000 + seed)
    P = int(rng.choice([64, 128, 192, 256, 448, 40, 136, 264]))
    n_pages, k_p = int(rng.integers(2, 9)), int(rng.integers(1, 7))
    H, n_q, n_loc = int(rng.integers(1, 6)), int(rng.integers(1, 701)), int(rng.integers(0, 301))
    per_head = bool(rng.integers(0, 2))
    kp, vp, q, kl, vl = _bank(f"rand{seed}", n_pages, P, H, n_q, n_loc)
    shape = (H, k_p) if per_head else (k_p,)
    ix = torch.from_numpy(rng.integers(0, n_pages, size=shape).astype(np.int32)).to(DEV)
    kb, vb, o, lse = _fused(q, kp, vp, ix, kl, vl)
    kb2, vb2, o2, lse2 = _two_launch(q, kp, vp, ix, kl, vl)
    assert torch.equal(o, o2) and torch.equal(lse, lse2), (P, n_pages, k_p, H, n_q, n_loc, per_head)
    assert torch.equal(kb, kb2) and torch.equal(vb, vb2)
    il = ix.long()
    for s_ in range(k_p):
        for h in range(H):
            page = int(il[h, s_]) if per_head else int(il[s_])
            assert torch.equal(kb[s_ * P:(s_ + 1) * P, h], kp[page, :, h])


@pytest.mark.parametrize("P,idx,per_head", [(32, [3, 0], False), (50, [1, 1, 2], False),
                                            (24, [[2, 0], [1, 3]], True)])
def test_fp32_pages_of_any_size(P, idx, per_head):
    """fp32 inputs: the CUDA-core kernel reads the pages itself (any page
    size), writes the buffer from each head's first CTA, and equals the
    two launches bit for bit and the oracle within 1e-5."""
    H = 2
    g = lambda shape, t: synth.normal(shape, synth.seed_of("gattn32", P, t), DEV,  # noqa: E731
                                      torch.float32)
    kp, vp = g((4, P, H, 64), "kp"), g((4, P, H, 64), "vp")
    q, kl, vl = g((37, H, 64), "q"), g((19, H, 64), "kl"), g((19, H, 64), "vl")
    ix = torch.tensor(idx, dtype=torch.int32, device=DEV)
    k_p = ix.shape[-1]
    kb = torch.full((k_p * P, H, 64), 7.0, device=DEV)
    vb = torch.full_like(kb, 7.0)
    o = torch.empty(q.shape, device=DEV)
    lse = torch.empty((H, 37), device=DEV)
    wa.wa_gather_attn(q, kp, vp, ix, kl, vl, o, kb, vb, lse)
    kb2, vb2 = torch.empty_like(kb), torch.empty_like(vb)
    if per_head:
        wa.wa_gather_pages_per_head(kp, vp, ix, kb2, vb2)
    else:
        wa.wa_gather_pages(kp, vp, ix, None, kb2, vb2)
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    wa.wa_block_attn(q, kb2, vb2, kl, vl, o2, lse2)
    wa.wa_check()
    assert torch.equal(kb, kb2) and torch.equal(vb, vb2)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    gather = O.gather_pages_per_head if per_head else O.gather_pages
    rk, rv = gather(np_of(kp), ix.cpu().numpy()), gather(np_of(vp), ix.cpu().numpy())
    assert np.array_equal(np_of(kb), rk)
    ref, ref_lse = O.block_attn(np_of(q), rk, rv, np_of(kl), np_of(vl))
    assert_attn_close(o, ref, torch.float32, "fp32 paged")
    assert np.abs(f64(lse) - ref_lse).max() <= 1e-5


def test_tiny_fp32_workload_chain_in_one_launch():
    """The tiny fp32 workload (1 head, d_k = 64, 2-frame pages of 32 tokens,
    8 pages in 2 chunks, K_p = 2 after the prompt stage): summaries,
    retrieval, then the gather and the attention in one launch, against the
    oracle within 1e-5."""
    c = synth.tiny_fp32_case(recall_chunk=1)
    kp, vp, q = c.k_pages.to(DEV), c.v_pages.to(DEV), c.q.to(DEV)
    kbar = torch.empty((c.n_pages, c.n_heads, c.head_dim), dtype=torch.float32, device=DEV)
    wa.wa_page_summarize(kp, kbar)
    ix = torch.empty(c.k_p, dtype=torch.int32, device=DEV)
    wa.wa_select_pages(q, kbar, c.prompt_cur.to(DEV), c.prompt_chunks.to(DEV), c.pages_per_chunk,
                       c.k_p, ix)
    kb = torch.empty((c.k_p * c.page_tokens, c.n_heads, c.head_dim), device=DEV)
    vb = torch.empty_like(kb)
    o = torch.empty(q.shape, device=DEV)
    wa.wa_gather_attn(q, kp, vp, ix, c.k_loc.to(DEV), c.v_loc.to(DEV), o, kb, vb)
    wa.wa_check()
    okp, ovp, oq = np_of(c.k_pages), np_of(c.v_pages), np_of(c.q)
    idx, _, ch = O.select_pages(oq, O.page_summarize(okp), np_of(c.prompt_cur),
                                np_of(c.prompt_chunks), c.pages_per_chunk, c.k_p)
    assert ch == 1 and ix.cpu().tolist() == idx.tolist()
    rk, rv = O.gather_pages(okp, idx), O.gather_pages(ovp, idx)
    assert np.array_equal(np_of(kb), rk) and np.array_equal(np_of(vb), rv)
    ref, _ = O.block_attn(oq, rk, rv, np_of(c.k_loc), np_of(c.v_loc))
    assert_attn_close(o, ref, torch.float32, "tiny chain in one launch")
