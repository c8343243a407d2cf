"""GPU parity of the HSA sparse branch (WorldAttention review page, HSA
section) through the C ABI against the fp64 oracle: block means, the pooled
block map and its Gini-adaptive block selection (sets compared exactly, with a
margin check that the case is not a tie within fp32 rounding), the
block-sparse attention (bf16 tolerance on the fp32 output; ragged buffer and
local blocks, forced key-range splits that leave CTAs without blocks, a head
with no blocks), the branch fused with the linear branch, and the one-layer
WorldAttention shape on sampled rows."""

import numpy as np
import pytest
import torch

import oracle as O
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
from tests._util import assert_attn_close, f64, np_of

pytestmark = pytest.mark.gpu
DEV = "cuda"
B_Q, B_MAIN, B_LOC = 64, 128, 64


def _case(n_q, n_main, n_loc, H, seed, peaked_heads=(), gain=3.0):
    """bf16 N(0,1) inputs; in the listed heads one buffer block and the queries
    share a direction, so those heads have a peaked block map."""
    s = lambda t: synth.seed_of("sparse", seed, t)  # noqa: E731
    q = synth.normal((n_q, H, 128), s("q"))
    km, vm = synth.normal((n_main, H, 128), s("km")), synth.normal((n_main, H, 128), s("vm"))
    kl, vl = synth.normal((n_loc, H, 128), s("kl")), synth.normal((n_loc, H, 128), s("vl"))
    for i, h in enumerate(peaked_heads):
        u = synth.normal((128,), s(("dir", h)))
        b = (3 * i + 1) % max(1, n_main // B_MAIN)
        km[b * B_MAIN:(b + 1) * B_MAIN, h, :] += gain * u
        q[:, h, :] += gain * u
    bf = lambda t: t.to(torch.bfloat16)  # noqa: E731
    return bf(q), bf(km), bf(vm), bf(kl), bf(vl)


def _gpu_select(q, km, kl, tau=None):
    H = q.shape[1]
    nqb = (q.shape[0] + B_Q - 1) // B_Q
    nmb = (km.shape[0] + B_MAIN - 1) // B_MAIN
    nlb = (kl.shape[0] + B_LOC - 1) // B_LOC
    qbar = torch.empty((nqb, H, 128), dtype=torch.float32, device=DEV)
    kbar = torch.empty((nmb + nlb, H, 128), dtype=torch.float32, device=DEV)
    wa.wa_block_means_segments([(q.to(DEV), B_Q, qbar), (km.to(DEV), B_MAIN, kbar[:nmb]),
                                (kl.to(DEV), B_LOC, kbar[nmb:])])
    sel = torch.full((H, nmb + nlb), -1, dtype=torch.int32, device=DEV)
    cnt = torch.empty(H, dtype=torch.int32, device=DEV)
    g = torch.empty(H, dtype=torch.float32, device=DEV)
    mass = torch.empty((H, nmb + nlb), dtype=torch.float32, device=DEV)
    t = None if tau is None else torch.tensor(tau, dtype=torch.float32, device=DEV)
    wa.wa_sparse_select(qbar, kbar, sel, cnt, tau=t, gini_out=g, mass_out=mass)
    wa.wa_check()
    c = cnt.cpu().numpy()
    sets = [sel[h, :c[h]].cpu().numpy() for h in range(H)]
    return sel, cnt, sets, f64(g), f64(mass)


def _assert_selection(sets, mass_ref, tau_ref, eps=2e-5):
    """Kept sets equal the oracle's; the oracle's boundary must clear fp32
    rounding (a tie within rounding means: change the seed)."""
    for h, ref in enumerate(O.sparse_select(mass_ref, tau=tau_ref)[0]):
        order = sorted(range(mass_ref.shape[1]), key=lambda b: (-mass_ref[h][b], b))
        cum = np.cumsum(mass_ref[h][order])
        k = len(ref)
        assert cum[k - 1] >= tau_ref[h] + eps or k == len(order), f"head {h}: tie at tau"
        if k > 1:
            assert cum[k - 2] < tau_ref[h] - eps, f"head {h}: tie at tau"
        if k < len(order):
            assert mass_ref[h][order[k - 1]] - mass_ref[h][order[k]] > eps * 1e-2, \
                f"head {h}: mass tie at the boundary"
        assert sets[h].tolist() == ref.tolist(), f"head {h}: {sets[h]} != {ref}"


@pytest.mark.parametrize("n,block", [(300, 128), (300, 64), (64, 64), (4680, 64), (1, 128)])
def test_block_means(n, block):
    x = synth.normal((n, 3, 128), synth.seed_of("bmeans", n, block), dtype=torch.bfloat16)
    nb = (n + block - 1) // block
    out = torch.empty((nb, 3, 128), dtype=torch.float32, device=DEV)
    wa.wa_block_means(x.to(DEV), block, out)
    wa.wa_check()
    ref = O.block_means(np_of(x), block)
    np.testing.assert_allclose(f64(out), ref, rtol=0, atol=2e-6)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_block_means_segments_one_launch(dtype):
    """Queries, buffer and local KV pooled in one launch: each set's means are
    those of its own wa_block_means call, bit for bit (ragged last blocks, a
    set large enough to split its blocks and one that is not), and match the
    oracle."""
    sets = [(synth.normal((300, 3, 128), synth.seed_of("bmseg", i), dtype=dtype), blk)
            for i, blk in enumerate((64,))]
    sets += [(synth.normal((4999, 3, 128), synth.seed_of("bmseg", 1), dtype=dtype), 128),
             (synth.normal((77, 3, 128), synth.seed_of("bmseg", 2), dtype=dtype), 64)]
    fused, alone = [], []
    for x, blk in sets:
        nb = (x.shape[0] + blk - 1) // blk
        fused.append(torch.full((nb, 3, 128), float("nan"), device=DEV))
        alone.append(torch.empty((nb, 3, 128), device=DEV))
    xs = [x.to(DEV) for x, _ in sets]
    wa.wa_block_means_segments([(x, blk, o) for x, (_, blk), o in zip(xs, sets, fused)])
    for x, (_, blk), o in zip(xs, sets, alone):
        wa.wa_block_means(x, blk, o)
    wa.wa_check()
    for (x, blk), f, a in zip(sets, fused, alone):
        assert torch.equal(f, a)
        np.testing.assert_allclose(f64(f), O.block_means(np_of(x), blk), rtol=0, atol=2e-6)


def test_select_matches_oracle_small():
    q, km, vm, kl, vl = _case(200, 640, 100, 3, 1, peaked_heads=(0,))
    _, _, sets, g, mass = _gpu_select(q, km, kl)
    mref = O.pooled_mass(np_of(q), np_of(km), np_of(kl))
    np.testing.assert_allclose(mass, mref, rtol=0, atol=2e-6)
    gref = np.array([O.gini(m) for m in mref])
    np.testing.assert_allclose(g, gref, rtol=0, atol=2e-5)
    assert g[0] > g[1] and len(sets[0]) < len(sets[1])
    _assert_selection(sets, mref, 1.0 - gref)


def test_select_given_tau():
    q, km, vm, kl, vl = _case(130, 1024, 200, 3, 2, peaked_heads=(1,))
    tau = [0.5, 0.9, 1.0]
    _, _, sets, _, _ = _gpu_select(q, km, kl, tau=tau)
    mref = O.pooled_mass(np_of(q), np_of(km), np_of(kl))
    assert len(sets[2]) == mref.shape[1]            # tau = 1 keeps every block
    _assert_selection(sets[:2], mref[:2], np.array(tau[:2]))


def _gpu_sparse_attn(q, km, vm, kl, vl, sel, cnt):
    o = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    d = lambda t: None if t is None else t.to(DEV)  # noqa: E731
    wa.wa_sparse_attn(q.to(DEV), d(km), d(vm), d(kl), d(vl), sel, cnt, o, B_MAIN, B_LOC)
    wa.wa_check()
    return o


def _sel_tensors(sets, n_kb):
    H = len(sets)
    sel = torch.full((H, n_kb), -1, dtype=torch.int32)
    cnt = torch.zeros(H, dtype=torch.int32)
    for h, s in enumerate(sets):
        sel[h, :len(s)] = torch.tensor(np.asarray(s, dtype=np.int32))
        cnt[h] = len(s)
    return sel.to(DEV), cnt.to(DEV)


@pytest.mark.parametrize("split", [None, 1, 3, 7])
def test_sparse_attn_given_blocks(monkeypatch, split):
    if split is None:
        monkeypatch.delenv("WA_ATTN_SPLIT", raising=False)
    else:
        monkeypatch.setenv("WA_ATTN_SPLIT", str(split))
    # 700 buffer rows: 6 blocks (last 60 rows); 150 local rows: 3 blocks (last 22)
    q, km, vm, kl, vl = _case(300, 700, 150, 3, 3)
    sets = [[0, 2, 5, 6, 8], [5], [1, 3, 4, 6, 7, 8]]
    sel, cnt = _sel_tensors(sets, 9)
    o = _gpu_sparse_attn(q, km, vm, kl, vl, sel, cnt)
    ref = O.sparse_attn(np_of(q), np_of(km), np_of(vm), np_of(kl), np_of(vl),
                        [np.array(s) for s in sets])
    assert_attn_close(o, ref, torch.bfloat16, f"split {split}")


def test_sparse_attn_every_block_is_dense_attention():
    q, km, vm, kl, vl = _case(260, 512, 200, 2, 4)
    n_kb = len(O.key_blocks(512, 200))
    sel, cnt = _sel_tensors([list(range(n_kb))] * 2, n_kb)
    o = _gpu_sparse_attn(q, km, vm, kl, vl, sel, cnt)
    ref, _ = O.block_attn(np_of(q), np_of(km), np_of(vm), np_of(kl), np_of(vl))
    assert_attn_close(o, ref, torch.bfloat16, "all blocks")


def test_sparse_attn_head_without_blocks(monkeypatch):
    monkeypatch.setenv("WA_ATTN_SPLIT", "2")
    q, km, vm, kl, vl = _case(100, 256, 64, 2, 5)
    sel, cnt = _sel_tensors([[0, 2], []], 3)
    o = _gpu_sparse_attn(q, km, vm, kl, vl, sel, cnt)
    assert torch.count_nonzero(o[:, 1, :]).item() == 0
    ref = O.sparse_attn(np_of(q)[:, :1], np_of(km)[:, :1], np_of(vm)[:, :1], np_of(kl)[:, :1],
                        np_of(vl)[:, :1], [np.array([0, 2])])
    assert_attn_close(o[:, :1, :], ref, torch.bfloat16, "head 0")


def test_hsa_branches_fused():
    """Sparse branch, then the linear branch accumulated with per-head gates
    (WorldAttention review page, HSA: o = w_attn o_sparse + w_lin o_lin)."""
    q, km, vm, kl, vl = _case(300, 1024, 128, 2, 6, peaked_heads=(0,))
    sel, cnt, sets, _, _ = _gpu_select(q, km, kl)
    o = _gpu_sparse_attn(q, km, vm, kl, vl, sel, cnt)
    L, r = 1024 + 128, 128
    ek = synth.normal((2, L, r), synth.seed_of("sparse", 6, "ek"), dtype=torch.bfloat16, std=L ** -0.5)
    ev = synth.normal((2, L, r), synth.seed_of("sparse", 6, "ev"), dtype=torch.bfloat16, std=L ** -0.5)
    wa_, wl_ = torch.tensor([0.7, 1.3], device=DEV), torch.tensor([0.4, 0.9], device=DEV)
    wa.wa_linear_branch(q.to(DEV), km.to(DEV), vm.to(DEV), kl.to(DEV), vl.to(DEV), ek.to(DEV),
                        ev.to(DEV), o, w_attn=wa_, w_lin=wl_)
    wa.wa_check()
    o_sp = O.sparse_attn(np_of(q), np_of(km), np_of(vm), np_of(kl), np_of(vl), sets)
    kc = np.concatenate([np_of(km), np_of(kl)])
    vc = np.concatenate([np_of(vm), np_of(vl)])
    o_lin = O.linear_branch(np_of(q), kc, vc, np_of(ek), np_of(ev))
    ref = O.fuse_branches(o_sp, o_lin, [0.7, 1.3], [0.4, 0.9])
    assert_attn_close(o, ref, torch.bfloat16, "fused")


def test_sparse_branch_worldattention_shape_sampled():
    """One layer at the WorldAttention shape: 49,920 buffer + 4,680 local
    tokens, 4,680 queries, 12 heads; two heads planted peaked.  Sets for every
    head; the output on sampled rows."""
    q, km, vm, kl, vl = _case(4680, 49920, 4680, 12, 7, peaked_heads=(2, 9))
    sel, cnt, sets, g, mass = _gpu_select(q, km, kl)
    qn, kmn, kln = np_of(q), np_of(km), np_of(kl)
    mref = O.pooled_mass(qn, kmn, kln)
    np.testing.assert_allclose(mass, mref, rtol=0, atol=2e-6)
    gref = np.array([O.gini(m) for m in mref])
    _assert_selection(sets, mref, 1.0 - gref)
    assert len(sets[2]) < len(sets[0]) and len(sets[9]) < len(sets[0])
    o = _gpu_sparse_attn(q, km, vm, kl, vl, sel, cnt)
    rows = np.random.default_rng(7).choice(4680, 48, replace=False)
    ref = O.sparse_attn(qn, kmn, np_of(vm), kln, np_of(vl), sets, rows=rows)
    assert_attn_close(o[torch.as_tensor(rows, device=DEV)], ref, torch.bfloat16, "sampled rows")
