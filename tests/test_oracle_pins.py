"""Pins for the fp64 oracle: each check compares it with something other than
itself -- values worked by hand or printed on the pages, brute force over all
pairs, closed forms, or a library routine for a special case -- chosen so that a
plausible slip (a dropped 1/P or 1/sqrt(d), a wrong tie rule, a transposed
operand, a wrong concatenation order) fails at least one of them.

CPU only; no GPU, no CUDA library.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.spatial.distance
import torch

import oracle as O
from sparse_kv_cache_page_gb300 import synth


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ----------------------------------------------------------------------------
# values printed on the pages / worked by hand
# ----------------------------------------------------------------------------

def test_worked_example_geometry(golden_dir):
    """WorldAttention review page, HKV section and worked example steps 3-4."""
    g = _load(golden_dir, "worked_example_geometry.json")
    assert g["k_p"] * g["frames_per_page"] * g["tokens_per_frame"] == g["active_tokens"] == 49920
    assert synth.PAGE_TOKENS == g["frames_per_page"] * g["tokens_per_frame"]
    assert synth.ACTIVE_TOKENS == g["active_tokens"]
    ex = g["linear_branch_example"]
    lrd = ex["L"] * ex["r"] * ex["d_k"]
    l2d = ex["L"] ** 2 * ex["d_k"]
    assert f"{lrd:.1e}" == f"{ex['L_r_dk_approx']:.1e}"
    assert f"{l2d:.1e}" == f"{ex['L2_dk_approx']:.1e}"
    assert round(ex["L"] / ex["r"]) == ex["L_over_r_approx"]


def test_hand_worked_selection(golden_dir):
    g = _load(golden_dir, "hand_worked_selection.json")
    kp = np.array(g["k_pages"], dtype=np.float64)
    q = np.array(g["q"], dtype=np.float64)
    kbar = O.page_summarize(kp)
    np.testing.assert_allclose(kbar, np.array(g["kbar"], dtype=np.float64), rtol=0, atol=1e-15)
    np.testing.assert_allclose(O.mean_query(q), np.array(g["qbar"], dtype=np.float64), atol=1e-15)
    alpha = O.page_scores(O.mean_query(q), kbar, range(3), head_dim=2)
    np.testing.assert_allclose(alpha, g["alpha"], rtol=0, atol=1e-12)
    idx, sc, chunk = O.select_pages(q, kbar, None, None, pages_per_chunk=3, k_p=g["k_p"])
    assert idx.tolist() == g["idx"] and chunk == -1
    np.testing.assert_allclose(sc, [g["alpha"][i] for i in g["idx"]], atol=1e-12)
    pc = np.array(g["prompt_chunks"], dtype=np.float64)
    assert O.prompt_top1(np.array(g["prompt_cur"], dtype=np.float64), pc) == g["chunk"]


def test_hand_worked_attention(golden_dir):
    g = _load(golden_dir, "hand_worked_attention.json")
    a = {k: np.array(g[k], dtype=np.float64) for k in ("q", "k_main", "v_main", "k_loc", "v_loc")}
    o, lse = O.block_attn(a["q"], a["k_main"], a["v_main"], a["k_loc"], a["v_loc"], scale=g["scale"])
    np.testing.assert_allclose(o, np.array(g["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(g["lse"]), rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# brute force and bilinearity
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n_heads,head_dim", [(1, 64), (3, 8)])
def test_mean_key_score_equals_bruteforce(n_heads, head_dim):
    """alpha_j = Qbar.Kbar_j / sqrt(d) equals, by bilinearity, the mean over all
    (query, key) pairs of q.k / sqrt(d), summed over heads -- computed here
    pair by pair."""
    n_pages, P, n_q = 8, 32 if n_heads == 1 else 5, 16 if n_heads == 1 else 7
    kp = _rand((n_pages, P, n_heads, head_dim), 1)
    q = _rand((n_q, n_heads, head_dim), 2)
    alpha = O.page_scores(O.mean_query(q), O.page_summarize(kp), range(n_pages), head_dim)
    for j in range(n_pages):
        tot = 0.0
        for h in range(n_heads):
            for i in range(n_q):
                for t in range(P):
                    tot += float(np.dot(q[i, h], kp[j, t, h]))
        brute = tot / (n_q * P * math.sqrt(head_dim))
        assert abs(brute - alpha[j]) <= 1e-12 * max(1.0, abs(brute))


def test_mean_query_and_summary_bruteforce():
    kp = _rand((3, 5, 2, 4), 3)
    q = _rand((6, 2, 4), 4)
    kb = O.page_summarize(kp)
    qb = O.mean_query(q)
    for j in range(3):
        for h in range(2):
            for e in range(4):
                assert abs(kb[j, h, e] - sum(kp[j, t, h, e] for t in range(5)) / 5) < 1e-14
    for h in range(2):
        for e in range(4):
            assert abs(qb[h, e] - sum(q[i, h, e] for i in range(6)) / 6) < 1e-14


def test_bf16_decode_exact():
    x = torch.tensor([1.0, -2.5, 3.140625, 0.0, -0.0, 65280.0, 1e-30], dtype=torch.bfloat16)
    u = x.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(O.decode_bf16(u), x.double().numpy())


# ----------------------------------------------------------------------------
# retrieval: prompt top-1 and page top-K against library routines
# ----------------------------------------------------------------------------

def test_prompt_top1_vs_scipy_cosine():
    for seed in range(20):
        pc = _rand((7, 32), 100 + seed)
        cur = _rand((32,), 200 + seed)
        dist = scipy.spatial.distance.cdist(cur[None, :], pc, metric="cosine")[0]
        assert O.prompt_top1(cur, pc) == int(np.argmin(dist))


def test_prompt_top1_ties_and_zero_norm():
    pc = _rand((5, 16), 7)
    pc[3] = pc[1]                 # exact duplicate of chunk 1: tie -> 1
    cur = pc[1] + 0.01 * _rand((16,), 8)
    assert O.prompt_top1(cur, pc) == 1
    pc2 = np.zeros((3, 16))
    pc2[2] = -cur                 # cos = -1; zero rows have cos 0 -> chunk 0
    assert O.prompt_top1(cur, pc2) == 0
    assert O.prompt_top1(np.zeros(16), pc) == 0   # all cos 0: lowest index


def test_topk_vs_torch_topk_distinct():
    for seed in range(20):
        a = _rand((40,), 300 + seed)
        cand = list(range(40))
        k = 1 + seed % 8
        idx, sc = O.topk_pages(a, cand, k)
        ref = torch.topk(torch.from_numpy(a), k).indices.sort().values.numpy()
        assert idx.tolist() == ref.tolist()
        np.testing.assert_array_equal(sc, a[idx])


def test_topk_ties_lowest_index():
    a = np.array([0.5, 0.9, 0.5, 0.9, 0.1, 0.5])
    idx, _ = O.topk_pages(a, range(6), 3)
    assert idx.tolist() == [0, 1, 3]
    idx, _ = O.topk_pages(a, [10, 11, 12, 13, 14, 15], 4)
    assert idx.tolist() == [10, 11, 12, 13]
    # brute force over all subsets: the chosen set maximises the sum of scores,
    # and among the maximisers it is the lexicographically smallest
    for seed in range(10):
        a = np.round(_rand((9,), 400 + seed), 1)  # rounding forces ties
        for k in (1, 3, 5):
            best = max(itertools.combinations(range(9), k),
                       key=lambda s: (sum(a[list(s)]), [-i for i in s]))
            idx, _ = O.topk_pages(a, range(9), k)
            assert idx.tolist() == list(best)


def test_topk_rejects_kp_above_candidates():
    with pytest.raises(ValueError):
        O.topk_pages(np.zeros(3), range(3), 4)


def test_duplicate_pages_tie_to_lowest_index():
    kp = _rand((6, 4, 1, 8), 11)
    kp[4] = kp[1]                                   # exact duplicate page
    q = kp[1].copy() * 3.0                          # queries point at page 1's keys
    kb = O.page_summarize(kp)
    idx, sc, _ = O.select_pages(q, kb, None, None, pages_per_chunk=6, k_p=1)
    assert idx.tolist() == [1]
    idx, sc, _ = O.select_pages(q, kb, None, None, pages_per_chunk=6, k_p=2)
    assert idx.tolist() == [1, 4]
    assert sc[0] == sc[1]


def test_prompt_stage_restricts_candidates():
    c = synth.tiny_fp32_case(recall_chunk=1)
    kb = O.page_summarize(synth.to_oracle(c.k_pages))
    idx, _, chunk = O.select_pages(synth.to_oracle(c.q), kb, synth.to_oracle(c.prompt_cur),
                                   synth.to_oracle(c.prompt_chunks), c.pages_per_chunk, c.k_p)
    assert chunk == 1
    assert all(4 <= j < 8 for j in idx) and len(idx) == 2 and idx[0] < idx[1]


# ----------------------------------------------------------------------------
# gather: library special case, bit exact
# ----------------------------------------------------------------------------

def test_gather_vs_index_select_bitexact():
    kp = torch.randn(9, 5, 2, 8).to(torch.bfloat16)
    idx = [7, 0, 3]
    ours = O.gather_pages(synth.to_oracle(kp), idx)
    ref = torch.index_select(kp, 0, torch.tensor(idx)).reshape(-1, 2, 8)
    np.testing.assert_array_equal(ours, synth.to_oracle(ref))


# ----------------------------------------------------------------------------
# attention: textbook special cases and an independent library
# ----------------------------------------------------------------------------

def test_kp_all_pages_equals_dense_attention():
    """Selecting every page reproduces dense attention over all cached tokens
    plus the local KV; the dense side is torch's SDPA in fp64 over the keys in
    a shuffled order (softmax attention does not depend on key order)."""
    c = synth.tiny_fp32_case()
    kp, vp = synth.to_oracle(c.k_pages), synth.to_oracle(c.v_pages)
    kb = O.page_summarize(kp)
    idx, _, chunk = O.select_pages(synth.to_oracle(c.q), kb, None, None, c.pages_per_chunk,
                                   k_p=c.n_pages)
    assert chunk == -1 and idx.tolist() == list(range(c.n_pages))
    kbuf, vbuf = O.gather_pages(kp, idx), O.gather_pages(vp, idx)
    o, lse = O.block_attn(synth.to_oracle(c.q), kbuf, vbuf, synth.to_oracle(c.k_loc),
                          synth.to_oracle(c.v_loc))
    k_all = torch.cat([c.k_pages.reshape(-1, 1, 64), c.k_loc]).double()
    v_all = torch.cat([c.v_pages.reshape(-1, 1, 64), c.v_loc]).double()
    perm = torch.randperm(k_all.shape[0], generator=torch.Generator().manual_seed(5))
    k_all, v_all = k_all[perm], v_all[perm]
    ref = torch.nn.functional.scaled_dot_product_attention(
        c.q.double().permute(1, 0, 2)[None], k_all.permute(1, 0, 2)[None],
        v_all.permute(1, 0, 2)[None])[0].permute(1, 0, 2).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    s = (c.q.double()[:, 0] @ k_all[:, 0].T) / 8.0
    np.testing.assert_allclose(lse[0], torch.logsumexp(s, dim=1).numpy(), atol=1e-12)


def test_softmax_rows_sum_to_one():
    q = _rand((5, 16), 21)
    k = _rand((300, 16), 22)
    v = _rand((300, 16), 23)
    _, lse, p = O.attention_rows(q, k, v, 0.25)
    assert np.all(np.abs(p.sum(axis=1) - 1.0) <= 1e-12)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(0.25 * q @ k.T, axis=1), atol=1e-12)


def test_attention_special_cases():
    q = _rand((4, 1, 8), 31)
    v1 = _rand((1, 1, 8), 32)
    k1 = _rand((1, 1, 8), 33)
    o, lse = O.block_attn(q, k1, v1, None, None)               # one key: O = v
    np.testing.assert_allclose(o, np.broadcast_to(v1, o.shape), atol=1e-15)
    kz = np.zeros((10, 1, 8))
    vz = _rand((10, 1, 8), 34)
    o, lse = O.block_attn(q, kz[:6], vz[:6], kz[6:], vz[6:])    # K = 0: O = mean(V)
    np.testing.assert_allclose(o, np.broadcast_to(vz.mean(axis=0), o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, np.full((1, 4), math.log(10)), atol=1e-14)
    k = _rand((50, 1, 8), 35)
    v = _rand((50, 1, 8), 36)
    qd = 1000.0 * k[[7, 7, 20, 41]]                              # one dominant logit per row
    o, _ = O.block_attn(qd, k[:30], v[:30], k[30:], v[30:])
    np.testing.assert_allclose(o[:, 0], v[[7, 7, 20, 41], 0], atol=1e-6)


def test_segment_order_main_then_local():
    """The main segment and the local segment form one key set: any split of
    the same keys gives the same output."""
    q = _rand((3, 2, 8), 41)
    k = _rand((20, 2, 8), 42)
    v = _rand((20, 2, 8), 43)
    o1, l1 = O.block_attn(q, k, v, None, None)
    o2, l2 = O.block_attn(q, k[:13], v[:13], k[13:], v[13:])
    o3, l3 = O.block_attn(q, None, None, k, v)
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(o1, o3, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-14)


# ----------------------------------------------------------------------------
# Linformer branch and fusion
# ----------------------------------------------------------------------------

def test_linformer_projection_bruteforce():
    x = _rand((11, 2, 4), 51)
    e = _rand((2, 11, 3), 52)
    xp = O.linformer_project(x, e)
    for h in range(2):
        for r in range(3):
            for c in range(4):
                assert abs(xp[h, r, c] - sum(e[h, l, r] * x[l, h, c] for l in range(11))) < 1e-12


def test_linformer_identity_and_permutation_reduce_to_dense():
    L, H, d = 24, 2, 8
    q = _rand((5, H, d), 61)
    k = _rand((L, H, d), 62)
    v = _rand((L, H, d), 63)
    dense, _ = O.block_attn(q, k, v, None, None)
    eye = np.broadcast_to(np.eye(L), (H, L, L)).copy()
    np.testing.assert_allclose(O.linear_branch(q, k, v, eye, eye), dense, atol=1e-13)
    perm = np.eye(L)[np.random.default_rng(64).permutation(L)]
    pe = np.broadcast_to(perm, (H, L, L)).copy()
    np.testing.assert_allclose(O.linear_branch(q, k, v, pe, pe), dense, atol=1e-13)


def test_fuse_branches():
    a = _rand((4, 3, 8), 71)
    b = _rand((4, 3, 8), 72)
    np.testing.assert_allclose(O.fuse_branches(a, b), a + b, atol=0)
    np.testing.assert_allclose(O.fuse_branches(a, b, [1, 1, 1], [0, 0, 0]), a, atol=0)
    f = O.fuse_branches(a, b, [0.5, 2.0, 1.0], [0.5, 0.0, -1.0])
    np.testing.assert_allclose(f[:, 1], 2.0 * a[:, 1], atol=0)
    np.testing.assert_allclose(f[:, 2], a[:, 2] - b[:, 2], atol=0)


# ----------------------------------------------------------------------------
# planted mistakes: the pins above must catch plausible slips in the oracle
# ----------------------------------------------------------------------------

def _mutant_scores(qbar, kbar, pages, head_dim):      # forgets 1/sqrt(d)
    return np.array([float((qbar * kbar[j]).sum()) for j in pages])


def _mutant_topk(alpha, pages, k_p):                   # ties to the highest index
    pages = list(pages)
    order = sorted(range(len(pages)), key=lambda i: (-alpha[i], -pages[i]))
    chosen = sorted(order[:k_p], key=lambda i: pages[i])
    return np.array([pages[i] for i in chosen], dtype=np.int32), alpha[chosen]


def test_planted_mistakes_are_caught(monkeypatch, golden_dir):
    monkeypatch.setattr(O.wa_oracle, "page_scores", _mutant_scores)
    monkeypatch.setattr(O, "page_scores", _mutant_scores)
    with pytest.raises(AssertionError):
        test_hand_worked_selection(golden_dir)
    monkeypatch.undo()
    monkeypatch.setattr(O.wa_oracle, "topk_pages", _mutant_topk)
    monkeypatch.setattr(O, "topk_pages", _mutant_topk)
    with pytest.raises(AssertionError):
        test_topk_ties_lowest_index()


# ----------------------------------------------------------------------------
# per-head page sets
# ----------------------------------------------------------------------------

def test_per_head_scores_bruteforce_and_sum():
    """alpha[h][j] is the mean over (query, key) pairs of head h of q.k/sqrt(d),
    pair by pair; summed over heads it is the shared page score."""
    n_pages, P, n_q, H, d = 5, 6, 4, 3, 8
    kp = _rand((n_pages, P, H, d), 51)
    q = _rand((n_q, H, d), 52)
    qb, kb = O.mean_query(q), O.page_summarize(kp)
    a = O.page_scores_per_head(qb, kb, range(n_pages), d)
    for h in range(H):
        for j in range(n_pages):
            brute = sum(float(np.dot(q[i, h], kp[j, t, h])) for i in range(n_q)
                        for t in range(P)) / (n_q * P * math.sqrt(d))
            assert abs(a[h, j] - brute) <= 1e-12 * max(1.0, abs(brute))
    np.testing.assert_allclose(a.sum(axis=0), O.page_scores(qb, kb, range(n_pages), d),
                               rtol=1e-12, atol=1e-14)


def test_per_head_selection_one_head_is_shared_selection():
    kp = _rand((12, 7, 1, 16), 53)
    q = _rand((9, 1, 16), 54)
    kb = O.page_summarize(kp)
    pc, cur = _rand((3, 10), 55), _rand((10,), 56)
    idx_h, sc_h, ch_h = O.select_pages_per_head(q, kb, cur, pc, 4, 2)
    idx, sc, ch = O.select_pages(q, kb, cur, pc, 4, 2)
    assert ch_h == ch and idx_h[0].tolist() == idx.tolist()
    np.testing.assert_allclose(sc_h[0], sc, rtol=1e-15)


def test_per_head_topk_bruteforce():
    """With distinct scores each head's top-k_p set is the unique k_p-subset of
    largest score sum: checked over all subsets."""
    kp = _rand((9, 3, 4, 8), 57)
    q = _rand((5, 4, 8), 58)
    kb = O.page_summarize(kp)
    idx, _, _ = O.select_pages_per_head(q, kb, None, None, 1, 3)
    a = O.page_scores_per_head(O.mean_query(q), kb, range(9), 8)
    for h in range(4):
        best = max(itertools.combinations(range(9), 3), key=lambda c: sum(a[h, j] for j in c))
        assert idx[h].tolist() == sorted(best)


def test_per_head_gather_bitexact_and_shared_case():
    kp = (np.arange(6 * 4 * 3 * 2, dtype=np.uint16).reshape(6, 4, 3, 2) * 7) ^ 0x3f00
    idx = np.array([[5, 1], [0, 3], [2, 2]], dtype=np.int32)
    buf = O.gather_pages_per_head(kp, idx)
    for h in range(3):
        for s_ in range(2):
            for t in range(4):
                assert (buf[s_ * 4 + t, h] == kp[idx[h, s_], t, h]).all()
    same = np.array([[4, 1]] * 3, dtype=np.int32)
    assert (O.gather_pages_per_head(kp, same) == O.gather_pages(kp, [4, 1])).all()
