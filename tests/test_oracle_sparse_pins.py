"""Pins for the oracle's HSA sparse branch (WorldAttention review page, HSA
section): block means, the pooled block map, the Gini coefficient, the
cumulative-mass block selection and the block-restricted attention, each
checked against something other than the oracle itself -- a hand-worked
example, the pairwise definition of the Gini coefficient, brute force over all
block subsets, token-level attention when every block is one token, dense
attention when every block is kept, and torch's SDPA on the kept tokens.

CPU only; no GPU, no CUDA library.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _hand_case():
    ln4, ln2 = math.log(4.0), math.log(2.0)
    q = np.array([0.5, 1.5]).reshape(2, 1, 1)
    km = np.array([ln4, ln4, ln2, ln2]).reshape(4, 1, 1)
    vm = np.array([1.0, 3.0, 5.0, 7.0]).reshape(4, 1, 1)
    kl = np.zeros((2, 1, 1))
    vl = np.array([100.0, 200.0]).reshape(2, 1, 1)
    return q, km, vm, kl, vl


def test_hand_worked_sparse(golden_dir):
    with open(os.path.join(golden_dir, "hand_worked_sparse.json")) as f:
        g = json.load(f)
    q, km, vm, kl, vl = _hand_case()
    mass = O.pooled_mass(q, km, kl, scale=1.0, b_q=2, b_inter=2, b_intra=1)
    np.testing.assert_allclose(mass[0], g["mass"], rtol=0, atol=1e-15)
    assert O.gini(mass[0]) == pytest.approx(g["gini_value"], abs=1e-15)
    sel, gg, tau = O.sparse_select(mass)
    assert tau[0] == pytest.approx(g["tau"], abs=1e-15)
    assert sel[0].tolist() == g["selected"]
    # the threshold read the other way round (tau = G) keeps a different set
    sel_wrong, _, _ = O.sparse_select(mass, tau=[gg[0]])
    assert sel_wrong[0].tolist() == g["selected_if_tau_were_gini"] != g["selected"]
    o = O.sparse_attn(q, km, vm, kl, vl, sel, scale=1.0, b_inter=2, b_intra=1)
    assert o[0, 0, 0] == pytest.approx(g["o_row0"], abs=1e-12)
    assert o[1, 0, 0] == pytest.approx(g["o_row1"], abs=1e-12)


def test_gini_closed_forms_and_pairwise_definition():
    assert O.gini(np.full(7, 0.3)) == pytest.approx(0.0, abs=1e-15)
    for n in (2, 5, 40):
        assert O.gini(np.eye(n)[3 % n]) == pytest.approx(1.0 - 1.0 / n, abs=1e-15)
    assert O.gini([0.5, 0.5, 0.0, 0.0]) == pytest.approx(0.5, abs=1e-15)
    rng = np.random.default_rng(5)
    for n in (3, 10, 57):
        x = rng.random(n) ** 3
        pair = np.abs(x[:, None] - x[None, :]).sum() / (2.0 * n * n * x.mean())
        assert O.gini(x) == pytest.approx(pair, rel=1e-12)


def test_block_means_ragged_brute_force():
    x = _rand((29, 2, 3), 11)
    m = O.block_means(x, 8)
    assert m.shape == (4, 2, 3)
    for b, (a, e) in enumerate([(0, 8), (8, 16), (16, 24), (24, 29)]):
        ref = np.zeros((2, 3))
        for r in range(a, e):
            ref += x[r]
        np.testing.assert_allclose(m[b], ref / (e - a), rtol=1e-13, atol=1e-15)


def test_key_blocks_worldattention_geometry():
    """49,920 retrieved tokens in blocks of B_inter = 128 and 4,680 chunk tokens
    in blocks of B_intra = 64 (WorldAttention review page, HSA section)."""
    kb = O.key_blocks(49920, 4680)
    main = [b for b in kb if b[0] == 0]
    loc = [b for b in kb if b[0] == 1]
    assert len(main) == 390 and all(e - a == 128 for _, a, e in main)
    assert len(loc) == 74 and loc[-1][2] - loc[-1][1] == 4680 - 73 * 64 == 8
    assert kb[:390] == main and kb[390:] == loc


def test_pooled_mass_blocks_of_one_token_is_token_attention():
    """With one token per block the pooled map is the token attention map; the
    block mass is then the attention probability averaged over queries."""
    q, km, kl = _rand((6, 2, 4), 1), _rand((5, 2, 4), 2), _rand((3, 2, 4), 3)
    mass = O.pooled_mass(q, km, kl, scale=0.7, b_q=1, b_inter=1, b_intra=1)
    kk = np.concatenate([km, kl], axis=0)
    for h in range(2):
        p = scipy.special.softmax(0.7 * q[:, h, :] @ kk[:, h, :].T, axis=1)
        np.testing.assert_allclose(mass[h], p.mean(axis=0), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(mass.sum(axis=1), 1.0, rtol=0, atol=1e-13)


def test_selection_is_minimal_brute_force():
    """The kept set is a smallest set of blocks whose mass reaches tau, and it
    is the top of the mass order (ties to the lower block index)."""
    rng = np.random.default_rng(9)
    for trial in range(40):
        n = int(rng.integers(1, 9))
        m = rng.random(n) ** 2
        if trial % 5 == 0 and n > 2:
            m[1] = m[0]                      # exact tie
        m = m / m.sum()
        tau = float(rng.random())
        sel, _, _ = O.sparse_select(m[None, :], tau=[tau])
        k = len(sel[0])
        best = min(len(c) for r in range(1, n + 1) for c in itertools.combinations(range(n), r)
                   if m[list(c)].sum() >= tau)
        assert k == best
        assert m[sel[0]].sum() >= tau
        top = sorted(range(n), key=lambda b: (-m[b], b))[:k]
        assert sorted(top) == sel[0].tolist()


def test_keep_every_block_is_dense_attention():
    """tau = 1 keeps every block, and the branch is then the dense attention
    over [buffer ; local] of the main path."""
    q, km, vm = _rand((10, 2, 8), 21), _rand((300, 2, 8), 22), _rand((300, 2, 8), 23)
    kl, vl = _rand((70, 2, 8), 24), _rand((70, 2, 8), 25)
    mass = O.pooled_mass(q, km, kl)
    sel, _, _ = O.sparse_select(mass, tau=[1.0, 1.0])
    assert [len(s) for s in sel] == [len(O.key_blocks(300, 70))] * 2
    o = O.sparse_attn(q, km, vm, kl, vl, sel)
    ref, _ = O.block_attn(q, km, vm, kl, vl)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)


def test_sparse_attn_matches_torch_sdpa_on_kept_tokens():
    q, km, vm = _rand((9, 3, 8), 31), _rand((400, 3, 8), 32), _rand((400, 3, 8), 33)
    kl, vl = _rand((100, 3, 8), 34), _rand((100, 3, 8), 35)
    blocks = O.key_blocks(400, 100)
    sel = [np.array([0, 2, 4, 5]), np.array([1, 3]), np.array([3, 5])]
    o = O.sparse_attn(q, km, vm, kl, vl, sel)
    for h in range(3):
        ks, vs = [], []
        for b in sel[h]:
            seg, a, e = blocks[b]
            ks.append((km if seg == 0 else kl)[a:e, h, :])
            vs.append((vm if seg == 0 else vl)[a:e, h, :])
        kt = torch.from_numpy(np.concatenate(ks))[None, None]
        vt = torch.from_numpy(np.concatenate(vs))[None, None]
        qt = torch.from_numpy(q[:, h, :])[None, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, 0].numpy()
        np.testing.assert_allclose(o[:, h, :], ref, rtol=1e-12, atol=1e-13)


def test_peaked_head_keeps_fewer_blocks_than_uniform_head():
    """Head-adaptive sparsity: a head whose queries align with one key block
    has a larger Gini coefficient and keeps fewer blocks than a head with flat
    scores."""
    rng = np.random.default_rng(41)
    d = 16
    km = rng.standard_normal((1024, 2, d)) * 0.05
    kl = rng.standard_normal((128, 2, d)) * 0.05
    q = rng.standard_normal((128, 2, d)) * 0.05
    direction = rng.standard_normal(d)
    km[256:384, 0, :] += 3.0 * direction       # head 0: one block stands out
    q[:, 0, :] += 3.0 * direction
    mass = O.pooled_mass(q, km, kl)
    sel, g, tau = O.sparse_select(mass)
    assert g[0] > g[1]
    assert len(sel[0]) < len(sel[1])
    assert 2 in sel[0]
