"""GPU parity of the Linformer-style low-rank branch and its gate fusion
(WorldAttention review page, HSA section), through the C ABI, against the
fp64 oracle; fp32 output, bf16 tolerances (max|err| <= 1e-2, mean <= 1e-3)."""

import numpy as np
import pytest
import torch

import oracle as O
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
from tests._util import assert_attn_close, f64, np_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(tag, n_q, n_main, n_loc, H, rank, device="cpu"):
    s = lambda t: synth.seed_of("lin", tag, t)  # noqa: E731
    g = lambda shape, t, std=1.0: synth.normal(shape, s(t), device, torch.bfloat16, std=std)  # noqa: E731
    L = n_main + n_loc
    c = dict(q=g((n_q, H, 128), "q"), km=g((n_main, H, 128), "km"), vm=g((n_main, H, 128), "vm"),
             kl=g((n_loc, H, 128), "kl") if n_loc else None,
             vl=g((n_loc, H, 128), "vl") if n_loc else None,
             ek=g((H, L, rank), "ek", L ** -0.5), ev=g((H, L, rank), "ev", L ** -0.5))
    return c


def _gpu(c, accumulate, w_attn=None, w_lin=None, o_init=None):
    d = lambda t: None if t is None else t.to(DEV)  # noqa: E731
    q = d(c["q"])
    o = torch.zeros(q.shape, dtype=torch.float32, device=DEV) if o_init is None else o_init.clone()
    wa.wa_linear_branch(q, d(c["km"]), d(c["vm"]), d(c["kl"]), d(c["vl"]), d(c["ek"]), d(c["ev"]),
                        o, d(w_attn), d(w_lin), accumulate=accumulate)
    wa.wa_check()
    return o


def _oracle_lin(c, rows=None):
    kcat = np.concatenate([np_of(c["km"])] + ([np_of(c["kl"])] if c["kl"] is not None else []))
    vcat = np.concatenate([np_of(c["vm"])] + ([np_of(c["vl"])] if c["vl"] is not None else []))
    return O.linear_branch(np_of(c["q"]), kcat, vcat, np_of(c["ek"]), np_of(c["ev"]), rows=rows)


@pytest.mark.parametrize("n_q,n_main,n_loc,H,rank", [
    (300, 1000, 77, 2, 256),      # ragged main tail, ragged local tail
    (130, 640, 0, 1, 128),        # main only, one rank block
    (64, 0, 333, 3, 384),         # local only, three rank blocks (512 TMEM columns)
    (200, 2000, 130, 2, 512),     # four rank blocks, two ring stages
])
def test_linear_branch_alone(n_q, n_main, n_loc, H, rank):
    c = _case(f"{n_q}-{n_main}-{rank}", n_q, n_main, n_loc, H, rank)
    o = _gpu(c, accumulate=False)
    ref = _oracle_lin(c)
    assert_attn_close(o, ref, torch.bfloat16, f"linear r={rank}")


def test_linear_branch_fused_with_attention_weights():
    """o = w_attn[h] * O_attn + w_lin[h] * O_lin with per-head weights, the
    attention output coming from wa_block_attn in the same buffer."""
    c = _case("fused", 250, 700, 90, 3, 256)
    d = lambda t: None if t is None else t.to(DEV)  # noqa: E731
    o = torch.empty(c["q"].shape, dtype=torch.float32, device=DEV)
    wa.wa_block_attn(d(c["q"]), d(c["km"]), d(c["vm"]), d(c["kl"]), d(c["vl"]), o)
    w_a = torch.tensor([0.5, 1.0, 2.0], dtype=torch.float32)
    w_l = torch.tensor([0.5, 1.0, -1.0], dtype=torch.float32)
    o = _gpu(c, accumulate=True, w_attn=w_a, w_lin=w_l, o_init=o)
    ref_attn, _ = O.block_attn(np_of(c["q"]), np_of(c["km"]), np_of(c["vm"]), np_of(c["kl"]),
                               np_of(c["vl"]))
    ref = O.fuse_branches(ref_attn, _oracle_lin(c), w_a.numpy(), w_l.numpy())
    assert_attn_close(o, ref, torch.bfloat16, "fused weights")
    # default weights (NULL) = equal-weight sum
    o2 = torch.empty_like(o)
    wa.wa_block_attn(d(c["q"]), d(c["km"]), d(c["vm"]), d(c["kl"]), d(c["vl"]), o2)
    o2 = _gpu(c, accumulate=True, o_init=o2)
    assert_attn_close(o2, O.fuse_branches(ref_attn, _oracle_lin(c)), torch.bfloat16, "equal weight")


def test_linear_branch_identity_projection_equals_dense_attention():
    """r = L = 128 and E = I: the low-rank branch is dense attention over the
    same 128 keys, so it must agree with wa_block_attn (and the oracle)."""
    H, L = 2, 128
    c = _case("eye", 200, L, 0, H, 128)
    eye = torch.eye(L, dtype=torch.bfloat16).expand(H, L, L).contiguous()
    c["ek"], c["ev"] = eye, eye.clone()
    o_lin = _gpu(c, accumulate=False)
    o_att = torch.empty_like(o_lin)
    wa.wa_block_attn(c["q"].to(DEV), c["km"].to(DEV), c["vm"].to(DEV), None, None, o_att)
    wa.wa_check()
    ref, _ = O.block_attn(np_of(c["q"]), np_of(c["km"]), np_of(c["vm"]), None, None)
    assert_attn_close(o_lin, ref, torch.bfloat16, "E = I")
    assert np.abs(f64(o_lin) - f64(o_att)).max() <= 1e-2


def test_linear_branch_worldattention_hybrid_shape_sampled():
    """Full hybrid shape: L = 49,920 retrieved + 4,680 local, rank 256,
    12 heads, E ~ N(0, 1/L) in bf16; fused with the dense branch at equal
    weight; oracle on 24 sampled rows."""
    H, n_q, n_main, n_loc, rank = 12, 4680, 49920, 4680, 256
    c = _case("hybrid", n_q, n_main, n_loc, H, rank, device=DEV)
    o = torch.empty(c["q"].shape, dtype=torch.float32, device=DEV)
    wa.wa_block_attn(c["q"], c["km"], c["vm"], c["kl"], c["vl"], o)
    o = _gpu(c, accumulate=True, o_init=o)
    assert torch.isfinite(o).all()
    rows = np.concatenate([np.arange(0, n_q, 211), [4679]])[:24]
    ref_attn, _ = O.block_attn(np_of(c["q"]), np_of(c["km"]), np_of(c["vm"]), np_of(c["kl"]),
                               np_of(c["vl"]), rows=rows)
    ref = O.fuse_branches(ref_attn, _oracle_lin(c, rows=rows))
    assert_attn_close(o[torch.from_numpy(rows).to(DEV)], ref, torch.bfloat16, "hybrid full shape")
