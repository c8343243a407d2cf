"""GPU parity of the NVFP4 page codec (libwa wa_nvfp4_*), the compressed DRAM
tier's FP4 form: E2M1 codes, E4M3 block scales, fp32 row scales and the
decoded bf16 values bit-exact against the oracle, whole and ragged row
counts, pages encoded into and gathered from pinned host memory, bad gather
indices; and the tier's effect on attention measured against the oracle's
own prediction on the same inputs."""

import numpy as np
import pytest
import torch

import oracle as O
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
from tests._util import BF16_MAX_ABS, BF16_MEAN_ABS, np_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rows(n, H, d, seed):
    x = synth.normal((n, H, d), synth.seed_of("fp4", seed))
    scale = torch.exp(synth.normal((n, H, 1), synth.seed_of("fp4", seed, "s")) * 3.0)
    block = torch.exp(synth.normal((n, H, d // 16, 1), synth.seed_of("fp4", seed, "b")) * 1.5)
    x = (x.reshape(n, H, d // 16, 16) * block).reshape(n, H, d) * scale
    x[1, 0] = 0.0                                       # a zero row
    x[2, 0, 5] = -0.0
    x[2, 0, 16:32] = 0.0                                # a zero block
    x[3, 0] = x[3, 0] * 1e-3                            # tiny values next to a large one
    x[3, 0, 0] = 100.0
    # row maxima of 1e-38 (bf16 subnormals: the division fallbacks), 1e-32 (a
    # tiny row maximum with a normal scale) and 3e38 (near the top of the bf16
    # range; finite, as the codec's inputs must be)
    for i, top in ((4, 1e-38), (5, 1e-32), (6, 3e38)):
        x[i, 0] = x[i, 0] / x[i, 0].abs().max() * top
    return x.to(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("d,n,H", [(64, 300, 3), (128, 300, 3), (256, 300, 3), (128, 301, 3),
                                   (64, 7, 1)])
def test_encode_decode_bitexact(d, n, H):
    """Whole and ragged row counts (the kernels take four rows per warp step)."""
    x = _rows(n, H, d, d + n)
    codes = torch.empty((n, H, d // 2), dtype=torch.uint8, device=DEV)
    bsc = torch.empty((n, H, d // 16), dtype=torch.uint8, device=DEV)
    rsc = torch.empty((n, H), dtype=torch.float32, device=DEV)
    wa.wa_nvfp4_encode(x.to(DEV), codes, bsc, rsc)
    out = torch.empty((n, H, d), dtype=torch.bfloat16, device=DEV)
    wa.wa_nvfp4_decode(codes, bsc, rsc, out)
    wa.wa_check()
    rc, rb, rg = O.nvfp4_encode_rows(np_of(x))
    assert np.array_equal(rsc.cpu().numpy(), rg)
    assert np.array_equal(bsc.cpu().numpy(), rb)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(_bits(out), O.bf16_bits(O.nvfp4_decode_rows(rc, rb, rg)))


def test_gather_decode_from_pinned_pages():
    n_pages, P, H, d = 6, 300, 4, 128
    k = _rows(n_pages * P, H, d, 7).to(DEV)
    codes = torch.empty((n_pages, P, H, d // 2), dtype=torch.uint8).pin_memory()
    bsc = torch.empty((n_pages, P, H, d // 16), dtype=torch.uint8).pin_memory()
    rsc = torch.empty((n_pages, P, H), dtype=torch.float32).pin_memory()
    wa.wa_nvfp4_encode(k, codes, bsc, rsc)      # written straight into pinned host memory
    wa.wa_check()
    rc, rb, rg = O.nvfp4_encode_rows(np_of(k))
    assert np.array_equal(codes.numpy().reshape(rc.shape), rc)
    assert np.array_equal(bsc.numpy().reshape(rb.shape), rb)
    idx = torch.tensor([5, 0, 3], dtype=torch.int32, device=DEV)
    out = torch.empty((3 * P, H, d), dtype=torch.bfloat16, device=DEV)
    wa.wa_gather_pages_nvfp4(codes, bsc, rsc, idx, out)
    wa.wa_check()
    dec = O.nvfp4_decode_rows(rc, rb, rg).reshape(n_pages, P, H, d)
    ref = O.bf16_bits(np.concatenate([dec[j] for j in (5, 0, 3)]))
    assert np.array_equal(_bits(out), ref)


def test_gather_decode_bad_index():
    # every code 0x22 (1.0 in both nibbles), block scale 0x38 (E4M3 1.0), row scale 1
    codes = torch.full((2, 16, 1, 64), 0x22, dtype=torch.uint8, device=DEV)
    bsc = torch.full((2, 16, 1, 8), 0x38, dtype=torch.uint8, device=DEV)
    rsc = torch.ones((2, 16, 1), dtype=torch.float32, device=DEV)
    out = torch.full((32, 1, 128), 3.0, dtype=torch.bfloat16, device=DEV)
    wa.wa_gather_pages_nvfp4(codes, bsc, rsc, torch.tensor([1, 2], dtype=torch.int32, device=DEV),
                             out)
    with pytest.raises(wa.WaError) as e:
        wa.wa_check()
    assert e.value.status == 5
    assert torch.all(out[:16] == 1.0) and torch.count_nonzero(out[16:]) == 0
    wa.wa_check()


def test_attention_over_nvfp4_pages():
    """Attention over NVFP4-stored N(0,1) pages: the GPU result equals the
    oracle's attention over the oracle-decoded pages (attention tolerance), and
    its distance from attention over the bf16 pages is the oracle's predicted
    distance on the same inputs (within the same tolerance).  The codec is
    lossy by design (E2M1: 3 magnitude bits below the block scale)."""
    H, NK, NQ, d = 4, 4096, 96, 128
    q = synth.normal((NQ, H, d), synth.seed_of("fp4q"), DEV, torch.bfloat16)
    k = synth.normal((NK, H, d), synth.seed_of("fp4k"), DEV, torch.bfloat16)
    v = synth.normal((NK, H, d), synth.seed_of("fp4v"), DEV, torch.bfloat16)
    dec = []
    for x in (k, v):
        c = torch.empty((NK, H, d // 2), dtype=torch.uint8, device=DEV)
        b = torch.empty((NK, H, d // 16), dtype=torch.uint8, device=DEV)
        r = torch.empty((NK, H), dtype=torch.float32, device=DEV)
        wa.wa_nvfp4_encode(x, c, b, r)
        y = torch.empty_like(x)
        wa.wa_nvfp4_decode(c, b, r, y)
        dec.append(y)
    o_bf16 = torch.empty((NQ, H, d), dtype=torch.float32, device=DEV)
    o_fp4 = torch.empty_like(o_bf16)
    wa.wa_block_attn(q, k, v, None, None, o_bf16)
    wa.wa_block_attn(q, dec[0], dec[1], None, None, o_fp4)
    wa.wa_check()
    kd = O.bf16_bits(O.nvfp4_decode_rows(*O.nvfp4_encode_rows(np_of(k))))
    vd = O.bf16_bits(O.nvfp4_decode_rows(*O.nvfp4_encode_rows(np_of(v))))
    assert np.array_equal(_bits(dec[0]), kd) and np.array_equal(_bits(dec[1]), vd)
    ref_fp4, _ = O.block_attn(np_of(q), kd, vd, None, None)
    ref_bf16, _ = O.block_attn(np_of(q), np_of(k), np_of(v), None, None)
    err = np.abs(o_fp4.double().cpu().numpy() - ref_fp4)
    assert err.max() <= BF16_MAX_ABS and err.mean() <= BF16_MEAN_ABS
    dist_gpu = np.abs(o_fp4.double().cpu().numpy() - o_bf16.double().cpu().numpy())
    dist_ref = np.abs(ref_fp4 - ref_bf16)
    assert abs(dist_gpu.mean() - dist_ref.mean()) <= BF16_MEAN_ABS
    assert dist_gpu.max() <= dist_ref.max() + BF16_MAX_ABS


def test_full_size_pages_sampled():
    """Two pages at the workload's full size (12,480 tokens x 12 heads x 128):
    row scales, block scales, codes and decoded values on a sample of 512
    (token, head) rows plus the first and last, against the oracle."""
    P, H, d = 12480, 12, 128
    x = synth.normal((2 * P, H, d), synth.seed_of("fp4full"), DEV, torch.bfloat16)
    codes = torch.empty((2 * P, H, d // 2), dtype=torch.uint8, device=DEV)
    bsc = torch.empty((2 * P, H, d // 16), dtype=torch.uint8, device=DEV)
    rsc = torch.empty((2 * P, H), dtype=torch.float32, device=DEV)
    out = torch.empty_like(x)
    wa.wa_nvfp4_encode(x, codes, bsc, rsc)
    wa.wa_nvfp4_decode(codes, bsc, rsc, out)
    wa.wa_check()
    rng = np.random.default_rng(3)
    t = np.concatenate([[0, 2 * P - 1], rng.integers(0, 2 * P, 512)])
    xs = np_of(x[torch.from_numpy(t).to(DEV)])
    rc, rb, rg = O.nvfp4_encode_rows(xs)
    tt = torch.from_numpy(t).to(DEV)
    assert np.array_equal(rsc[tt].cpu().numpy(), rg)
    assert np.array_equal(bsc[tt].cpu().numpy(), rb)
    assert np.array_equal(codes[tt].cpu().numpy(), rc)
    assert np.array_equal(_bits(out[tt]), O.bf16_bits(O.nvfp4_decode_rows(rc, rb, rg)))
