"""GPU parity of the FP8 E4M3 page codec (compressed DRAM tier) through the C
ABI against the oracle: codes and scales bit-exact (both sides divide in IEEE
fp32 and round to nearest even), decoded bf16 bit-exact, the gather-decode of
selected pages from pinned host memory bit-exact, a bad page index reported,
and attention over FP8-stored pages close to attention over the bf16 pages."""

import numpy as np
import pytest
import torch

import oracle as O
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
from tests._util import f64, np_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rows(n, H, d, seed):
    x = synth.normal((n, H, d), synth.seed_of("fp8", seed))
    scale = torch.exp(synth.normal((n, H, 1), synth.seed_of("fp8", seed, "s")) * 3.0)
    x = x * scale
    x[1, 0] = 0.0                                       # a zero row
    x[2, 0, 5] = -0.0
    x[3, 0] = x[3, 0] * 1e-3                            # values that reach subnormal codes
    x[3, 0, 0] = 100.0
    # row maxima of 1e-38 (bf16 subnormals: the division fallbacks), 1e-32 (a
    # tiny row maximum with a normal scale) and 3e38 (near the top of the bf16
    # range; finite, as the codec's inputs must be)
    for i, top in ((4, 1e-38), (5, 1e-32), (6, 3e38)):
        x[i, 0] = x[i, 0] / x[i, 0].abs().max() * top
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("d,n,H", [(64, 300, 3), (128, 300, 3), (256, 300, 3), (128, 301, 3),
                                   (64, 7, 1)])
def test_encode_decode_bitexact(d, n, H):
    """Whole and ragged row counts (the kernels take four rows per warp step)."""
    x = _rows(n, H, d, d + n)
    codes = torch.empty((n, H, d), dtype=torch.uint8, device=DEV)
    scales = torch.empty((n, H), dtype=torch.float32, device=DEV)
    wa.wa_fp8_encode(x.to(DEV), codes, scales)
    out = torch.empty((n, H, d), dtype=torch.bfloat16, device=DEV)
    wa.wa_fp8_decode(codes, scales, out)
    wa.wa_check()
    rc, rs = O.fp8_encode_rows(np_of(x))
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)
    ref = O.bf16_bits(O.fp8_decode_rows(rc, rs))
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), ref)


def test_gather_decode_from_pinned_pages():
    n_pages, P, H, d = 6, 300, 4, 128
    k = _rows(n_pages * P, H, d, 7).to(DEV)
    codes = torch.empty((n_pages, P, H, d), dtype=torch.uint8).pin_memory()
    scales = torch.empty((n_pages, P, H), dtype=torch.float32).pin_memory()
    wa.wa_fp8_encode(k, codes, scales)        # written straight into pinned host memory
    wa.wa_check()
    rc, rs = O.fp8_encode_rows(np_of(k))
    assert np.array_equal(codes.numpy().reshape(rc.shape), rc)
    idx = torch.tensor([5, 0, 3], dtype=torch.int32, device=DEV)
    out = torch.empty((3 * P, H, d), dtype=torch.bfloat16, device=DEV)
    wa.wa_gather_pages_fp8(codes, scales, idx, out)
    wa.wa_check()
    dec = O.fp8_decode_rows(rc, rs).reshape(n_pages, P, H, d)
    ref = O.bf16_bits(np.concatenate([dec[j] for j in (5, 0, 3)]))
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), ref)


def test_gather_decode_bad_index():
    codes = torch.zeros((2, 16, 1, 128), dtype=torch.uint8, device=DEV) + 0x38   # all 1.0
    scales = torch.ones((2, 16, 1), dtype=torch.float32, device=DEV)
    out = torch.full((32, 1, 128), 3.0, dtype=torch.bfloat16, device=DEV)
    wa.wa_gather_pages_fp8(codes, scales, torch.tensor([1, 2], dtype=torch.int32, device=DEV), out)
    with pytest.raises(wa.WaError) as e:
        wa.wa_check()
    assert e.value.status == 5
    assert torch.all(out[:16] == 1.0) and torch.count_nonzero(out[16:]) == 0
    wa.wa_check()


def test_attention_over_fp8_pages_close_to_bf16():
    """Quality of the compressed tier on N(0,1) pages: attention over the
    decoded pages against attention over the originals (not a parity bar: the
    codec is lossy by design, 3 mantissa bits)."""
    H, P = 12, 2048
    q = synth.normal((512, H, 128), synth.seed_of("fp8q"), DEV, torch.bfloat16)
    k = synth.normal((4 * P, H, 128), synth.seed_of("fp8k"), DEV, torch.bfloat16)
    v = synth.normal((4 * P, H, 128), synth.seed_of("fp8v"), DEV, torch.bfloat16)
    kc = torch.empty((4 * P, H, 128), dtype=torch.uint8, device=DEV)
    ks = torch.empty((4 * P, H), dtype=torch.float32, device=DEV)
    vc, vs = torch.empty_like(kc), torch.empty_like(ks)
    wa.wa_fp8_encode(k, kc, ks)
    wa.wa_fp8_encode(v, vc, vs)
    kd, vd = torch.empty_like(k), torch.empty_like(v)
    wa.wa_fp8_decode(kc, ks, kd)
    wa.wa_fp8_decode(vc, vs, vd)
    o1 = torch.empty((512, H, 128), dtype=torch.float32, device=DEV)
    o2 = torch.empty_like(o1)
    wa.wa_block_attn(q, k, v, None, None, o1)
    wa.wa_block_attn(q, kd, vd, None, None, o2)
    wa.wa_check()
    err = (o1 - o2).abs()
    assert err.max().item() < 2e-2 and err.mean().item() < 2e-3, (err.max().item(), err.mean().item())


def test_full_size_pages_sampled():
    """Two pages at the workload's full size (12,480 tokens x 12 heads x 128):
    codes, scales and decoded values on a sample of 512 (token, head) rows plus
    the first and last, against the oracle."""
    P, H, d = 12480, 12, 128
    x = synth.normal((2 * P, H, d), synth.seed_of("fp8full"), DEV, torch.bfloat16)
    codes = torch.empty((2 * P, H, d), dtype=torch.uint8, device=DEV)
    scales = torch.empty((2 * P, H), dtype=torch.float32, device=DEV)
    out = torch.empty_like(x)
    wa.wa_fp8_encode(x, codes, scales)
    wa.wa_fp8_decode(codes, scales, out)
    wa.wa_check()
    rng = np.random.default_rng(4)
    t = torch.from_numpy(np.concatenate([[0, 2 * P - 1], rng.integers(0, 2 * P, 512)])).to(DEV)
    rc, rs = O.fp8_encode_rows(np_of(x[t]))
    assert np.array_equal(scales[t].cpu().numpy(), rs)
    assert np.array_equal(codes[t].cpu().numpy(), rc)
    ref = O.bf16_bits(O.fp8_decode_rows(rc, rs))
    assert np.array_equal(out[t].view(torch.int16).cpu().numpy().view(np.uint16), ref)
