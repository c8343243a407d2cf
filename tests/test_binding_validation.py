"""Host-side checks of the Python binding (no GPU): the C ABI takes plain
pointers and cannot see buffer sizes, so the binding refuses a buffer of the
wrong dtype, size or layout before any call reaches the library."""

import pytest
import torch

import sparse_kv_cache_page_gb300 as wa

U8, F32, BF16, I32 = torch.uint8, torch.float32, torch.bfloat16, torch.int32


def _z(*shape, dtype=BF16):
    return torch.zeros(shape, dtype=dtype)


def _raises(fn, *args):
    with pytest.raises(ValueError):
        fn(*args)


def test_gather_pages_buffers():
    kp, idx = _z(3, 16, 2, 64), torch.tensor([0, 2], dtype=I32)
    _raises(wa.wa_gather_pages, kp, None, None, idx, _z(31, 2, 64), None)          # short
    _raises(wa.wa_gather_pages, kp, None, None, idx, _z(32, 2, 64, dtype=F32), None)
    _raises(wa.wa_gather_pages, kp, kp, None, idx, _z(32, 2, 64), None)            # v without buffer
    _raises(wa.wa_gather_pages, kp, _z(3, 16, 2, 32), None, idx, _z(32, 2, 64), _z(32, 2, 64))
    _raises(wa.wa_gather_pages, kp, kp, None, idx, _z(32, 2, 64), _z(30, 2, 64))
    _raises(wa.wa_gather_pages, kp, None, None, idx.long(), _z(32, 2, 64), None)


def test_gather_per_head_buffers():
    kp, idx = _z(3, 16, 2, 64), torch.zeros((2, 2), dtype=I32)
    _raises(wa.wa_gather_pages_per_head, kp, None, idx, _z(31, 2, 64), None)
    _raises(wa.wa_gather_pages_per_head, kp, kp, idx, _z(32, 2, 64), _z(32, 2, 63))
    _raises(wa.wa_gather_pages_per_head, kp, None, idx.t(), _z(32, 2, 64), None)


def test_fp8_codec_buffers():
    x = _z(10, 2, 64)
    _raises(wa.wa_fp8_encode, x, _z(10, 2, 63, dtype=U8), _z(10, 2, dtype=F32))
    _raises(wa.wa_fp8_encode, x.float(), _z(10, 2, 64, dtype=U8), _z(10, 2, dtype=F32))
    _raises(wa.wa_fp8_encode, x, _z(10, 2, 64, dtype=U8), _z(10, 1, dtype=F32))
    _raises(wa.wa_fp8_decode, _z(10, 2, 64, dtype=U8), _z(10, 2, dtype=F32), _z(11, 2, 64))
    _raises(wa.wa_fp8_decode, _z(10, 2, 64, dtype=U8), _z(10, 2, dtype=BF16), x)
    pages, idx = _z(4, 8, 2, 64, dtype=U8), torch.tensor([1, 3], dtype=I32)
    _raises(wa.wa_gather_pages_fp8, pages, _z(4, 8, 2, dtype=F32), idx, _z(15, 2, 64))
    _raises(wa.wa_gather_pages_fp8, pages, _z(4, 8, 1, dtype=F32), idx, _z(16, 2, 64))


def test_nvfp4_codec_buffers():
    x = _z(10, 2, 64)
    codes, bs, rs = _z(10, 2, 32, dtype=U8), _z(10, 2, 4, dtype=U8), _z(10, 2, dtype=F32)
    _raises(wa.wa_nvfp4_encode, x, _z(10, 2, 31, dtype=U8), bs, rs)
    _raises(wa.wa_nvfp4_encode, x, codes, _z(10, 2, 3, dtype=U8), rs)
    _raises(wa.wa_nvfp4_encode, _z(10, 2, 40), codes, bs, rs)                      # d % 16
    _raises(wa.wa_nvfp4_decode, codes, bs, rs, _z(10, 2, 64, dtype=F32))
    _raises(wa.wa_nvfp4_decode, codes, bs, _z(9, 2, dtype=F32), x)
    pages = (_z(4, 8, 2, 32, dtype=U8), _z(4, 8, 2, 4, dtype=U8), _z(4, 8, 2, dtype=F32))
    idx = torch.tensor([0, 3], dtype=I32)
    _raises(wa.wa_gather_pages_nvfp4, *pages, idx, _z(15, 2, 64))
    _raises(wa.wa_gather_pages_nvfp4, pages[0], pages[1][:, :, :, :3].contiguous(), pages[2], idx,
            _z(16, 2, 64))


def test_attention_buffers():
    q, kv = _z(8, 2, 64), _z(16, 2, 64)
    o = _z(8, 2, 64, dtype=F32)
    _raises(wa.wa_block_attn, q, kv, None, None, None, o)                          # v missing
    _raises(wa.wa_block_attn, q, kv, _z(15, 2, 64), None, None, o)                 # rows differ
    _raises(wa.wa_block_attn, q, kv, kv, _z(4, 3, 64), _z(4, 3, 64), o)            # heads differ
    _raises(wa.wa_block_attn, q, kv.float(), kv.float(), None, None, o)            # dtype
    _raises(wa.wa_block_attn, q, kv, kv, None, None, _z(8, 2, 64, dtype=torch.float16))
    _raises(wa.wa_block_attn, q, kv, kv, None, None, o, _z(2, 7, dtype=F32))       # short lse


def test_linear_branch_buffers():
    q, kv, o = _z(8, 2, 128), _z(16, 2, 128), _z(8, 2, 128, dtype=F32)
    e = _z(2, 16, 128)
    _raises(wa.wa_linear_branch, q, kv, kv, None, None, _z(2, 15, 128), _z(2, 15, 128), o)
    _raises(wa.wa_linear_branch, q, kv, kv, None, None, e, _z(2, 16, 256), o)
    _raises(wa.wa_linear_branch, q, kv, kv, None, None, e, e, o, _z(3, dtype=F32))
    _raises(wa.wa_linear_branch, q, kv, kv, None, None, e.float(), e.float(), o)


def test_gather_attn_buffers():
    q, kp = _z(20, 2, 128), _z(3, 64, 2, 128)
    idx, kl = torch.tensor([2, 0], dtype=I32), _z(8, 2, 128)
    o = _z(20, 2, 128, dtype=F32)
    buf = _z(128, 2, 128)
    ga = wa.wa_gather_attn
    _raises(ga, q, kp, kp, idx, kl, kl, o, _z(127, 2, 128), buf)                       # short buffer
    _raises(ga, q, kp, kp, idx, kl, kl, o, buf, None)                                   # k without v
    _raises(ga, q, kp, kp, idx.long(), kl, kl, o, buf, buf)                             # int64 indices
    _raises(ga, q, kp, _z(3, 64, 2, 64), idx, kl, kl, o, buf, buf)                      # v pages shape
    _raises(ga, q, kp, kp, torch.zeros((3, 2), dtype=I32), kl, kl, o, buf, buf)         # per-head rows != H
    _raises(ga, q, kp, kp, idx, kl, None, o, buf, buf)                                  # k_loc without v_loc
    _raises(ga, q, kp, kp, idx, kl, kl, _z(20, 2, 128, dtype=torch.float16), buf, buf)  # o dtype
    _raises(ga, q, kp.float(), kp.float(), idx, kl, kl, o, buf, buf)                    # pages dtype
    _raises(ga, q, kp, kp, idx, kl, kl, o, buf, buf, _z(2, 19, dtype=F32))              # short lse
