"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching the
GPU (no compute call runs here)."""

import ctypes
import os
import re

import pytest

import sparse_kv_cache_page_gb300 as wa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "wa.h")).read()
    return sorted(set(re.findall(r"^\s*(?:wa_status|const char\*)\s+(wa_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(wa.lib_path()):
        from sparse_kv_cache_page_gb300 import build
        build.build()
    return wa.load()


def test_header_declares_the_five_calls():
    names = _declared()
    for n in ("wa_page_summarize", "wa_select_pages", "wa_gather_pages", "wa_block_attn",
              "wa_linear_branch"):
        assert n in names
    assert sorted(wa.EXPORTED_SYMBOLS) == names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), n
    assert wa.wa_version().startswith("wa ")
    for st in range(10):
        assert lib.wa_strerror(st)


def test_host_validation_without_gpu(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)           # never dereferenced: validation fails first
    mis = P(0x1004)            # misaligned
    # NULL pointers / bad sizes -> WA_ERR_INVALID_ARG (1)
    assert lib.wa_page_summarize(None, 1, 1, 1, 1, 128, fake, None) == 1
    assert lib.wa_page_summarize(fake, 1, 0, 1, 1, 128, fake, None) == 1
    # bad dtype -> WA_ERR_DTYPE (3); unsupported row width -> WA_ERR_SHAPE (2)
    assert lib.wa_page_summarize(fake, 7, 1, 1, 1, 128, fake, None) == 3
    assert lib.wa_page_summarize(fake, 1, 1, 1, 1, 3, fake, None) == 2
    # misaligned -> WA_ERR_ALIGN (4)
    assert lib.wa_page_summarize(mis, 1, 1, 1, 1, 128, fake, None) == 4
    # k_p above the candidates -> WA_ERR_INVALID_ARG
    assert lib.wa_select_pages(fake, 1, 10, 1, 128, fake, 8, None, None, 0, 0, 4, 9, fake, None,
                               None, None) == 1
    assert lib.wa_select_pages(fake, 1, 10, 1, 128, fake, 8, fake, fake, 2, 16, 4, 5, fake, None,
                               None, None) == 1
    # prompt chunks claiming more pages than exist
    assert lib.wa_select_pages(fake, 1, 10, 1, 128, fake, 8, fake, fake, 3, 16, 4, 2, fake, None,
                               None, None) == 1
    # attention: both segments empty; bf16 head_dim != 128 -> SHAPE
    assert lib.wa_block_attn(fake, 4, None, None, 0, None, None, 0, 1, 1, 128, ctypes.c_float(0),
                             fake, 1, None, None) == 1
    assert lib.wa_block_attn(fake, 4, fake, fake, 8, None, None, 0, 1, 1, 64, ctypes.c_float(0),
                             fake, 1, None, None) == 2
    assert lib.wa_block_attn(fake, 4, fake, fake, 8, None, None, 0, 0, 1, 260, ctypes.c_float(0),
                             fake, 0, None, None) == 2
    # fp32 inputs with a bf16 output -> WA_ERR_DTYPE
    assert lib.wa_block_attn(fake, 4, fake, fake, 8, None, None, 0, 0, 1, 64, ctypes.c_float(0),
                             fake, 1, None, None) == 3
    # gather: v pointer without v buffer
    assert lib.wa_gather_pages(fake, fake, 1, 4, 8, 1, 128, fake, None, 2, fake, None, None) == 1
    # gather + attention: fp32 inputs with a bf16 output -> DTYPE; bf16 pages not a multiple of
    # 8 rows, bf16 head_dim != 128, fp32 head_dim over 256 -> SHAPE; a key buffer without a value
    # buffer, no indices -> INVALID_ARG; misaligned -> ALIGN
    f0 = ctypes.c_float(0)
    assert lib.wa_gather_attn(fake, 4, fake, fake, 8, 64, fake, 2, 0, None, None, None, None, 0,
                              0, 1, 128, f0, fake, 1, None, None) == 3
    assert lib.wa_gather_attn(fake, 4, fake, fake, 8, 100, fake, 2, 0, None, None, None, None, 0,
                              0, 1, 260, f0, fake, 0, None, None) == 2
    assert lib.wa_gather_attn(fake, 4, fake, fake, 8, 100, fake, 2, 0, None, None, None, None, 0,
                              1, 1, 128, f0, fake, 1, None, None) == 2
    assert lib.wa_gather_attn(fake, 4, fake, fake, 8, 12, fake, 2, 0, None, None, None, None, 0,
                              1, 1, 128, f0, fake, 1, None, None) == 2
    assert lib.wa_gather_attn(fake, 4, fake, fake, 8, 64, fake, 2, 0, None, None, None, None, 0,
                              1, 1, 64, f0, fake, 1, None, None) == 2
    assert lib.wa_gather_attn(fake, 4, fake, fake, 8, 64, fake, 2, 0, fake, None, None, None, 0,
                              1, 1, 128, f0, fake, 1, None, None) == 1
    assert lib.wa_gather_attn(fake, 4, fake, fake, 8, 64, None, 2, 0, None, None, None, None, 0,
                              1, 1, 128, f0, fake, 1, None, None) == 1
    assert lib.wa_gather_attn(fake, 4, mis, fake, 8, 64, fake, 2, 0, None, None, None, None, 0,
                              1, 1, 128, f0, fake, 1, None, None) == 4
    # linear branch: fp32 not supported, bad rank
    assert lib.wa_linear_branch(fake, 4, fake, fake, 8, None, None, 0, fake, fake, 256, 0, 1, 128,
                                ctypes.c_float(0), None, None, 1, fake, 0, None) == 3
    assert lib.wa_linear_branch(fake, 4, fake, fake, 8, None, None, 0, fake, fake, 100, 1, 1, 128,
                                ctypes.c_float(0), None, None, 1, fake, 1, None) == 2


def test_fault_and_wait_limit_setters(lib):
    """The fault-injection and wait-limit setters are host-only: they accept
    the documented modes, refuse others, and restore the defaults."""
    for mode in (wa.WA_FAULT_ALLOC, wa.WA_FAULT_COPY, wa.WA_FAULT_WAIT, wa.WA_FAULT_NONE):
        assert lib.wa_set_fault(mode) == 0
    assert lib.wa_set_fault(4) == 1 and lib.wa_set_fault(-1) == 1
    assert lib.wa_set_wait_limit_ns(1000) == 0
    assert lib.wa_set_wait_limit_ns(0) == 0          # back to the 4 s default
    assert lib.wa_scratch_bytes(None) == 1


def test_library_loads_with_a_fault_mode_in_the_environment():
    """The library reads WA_FAULT when it loads (its effect is checked on the
    GPU); loading with it set works and the setter still behaves."""
    import subprocess
    import sys
    code = ("import ctypes, sparse_kv_cache_page_gb300 as wa; lib = wa.load(); "
            "print(lib.wa_set_fault(0), lib.wa_set_fault(9))")
    env = dict(os.environ, WA_FAULT="alloc")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split() == ["0", "1"]
