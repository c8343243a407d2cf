"""wa_select_pages_noalloc: the page retrieval for callers that must not
allocate device memory while running (a server that has given all free HBM
to its own pool, or a latency-critical loop that cannot afford the stall of a
cudaMalloc).  Its scratch is a fixed array inside the library, so its results
must equal those of wa_select_pages, call after call, even though every call
reuses that array with the previous call's contents still in it.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc_fn():
    fn = wa.load().wa_select_pages_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.restype = I
    fn.argtypes = [P, I, I, I, I, P, I, P, P, I, I, I, I, P, P, P, P]
    return fn


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _inputs(tag, n_q, n_heads, head_dim, n_pages, n_chunks, ppc, pdim, dtype):
    s = lambda t: synth.seed_of("noalloc", tag, t)  # noqa: E731
    q = synth.normal((n_q, n_heads, head_dim), s("q"), DEV, dtype)
    kbar = synth.normal((n_pages, n_heads, head_dim), s("kbar"), DEV, std=0.05)
    pc = synth.normal((n_chunks, pdim), s("pc"), DEV) if n_chunks else None
    cur = (pc[n_chunks // 2] + 0.5 * synth.normal((pdim,), s("cur"), DEV)) if n_chunks else None
    return q, kbar, cur, pc


def _both(fn, q, kbar, cur, pc, ppc, k_p):
    """Run the allocating and the non-allocating entry point on the same inputs."""
    n_q, h, d = q.shape
    n_chunks, pdim = (pc.shape if pc is not None else (0, 0))
    dt = 1 if q.dtype == torch.bfloat16 else 0
    out = []
    for use_noalloc in (False, True):
        idx = torch.full((k_p,), -1, dtype=torch.int32, device=DEV)
        sc = torch.full((k_p,), float("nan"), dtype=torch.float32, device=DEV)
        ch = torch.full((1,), -9, dtype=torch.int32, device=DEV)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        args = (_p(q), dt, n_q, h, d, _p(kbar), kbar.shape[0], _p(cur), _p(pc), n_chunks, pdim,
                ppc, k_p, _p(idx), _p(sc), _p(ch), stream)
        if use_noalloc:
            st = fn(*args)
            assert st == 0, wa.load().wa_strerror(st)
        else:
            wa.wa_select_pages(q, kbar, cur, pc, ppc, k_p, idx, sc, ch)
        wa.wa_check()
        out.append((idx.cpu().numpy(), sc.cpu().numpy(), int(ch.item())))
    return out


def test_noalloc_select_matches_allocating_entry_point_twice():
    fn = _noalloc_fn()
    # call 1: the one-layer WorldAttention shape (12 heads, d 128, 40 pages in
    # 5 chunks, prompt dim 4096, top-4), bf16 queries
    q, kbar, cur, pc = _inputs("a", 4680, 12, 128, 40, 5, 8, 4096, torch.bfloat16)
    (i0, s0, c0), (i1, s1, c1) = _both(fn, q, kbar, cur, pc, 8, 4)
    assert c0 == c1 == 2
    assert i0.tolist() == i1.tolist() and all(16 <= j < 24 for j in i0)
    assert np.abs(s0 - s1).max() <= 1e-6
    # call 2, right after: other shapes and no prompt stage (the array still
    # holds call 1's partial sums and ticket)
    q, kbar, cur, pc = _inputs("b", 1000, 4, 64, 300, 0, 1, 0, torch.float32)
    (i0, s0, c0), (i1, s1, c1) = _both(fn, q, kbar, cur, pc, 1, 7)
    assert c0 == c1 == -1
    assert i0.tolist() == i1.tolist()
    assert np.abs(s0 - s1).max() <= 1e-6
    # and a third call repeating the first inputs' shape with fresh values
    q, kbar, cur, pc = _inputs("c", 4680, 12, 128, 40, 5, 8, 4096, torch.bfloat16)
    (i0, s0, c0), (i1, s1, c1) = _both(fn, q, kbar, cur, pc, 8, 4)
    assert c0 == c1 and i0.tolist() == i1.tolist() and np.abs(s0 - s1).max() <= 1e-6


def test_noalloc_select_rejects_requests_beyond_its_array():
    fn = _noalloc_fn()
    # 64 heads scoring 8,192 pages without a prompt stage need 64 x 8,192 floats
    # of per-head partial scores plus 5 row blocks x 8,192 of query partials:
    # more than the 2 MiB array (the buffers are real, though nothing runs)
    q = torch.empty((9728, 64, 128), dtype=torch.float32, device=DEV)
    kbar = torch.empty((8192, 64, 128), dtype=torch.float32, device=DEV)
    idx = torch.empty(2, dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = fn(_p(q), 0, 9728, 64, 128, _p(kbar), 8192, None, None, 0, 0, 1, 2, _p(idx), None, None,
            stream)
    assert st == 2   # WA_ERR_SHAPE, nothing enqueued


_FRESH = r'''
import ctypes, sys, torch
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
lib = wa.load()
fn = lib.wa_select_pages_noalloc
P, I = ctypes.c_void_p, ctypes.c_int
fn.restype = I
fn.argtypes = [P, I, I, I, I, P, I, P, P, I, I, I, I, P, P, P, P]
p = lambda t: ctypes.c_void_p(t.data_ptr())
s = lambda t: synth.seed_of("noalloc_fresh", t)
q = synth.normal((4680, 12, 128), s("q"), "cuda", torch.bfloat16)
kbar = synth.normal((40, 12, 128), s("kbar"), "cuda", std=0.05)
pc = synth.normal((5, 4096), s("pc"), "cuda")
cur = (pc[3] + 0.5 * synth.normal((4096,), s("cur"), "cuda")).contiguous()
idx = torch.full((4,), -1, dtype=torch.int32, device="cuda")
ch = torch.full((1,), -9, dtype=torch.int32, device="cuda")
stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
args = (p(q), 1, 4680, 12, 128, p(kbar), 40, p(cur), p(pc), 5, 4096, 8, 4, p(idx), None, p(ch),
        stream)
torch.cuda.synchronize()
before = wa.wa_scratch_bytes()
assert fn(*args) == 0
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
for _ in range(5):
    assert fn(*args) == 0
torch.cuda.synchronize()
free2 = torch.cuda.mem_get_info()[0]
print(before, wa.wa_scratch_bytes(), free1, free2, *idx.cpu().tolist(), int(ch.item()))
'''


def test_noalloc_select_allocates_nothing_in_a_fresh_process():
    """In a process where the library has made no allocation yet, calls of
    the non-allocating entry point leave the library's arena unallocated and
    the device's free memory unchanged (after the first call, which loads the
    library's kernels); its indices equal the allocating entry point's."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH], cwd=root, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    before, after, free1, free2, *rest = (int(x) for x in r.stdout.split())
    assert before == 0 and after == 0
    assert free1 == free2
    idx, ch = rest[:4], rest[4]
    s = lambda t: synth.seed_of("noalloc_fresh", t)  # noqa: E731
    q = synth.normal((4680, 12, 128), s("q"), DEV, torch.bfloat16)
    kbar = synth.normal((40, 12, 128), s("kbar"), DEV, std=0.05)
    pc = synth.normal((5, 4096), s("pc"), DEV)
    cur = (pc[3] + 0.5 * synth.normal((4096,), s("cur"), DEV)).contiguous()
    ref_idx = torch.full((4,), -1, dtype=torch.int32, device=DEV)
    ref_ch = torch.full((1,), -9, dtype=torch.int32, device=DEV)
    wa.wa_select_pages(q, kbar, cur, pc, 8, 4, ref_idx, chunk_out=ref_ch)
    wa.wa_check()
    assert ch == int(ref_ch.item()) == 3
    assert idx == ref_idx.cpu().tolist()
