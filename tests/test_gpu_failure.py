"""Failure handling on the GPU, with every failure made on the host side:

* a bounded device wait that runs out: the attention kernel's copy producer
  withholds the query tiles (WA_FAULT_WAIT), so every wait on them reaches the
  host-set limit; the kernel records WA_ERR_TIMEOUT, drains its copies and
  MMAs, frees its tensor memory and returns; an ordinary call in the same
  process then matches the oracle;
* an allocation that fails (WA_FAULT_ALLOC): WA_ERR_OOM, nothing enqueued;
* a host-to-device page copy that fails (WA_FAULT_COPY): WA_ERR_CUDA.

No test here faults, traps or hangs the GPU: the only device-side failure is a
wait that gives up at its limit.
"""

import os
import subprocess
import sys
import time

import numpy as np
import pytest
import torch

import oracle as O
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
from tests._util import assert_attn_close, np_of

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(autouse=True)
def _defaults():
    yield
    wa.wa_set_fault(wa.WA_FAULT_NONE)
    wa.wa_set_wait_limit_ns(0)


def _attn_inputs(tag, n_q=300, n_main=1000, n_loc=100, h=2):
    g = lambda shape, t: synth.normal(shape, synth.seed_of("fail", tag, t), DEV, torch.bfloat16)  # noqa: E731
    return (g((n_q, h, 128), "q"), g((n_main, h, 128), "km"), g((n_main, h, 128), "vm"),
            g((n_loc, h, 128), "kl"), g((n_loc, h, 128), "vl"))


@pytest.mark.parametrize("split", [None, "2"])
def test_wait_limit_reached_gives_timeout_then_ordinary_calls_work(monkeypatch, split):
    if split:
        monkeypatch.setenv("WA_ATTN_SPLIT", split)
    q, km, vm, kl, vl = _attn_inputs("timeout")
    o = torch.full(q.shape, 7.0, dtype=torch.float32, device=DEV)
    wa.wa_check()
    limit_s = 0.02
    wa.wa_set_wait_limit_ns(int(limit_s * 1e9))
    wa.wa_set_fault(wa.WA_FAULT_WAIT)
    t0 = time.perf_counter()
    wa.wa_block_attn(q, km, vm, kl, vl, o)          # the launch itself succeeds
    with pytest.raises(wa.WaError) as e:
        wa.wa_check()
    elapsed = time.perf_counter() - t0
    assert e.value.status == 8                      # WA_ERR_TIMEOUT
    assert limit_s <= elapsed < 2.0, elapsed        # the host-set limit, not the 4 s default
    wa.wa_check()                                   # the status word was cleared

    wa.wa_set_fault(wa.WA_FAULT_NONE)
    wa.wa_set_wait_limit_ns(0)
    for _ in range(2):                              # the context and the counters are intact
        wa.wa_block_attn(q, km, vm, kl, vl, o)
        wa.wa_check()
        ref, _ = O.block_attn(np_of(q), np_of(km), np_of(vm), np_of(kl), np_of(vl))
        assert_attn_close(o, ref, torch.bfloat16, "after a timeout")


def test_wait_limit_in_the_fused_gather_attention():
    """The same withheld query tiles in the gather + attention launch, whose
    store warp also waits on the ring: the launch ends with WA_ERR_TIMEOUT
    (copies and stores drained), and an ordinary call then matches the
    two-launch path bit for bit."""
    q, km, vm, kl, vl = _attn_inputs("fused", n_q=600, n_main=1024, n_loc=100)
    kp, vp = km.reshape(8, 128, 2, 128), vm.reshape(8, 128, 2, 128)
    idx = torch.tensor([6, 1, 3], dtype=torch.int32, device=DEV)
    kb = torch.empty((384, 2, 128), dtype=torch.bfloat16, device=DEV)
    vb = torch.empty_like(kb)
    o = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    wa.wa_check()
    wa.wa_set_wait_limit_ns(20_000_000)
    wa.wa_set_fault(wa.WA_FAULT_WAIT)
    wa.wa_gather_attn(q, kp, vp, idx, kl, vl, o, kb, vb)
    with pytest.raises(wa.WaError) as e:
        wa.wa_check()
    assert e.value.status == 8
    wa.wa_set_fault(wa.WA_FAULT_NONE)
    wa.wa_set_wait_limit_ns(0)
    wa.wa_gather_attn(q, kp, vp, idx, kl, vl, o, kb, vb)
    wa.wa_check()
    kb2, vb2 = torch.empty_like(kb), torch.empty_like(vb)
    o2 = torch.empty_like(o)
    wa.wa_gather_pages(kp, vp, idx, None, kb2, vb2)
    wa.wa_block_attn(q, kb2, vb2, kl, vl, o2)
    wa.wa_check()
    assert torch.equal(kb, kb2) and torch.equal(vb, vb2) and torch.equal(o, o2)


def test_linear_branch_runs_under_a_short_wait_limit():
    """A limit far above the kernels' real waits changes nothing."""
    q, km, vm, kl, vl = _attn_inputs("lin", n_q=256, n_main=512, n_loc=128)
    L, r = 640, 128
    ek = synth.normal((2, L, r), synth.seed_of("fail", "ek"), DEV, torch.bfloat16, std=L ** -0.5)
    ev = synth.normal((2, L, r), synth.seed_of("fail", "ev"), DEV, torch.bfloat16, std=L ** -0.5)
    o = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    wa.wa_set_wait_limit_ns(50_000_000)
    wa.wa_linear_branch(q, km, vm, kl, vl, ek, ev, o, accumulate=False)
    wa.wa_check()
    kc = np.concatenate([np_of(km), np_of(kl)])
    vc = np.concatenate([np_of(vm), np_of(vl)])
    ref = O.linear_branch(np_of(q), kc, vc, np_of(ek), np_of(ev))
    assert_attn_close(o, ref, torch.bfloat16, "linear branch")


def test_alloc_failure_reports_oom_and_enqueues_nothing():
    kp = synth.normal((3, 64, 2, 128), synth.seed_of("fail", "alloc"), DEV, torch.bfloat16)
    kbar = torch.full((3, 2, 128), -1.0, dtype=torch.float32, device=DEV)
    wa.wa_shutdown()                                # free the arena: the next call must allocate
    assert wa.wa_scratch_bytes() == 0
    wa.wa_set_fault(wa.WA_FAULT_ALLOC)
    with pytest.raises(wa.WaError) as e:
        wa.wa_page_summarize(kp, kbar)
    assert e.value.status == 6                      # WA_ERR_OOM
    torch.cuda.synchronize()
    assert wa.wa_scratch_bytes() == 0
    assert torch.all(kbar == -1.0)
    with pytest.raises(wa.WaError) as e:
        wa.WaCache(2, 128, 64, 2, hbm_pages=4, host_pages=4, max_chunks=4)
    assert e.value.status == 6
    wa.wa_set_fault(wa.WA_FAULT_NONE)
    wa.wa_page_summarize(kp, kbar)
    wa.wa_check()
    assert wa.wa_scratch_bytes() > 0
    assert np.abs(kbar.double().cpu().numpy() - O.page_summarize(np_of(kp))).max() < 1e-6


def test_alloc_fault_from_environment_in_a_fresh_process():
    code = ("import torch, sparse_kv_cache_page_gb300 as wa\n"
            "x = torch.zeros((2, 16, 1, 128), dtype=torch.bfloat16, device='cuda')\n"
            "kb = torch.zeros((2, 1, 128), dtype=torch.float32, device='cuda')\n"
            "try:\n    wa.wa_page_summarize(x, kb)\n    print('no-error')\n"
            "except wa.WaError as e:\n    print('status', e.status)\n"
            "wa.wa_set_fault(wa.WA_FAULT_NONE)\nwa.wa_page_summarize(x, kb)\nwa.wa_check()\n"
            "print('then', wa.wa_scratch_bytes() > 0)\n")
    env = dict(os.environ, WA_FAULT="alloc")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split() == ["status", "6", "then", "True"]


def test_copy_failure_from_pinned_pages_reports_cuda_error():
    kp = synth.normal((4, 100, 2, 128), synth.seed_of("fail", "copy"), "cpu",
                      torch.bfloat16).pin_memory()
    idx = torch.tensor([3, 1], dtype=torch.int32)
    kb = torch.full((200, 2, 128), 3.0, dtype=torch.bfloat16, device=DEV)
    wa.wa_set_fault(wa.WA_FAULT_COPY)
    with pytest.raises(wa.WaError) as e:
        wa.wa_gather_pages(kp, None, None, idx, kb, None)
    assert e.value.status == 7                      # WA_ERR_CUDA
    torch.cuda.synchronize()
    assert torch.all(kb == 3.0)
    wa.wa_set_fault(wa.WA_FAULT_NONE)
    wa.wa_gather_pages(kp, None, None, idx, kb, None)
    wa.wa_check()
    assert np.array_equal(np_of(kb), O.gather_pages(np_of(kp), [3, 1]))
