"""Benchmark of the page-retrieval sparse-attention path for one chunk.

Workload (default): one layer at the WorldAttention shape -- 12 heads,
d_k = 128, bf16, 40 cached pages of 12,480 tokens (5 chunks x 8 pages) in HBM,
prompt embeddings of dim 4096, top-1 chunk then top-4 pages (49,920 tokens),
4,680 query tokens attending to the gathered buffer + 4,680 local tokens.

One step = the whole path: page summaries of all 40 cached pages, two-stage
retrieval, gather of the 4 pages (K and V) into the contiguous buffer, and
block attention.  Inputs are resident in HBM before timing; the page bank
(3.07 GB) is larger than L2, and each step's summaries stream all of it, so
L2 holds nothing useful from one step to the next.

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle on a
bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import contextlib
import datetime
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "chunk attention latency (ms) & TFLOP/s at 49,920 retrieved tokens; gather GB/s"
WORKLOAD = "worldattention_1layer: H=12 d=128 bf16, 40 pages x 12480 tok, top-1 of 5 chunks, K_p=4 (49,920), n_q=4680 + 4680 local"

H, D, P, N_PAGES, PPC, N_CHUNKS, PDIM, KP, NQ, NLOC = 12, 128, 12480, 40, 8, 5, 4096, 4, 4680, 4680

# DRAM bytes read + written per launch of the attention kernel, from one ncu capture of the
# current kernel (profiles/attention_worldattention_1layer.md); None once the kernel changes.
ATTN_TRAFFIC_BYTES = 393.66e6
# the same for the gather+attention launch, the kernel's paged form
# (profiles/gather_attention_worldattention_1layer.md)
FUSED_TRAFFIC_BYTES = 678.13e6


def attn_flops(n_q, n_kv, d, h):
    """Matmul FLOPs of softmax attention: 2*n_q*n_kv*d for Q K^T and again for P V."""
    return 4.0 * n_q * n_kv * d * h


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            j = json.load(f)
        return j["hbm_gbs"], j["bf16_tflops"], j.get("bf16_tflops_sustained", j["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def tensor_peak(timed_ms):
    """The measured bf16 peak that applies to a timed region: the burst figure
    for a region shorter than 2 s (the kernel never reaches the sustained
    power-capped clock), the sustained one for longer regions."""
    _, burst, sus, src = peaks()
    if timed_ms < 2000.0:
        return burst, f"{src} bf16 burst (timed region {timed_ms:.0f} ms)"
    return sus, f"{src} bf16 sustained (timed region {timed_ms:.0f} ms)"


class Clocks:
    """nvidia-smi sampling during the timed region: the sampler is started
    and seen producing before the region begins, and only the samples whose
    timestamps fall inside the region are summarised."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None
        # raw samples (the JSON line carries their summary); WA_CLOCKS_DIR keeps them
        self.path = os.path.join(os.environ.get("WA_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"clocks_bench_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}",
                 "--query-gpu=timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
                 "clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            # the sampler takes a moment to start: wait (up to 5 s) for its first line
            deadline = time.time() + 5.0
            while time.time() < deadline and self.proc.poll() is None:
                if os.path.getsize(self.path) > 0:
                    break
                time.sleep(0.01)
        except Exception:
            self.proc = None
        self.t0 = time.time()
        return self

    def __exit__(self, *a):
        self.t1 = time.time()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows, inside = [], []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts[1:])
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    except ValueError:
                        continue
                    if self.t0 <= ts <= self.t1:
                        inside.append(parts[1:])
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        outside = not inside
        rows = rows if outside else inside
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
               "samples": len(rows)}
        if outside:
            out["samples_are"] = "around the timed region (none fell inside it)"
        return out


def dist_init(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def run_gpu(args, world, rank, local, hybrid=False, per_head=False):
    import torch

    import sparse_kv_cache_page_gb300 as wa
    from sparse_kv_cache_page_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wa.load()
    c = synth.worldattention_case(device=dev, layer=rank, recall_chunk=3)
    kp, vp, q, kl, vl = c.k_pages, c.v_pages, c.q, c.k_loc, c.v_loc
    pcur, pch = c.prompt_cur, c.prompt_chunks
    kbar = torch.empty((N_PAGES, H, D), dtype=torch.float32, device=dev)
    idx = torch.empty((H, KP) if per_head else (KP,), dtype=torch.int32, device=dev)
    kbuf = torch.empty((KP * P, H, D), dtype=torch.bfloat16, device=dev)
    vbuf = torch.empty_like(kbuf)
    o = torch.empty(q.shape, dtype=torch.float32, device=dev)   # fp32 result (tested tolerance)
    chunk = torch.empty(1, dtype=torch.int32, device=dev)

    def select(q_, kbar_, pcur_, pch_, ppc_, kp_, idx_):
        if per_head:
            wa.wa_select_pages_per_head(q_, kbar_, pcur_, pch_, ppc_, kp_, idx_)
        else:
            wa.wa_select_pages(q_, kbar_, pcur_, pch_, ppc_, kp_, idx_, chunk_out=chunk)

    def gather(idx_):
        if per_head:
            wa.wa_gather_pages_per_head(kp, vp, idx_, kbuf, vbuf)
        else:
            wa.wa_gather_pages(kp, vp, idx_, None, kbuf, vbuf)

    def gather_attn(q_, idx_, kl_, vl_, o_):
        # gather and attention in one launch: the attention's tile copies read
        # the selected pages, and the buffer is written from on-chip memory
        wa.wa_gather_attn(q_, kp, vp, idx_, kl_, vl_, o_, kbuf, vbuf)
    stream = torch.cuda.current_stream()
    L, RANK = KP * P + NLOC, 256
    if hybrid:
        ek = synth.normal((H, L, RANK), synth.seed_of("hybrid", "ek"), dev, torch.bfloat16,
                          std=L ** -0.5)
        ev = synth.normal((H, L, RANK), synth.seed_of("hybrid", "ev"), dev, torch.bfloat16,
                          std=L ** -0.5)

    def names_of(fused):
        return (("summarize", "select") + (("gather_attention",) if fused else ("gather", "attention"))
                + (("linear",) if hybrid else ()))

    def summarize(n_summ):
        # n_summ = N_PAGES: every cached page (the worst case); n_summ = PPC:
        # only the newest chunk's pages, as when summaries are taken at insert
        wa.wa_page_summarize(kp[N_PAGES - n_summ:], kbar[N_PAGES - n_summ:])

    def step(marks=None, n_summ=N_PAGES, fused=True):
        """One chunk: summaries, retrieval, gather and attention (one launch,
        or, with fused=False, the gather and the attention as two)."""
        n = [0]

        def mark():
            if marks is not None:
                marks[n[0]].record(stream)
            n[0] += 1
        mark()
        summarize(n_summ)
        mark()
        select(q, kbar, pcur, pch, PPC, KP, idx)
        mark()
        if fused:
            gather_attn(q, idx, kl, vl, o)
        else:
            gather(idx)
            mark()
            wa.wa_block_attn(q, kbuf, vbuf, kl, vl, o)
        mark()
        if hybrid:
            wa.wa_linear_branch(q, kbuf, vbuf, kl, vl, ek, ev, o)
            mark()

    def timed_steps(n_summ, clk=None, marked=False, fused=True):
        """Time args.steps steps; with `marked`, an event between every two
        kernels gives the per-kernel intervals (the events also serialise the
        kernels' launches, so the headline total is taken without them)."""
        names = names_of(fused)
        for _ in range(args.warmup):
            step(n_summ=n_summ, fused=fused)
        wa.wa_check()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
               for _ in range(args.steps)] if marked else None
        barrier(world)
        torch.cuda.synchronize()
        with (clk if clk is not None else contextlib.nullcontext()):
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for k in range(args.steps):
                step(evs[k] if marked else None, n_summ=n_summ, fused=fused)
            t1.record(stream)
            torch.cuda.synchronize()
        barrier(world)
        wa.wa_check()
        total = max_over_ranks(t0.elapsed_time(t1), world)
        if not marked:
            return total, None
        per_ = {n: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1])
                                   for k in range(args.steps))
                for i, n in enumerate(names)}
        return total, per_

    clk = Clocks(local)
    total_ms, _ = timed_steps(N_PAGES, clk)
    ms_step = total_ms / args.steps
    marked_ms, per = timed_steps(N_PAGES, marked=True)
    total_ins, _ = timed_steps(PPC)
    ms_step_ins = total_ins / args.steps
    _, per_ins = timed_steps(PPC, marked=True)
    # the same step with the gather and the attention as two launches
    total_two, _ = timed_steps(N_PAGES, fused=False)
    ms_step_two = total_two / args.steps
    _, per_two = timed_steps(N_PAGES, marked=True, fused=False)

    # end to end through the public API: per step, the chunk's inputs come from
    # pinned host memory and the output goes back to pinned host memory.  The
    # copies run on a copy stream, double-buffered, so that step k+1's inputs
    # travel while step k computes (every copy is inside the timed region).
    hq = q.cpu().pin_memory()
    hkl, hvl = kl.cpu().pin_memory(), vl.cpu().pin_memory()
    hpc = pcur.cpu().pin_memory()
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    dbuf = [(torch.empty_like(q), torch.empty_like(kl), torch.empty_like(vl), torch.empty_like(pcur),
             torch.empty_like(o)) for _ in range(2)]
    cs = torch.cuda.Stream()

    def e2e_run(n, n_summ=N_PAGES):
        """n steps through the public API.  The copies run on the copy stream
        beside the retrieval and the gather + attention (compute-bound), not
        beside the HBM-bound summaries: once step k's summaries are done, so is
        step k-1, and step k-1's output goes back and step k+1's inputs come in
        while step k runs on.  Apart from the wait for its own inputs, no event
        sits between a step's kernels, so each launch keeps overlapping the
        previous kernel's drain."""
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_mid = [torch.cuda.Event() for _ in range(n)]
        ev_last = torch.cuda.Event()
        cs.wait_stream(stream)

        def h2d(k):
            dq, dkl, dvl, dpc, _ = dbuf[k % 2]
            with torch.cuda.stream(cs):
                dq.copy_(hq, non_blocking=True)
                dkl.copy_(hkl, non_blocking=True)
                dvl.copy_(hvl, non_blocking=True)
                dpc.copy_(hpc, non_blocking=True)
                ev_in[k].record(cs)

        def d2h(k):
            with torch.cuda.stream(cs):
                ho[k % 2].copy_(dbuf[k % 2][4], non_blocking=True)

        h2d(0)
        for k in range(n):
            dq, dkl, dvl, dpc, do = dbuf[k % 2]
            # the summaries read only the resident page bank: they run while this
            # step's inputs may still be arriving
            summarize(n_summ)
            ev_mid[k].record(stream)
            stream.wait_event(ev_in[k])
            select(dq, kbar, dpc, pch, PPC, KP, idx)
            gather_attn(dq, idx, dkl, dvl, do)
            if hybrid:
                wa.wa_linear_branch(dq, kbuf, vbuf, dkl, dvl, ek, ev, do)
            # after this step's summaries (so after all of step k-1): step k-1's
            # output goes back, then step k+1's inputs arrive into the buffers
            # that step k-1 read
            with torch.cuda.stream(cs):
                cs.wait_event(ev_mid[k])
            if k >= 1:
                d2h(k - 1)
            if k + 1 < n:
                h2d(k + 1)
        ev_last.record(stream)
        with torch.cuda.stream(cs):
            cs.wait_event(ev_last)
        d2h(n - 1)
        stream.wait_stream(cs)

    def e2e_timed(n_summ):
        e2e_run(max(2, args.warmup), n_summ)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(args.steps, n_summ)
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), world) / args.steps

    e2e_ms = e2e_timed(N_PAGES)
    e2e_ms_ins = e2e_timed(PPC)
    h2d_bytes = sum(t.numel() * t.element_size() for t in (hq, hkl, hvl, hpc))
    d2h = ho[0].numel() * ho[0].element_size()
    assert torch.equal(ho[(args.steps - 1) % 2], dbuf[(args.steps - 1) % 2][4].cpu())

    hbm, tf_burst, tf_sus, src = peaks()
    tf_peak, peak_src = tensor_peak(total_ms)
    n_kv = KP * P + NLOC
    flops = attn_flops(NQ, n_kv, D, H)
    attn_tflops = flops / (per["gather_attention"] * 1e-3) / 1e12
    attn_tflops_two = flops / (per_two["attention"] * 1e-3) / 1e12
    context = None if (hybrid or per_head or args.no_context) else sdpa_context(q, kbuf, vbuf, kl,
                                                                                vl, flops)
    gather_bytes = 2 * 2 * KP * P * H * D * 2          # K and V, read + write
    summ_bytes = N_PAGES * P * H * D * 2
    value = world * flops / (ms_step * 1e-3) / 1e12
    launches_per_step = 3 + (3 if hybrid else 0)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), WorldAttention shapes)",
        "config": headline_config(world),
        "chunk_latency_ms": round(ms_step, 4),
        "chunk_latency_is": f"worst case: each step summarises all {N_PAGES} cached pages",
        "kernels_ms": {k: round(v, 4) for k, v in per.items()},
        "kernels_ms_are": "event intervals from a separate pass with an event between every two "
                          f"kernels (step {marked_ms / args.steps:.4f} ms there: the events "
                          "serialise the launches that the unmarked step overlaps)",
        "chunk_latency_ms_insert": round(ms_step_ins, 4),
        "chunk_latency_insert_is": f"summaries taken at insert: each step summarises only the "
                                   f"{PPC} pages of the newest chunk, then retrieval over all "
                                   f"{N_PAGES} summaries, gather and attention",
        "kernels_ms_insert": {k: round(v, 4) for k, v in per_ins.items()},
        "value_insert": round(world * flops / (ms_step_ins * 1e-3) / 1e12, 2),
        "chunk_latency_ms_two_launch": round(ms_step_two, 4),
        "two_launch_is": "the same step with the gather and the attention as separate launches "
                         "(wa_gather_pages, then wa_block_attn over the buffer)",
        "kernels_ms_two_launch": {k: round(v, 4) for k, v in per_two.items()},
        "attn_tflops": round(attn_tflops, 1),
        "attn_tflops_is": "attention FLOPs / the gather+attention launch (which also writes the "
                          "gathered buffer)",
        "attn_tflops_two_launch": round(attn_tflops_two, 1),
        "gather_gbs": round(gather_bytes / (per_two["gather"] * 1e-3) / 1e9, 1),
        "summarize_gbs": round(summ_bytes / (per["summarize"] * 1e-3) / 1e9, 1),
        "roofline": {"bound": "tensor", "achieved": round(attn_tflops, 1), "peak": tf_peak,
                     "unit": "TFLOP/s", "frac": round(attn_tflops / tf_peak, 4),
                     "traffic": FUSED_TRAFFIC_BYTES if not hybrid else None,
                     "kernel": "k_block_attn_tc, paged form (gather fused)",
                     "peak_source": peak_src,
                     "frac_of_sustained": round(attn_tflops / tf_sus, 4),
                     "two_launch_attention": {"kernel": "k_block_attn_tc",
                                              "achieved": round(attn_tflops_two, 1),
                                              "frac": round(attn_tflops_two / tf_peak, 4),
                                              "traffic": ATTN_TRAFFIC_BYTES if not hybrid
                                              else None},
                     # the same attention FLOPs over the two launches' time (gather +
                     # attention), the work the one launch replaces
                     "two_launch_gather_attention_frac": round(
                         flops / ((per_two["gather"] + per_two["attention"]) * 1e-3) / 1e12
                         / tf_peak, 4)},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h, "copies": "copy stream, double-buffered: once step k's "
                                                       "summaries are done, step k-1's output goes "
                                                       "back and step k+1's inputs come in, beside "
                                                       "step k's retrieval and gather+attention",
                "ms_per_step_insert": round(e2e_ms_ins, 4),
                "value_insert": round(world * flops / (e2e_ms_ins * 1e-3) / 1e12, 2)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    idx_bench = idx.clone()
    if context is not None:
        line["context_sdpa"] = context
    if per_head:
        line["config"]["workload"] = ("per_head: " + WORKLOAD + " with a top-4 page set per head "
                                      "(per-head scores, per-head gather into the token-major "
                                      "buffer)")
        line.pop("cpu_baseline", None)
    if hybrid:
        proj_bytes = 2 * H * L * RANK * 2 + 2 * L * H * D * 2
        line["config"]["workload"] = ("hybrid: " + WORKLOAD + " + Linformer branch rank 256 "
                                      "(E_K, E_V [12][54600][256] bf16), equal-weight fusion")
        line["linear_ms"] = round(per["linear"], 4)
        line["linear_read_gbs"] = round(proj_bytes / (per["linear"] * 1e-3) / 1e9, 1)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not hybrid and not per_head:
        # the last timed step's indices and output, checked against the oracle
        line["cpu_baseline"], line["parity"] = cpu_baseline_gpu_arm(c, kp, vp, o, idx_bench, chunk,
                                                                    kbuf, vbuf)
    return line


def sdpa_context(q, kbuf, vbuf, kl, vl, flops):
    """Context only, not on the path: PyTorch's own attention
    (torch.nn.functional.scaled_dot_product_attention) on the same bf16 queries
    and [buffer (+) local] keys and values, per backend PyTorch offers here,
    head-major copies made outside the timing, bf16 output."""
    import torch
    import torch.nn.functional as F
    from torch.nn.attention import SDPBackend, sdpa_kernel

    qh = q.permute(1, 0, 2).unsqueeze(0).contiguous()
    kh = torch.cat([kbuf, kl]).permute(1, 0, 2).unsqueeze(0).contiguous()
    vh = torch.cat([vbuf, vl]).permute(1, 0, 2).unsqueeze(0).contiguous()
    out = {}
    for name in ("CUDNN_ATTENTION", "FLASH_ATTENTION", "EFFICIENT_ATTENTION"):
        be = getattr(SDPBackend, name, None)
        if be is None:
            continue
        try:
            with sdpa_kernel([be]):
                for _ in range(3):
                    F.scaled_dot_product_attention(qh, kh, vh)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(10):
                    F.scaled_dot_product_attention(qh, kh, vh)
                e1.record()
                torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / 10
            out[name.lower()] = {"ms": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}
        except Exception as e:   # backend not available for this GPU / shape
            out[name.lower()] = {"unavailable": type(e).__name__}
    del qh, kh, vh
    return out


def run_hsa(args, world, rank, local):
    """One chunk with the HSA branches in place of dense attention
    (WorldAttention review page, HSA section): retrieval as in the headline
    workload (summaries, two-stage selection, gather), then the sparse branch
    -- block means of the queries (64), the buffer (128) and the local tokens
    (64), the pooled block map and Gini-adaptive block selection per head,
    block-sparse attention over the kept blocks -- and the Linformer branch
    (rank 256) fused with equal per-head weights.  Synthetic structure: in 4
    of the 12 heads (0, 3, 6, 9) the queries and one 128-token block of every
    page share a direction (gain 3), so those heads have peaked block maps;
    the other heads are N(0,1) with near-uniform maps."""
    import torch

    import sparse_kv_cache_page_gb300 as wa
    from sparse_kv_cache_page_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wa.load()
    c = synth.worldattention_case(device=dev, layer=rank, recall_chunk=3)
    kp, vp, q, kl, vl = c.k_pages, c.v_pages, c.q, c.k_loc, c.v_loc
    pcur, pch = c.prompt_cur, c.prompt_chunks
    peaked = (0, 3, 6, 9)
    for i, h in enumerate(peaked):
        u = synth.normal((D,), synth.seed_of("hsa", rank, "dir", h), dev).to(torch.bfloat16)
        blk = 37 + 11 * i
        kp[:, blk * 128:(blk + 1) * 128, h, :] += 3.0 * u
        q[:, h, :] += 3.0 * u
    kbar = torch.empty((N_PAGES, H, D), dtype=torch.float32, device=dev)
    idx = torch.empty(KP, dtype=torch.int32, device=dev)
    kbuf = torch.empty((KP * P, H, D), dtype=torch.bfloat16, device=dev)
    vbuf = torch.empty_like(kbuf)
    o = torch.empty(q.shape, dtype=torch.float32, device=dev)
    nqb, nmb, nlb = -(-NQ // 64), KP * P // 128, -(-NLOC // 64)
    qbar = torch.empty((nqb, H, D), dtype=torch.float32, device=dev)
    kbb = torch.empty((nmb + nlb, H, D), dtype=torch.float32, device=dev)
    sel = torch.empty((H, nmb + nlb), dtype=torch.int32, device=dev)
    cnt = torch.empty(H, dtype=torch.int32, device=dev)
    gini = torch.empty(H, dtype=torch.float32, device=dev)
    L, RANK = KP * P + NLOC, 256
    ek = synth.normal((H, L, RANK), synth.seed_of("hybrid", "ek"), dev, torch.bfloat16, std=L ** -0.5)
    ev = synth.normal((H, L, RANK), synth.seed_of("hybrid", "ev"), dev, torch.bfloat16, std=L ** -0.5)
    stream = torch.cuda.current_stream()
    names = ("summarize", "select", "gather", "block_means", "block_select", "sparse_attention",
             "linear")

    def step(marks=None):
        def mark(i):
            if marks is not None:
                marks[i].record(stream)
        mark(0)
        wa.wa_page_summarize(kp, kbar)
        mark(1)
        wa.wa_select_pages(q, kbar, pcur, pch, PPC, KP, idx)
        mark(2)
        wa.wa_gather_pages(kp, vp, idx, None, kbuf, vbuf)
        mark(3)
        wa.wa_block_means_segments([(q, 64, qbar), (kbuf, 128, kbb[:nmb]), (kl, 64, kbb[nmb:])])
        mark(4)
        wa.wa_sparse_select(qbar, kbb, sel, cnt, gini_out=gini)
        mark(5)
        wa.wa_sparse_attn(q, kbuf, vbuf, kl, vl, sel, cnt, o, 128, 64)
        mark(6)
        wa.wa_linear_branch(q, kbuf, vbuf, kl, vl, ek, ev, o)
        mark(7)

    for _ in range(args.warmup):
        step()
    wa.wa_check()
    # headline: no events between kernels (they would serialise the launches)
    barrier(world)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for k in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    wa.wa_check()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    ms = total_ms / args.steps
    # per-kernel intervals from a separate pass with an event between every two kernels
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    for k in range(args.steps):
        step(evs[k])
    torch.cuda.synchronize()
    wa.wa_check()
    per = {n: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps))
           for i, n in enumerate(names)}
    counts = cnt.cpu().tolist()
    selc = sel.cpu()
    kept_keys = []
    for h in range(H):
        blocks = selc[h, :counts[h]].tolist()
        kept_keys.append(sum(128 if b < nmb else min(64, NLOC - 64 * (b - nmb)) for b in blocks))
    sparse_flops = 4.0 * NQ * D * sum(kept_keys)
    dense_flops = attn_flops(NQ, KP * P + NLOC, D, H)
    hbm, tf_burst, tf_sus, src = peaks()
    tf_peak, peak_src = tensor_peak(total_ms)
    sp_tflops = sparse_flops / (per["sparse_attention"] * 1e-3) / 1e12
    return {
        "metric": METRIC, "value": round(world * dense_flops / (ms * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (planted peaked heads 0, 3, 6, 9)",
        "config": {"workload": "hsa: " + WORKLOAD + " with the HSA branches: sparse (blocks 128 "
                               "buffer / 64 local / 64 query, tau_h = 1 - Gini) + Linformer "
                               "rank 256, equal-weight fusion",
                   "value_is": "dense-equivalent attention FLOPs of the chunk / whole-step time"},
        "kernels_ms": {k: round(v, 4) for k, v in per.items()},
        "kept_blocks": counts, "n_blocks": nmb + nlb,
        "kept_key_fraction": round(sum(kept_keys) / (H * (KP * P + NLOC)), 4),
        "gini": [round(x, 4) for x in gini.cpu().tolist()],
        "sparse_attn_tflops": round(sp_tflops, 1),
        "roofline": {"bound": "tensor", "achieved": round(sp_tflops, 1), "peak": tf_peak,
                     "unit": "TFLOP/s", "frac": round(sp_tflops / tf_peak, 4), "traffic": None,
                     "peak_source": peak_src, "frac_of_sustained": round(sp_tflops / tf_sus, 4),
                     "kernel": "k_block_attn_tc (block-sparse form)"},
        # per step: summaries, select, gather, block means (one launch), pooled scores,
        # block select, sparse tiles, block-sparse attention, projection, reduce,
        # low-rank attention
        "gpu_launches": 11 * args.steps, "clocks": clk.summary(),
    }


def run_cache(args, world, rank, local):
    """Generation loop over the KV cache manager: 12 chunks (a 60-second video
    as 12 five-second chunks, WorldAttention review page, worked example), each
    8 pages of 12,480 tokens, an HBM tier of 16 pages and a pinned DRAM tier of
    96.  Per chunk after the first: retrieval of the top-4 pages (prompt stage
    over the past chunks, page stage, pages fetched from either tier, DRAM pages
    promoted), attention of the chunk's queries over them plus the chunk's own
    KV, then the chunk's KV appended (summaries at insert, least recently used
    pages offloaded to DRAM).  One bench step = the 11 chunks of one video."""
    import torch

    import sparse_kv_cache_page_gb300 as wa
    from sparse_kv_cache_page_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wa.load()
    NCH, PDIM = 12, 4096
    g = lambda shape, t, dt=torch.bfloat16: synth.normal(shape, synth.seed_of("cache", rank, t),  # noqa: E731
                                                         dev, dt)
    ks = [g((PPC * P, H, D), ("k", m)) for m in range(NCH)]
    vs = [g((PPC * P, H, D), ("v", m)) for m in range(NCH)]
    prompts = [g((PDIM,), ("prompt", m), torch.float32) for m in range(NCH)]
    qs = [g((NQ, H, D), ("q", m)) for m in range(NCH)]
    # chunk m's prompt recalls an earlier chunk, (5 m + 3) mod m (a scene revisited)
    curs = [None] + [prompts[(5 * m + 3) % m] + 0.5 * g((PDIM,), ("cur", m), torch.float32)
                     for m in range(1, NCH)]
    kb = torch.empty((KP * P, H, D), dtype=torch.bfloat16, device=dev)
    vb = torch.empty_like(kb)
    o = torch.empty((NQ, H, D), dtype=torch.float32, device=dev)

    # the tiers are allocated once per cache (HBM slots, staging ring and pinned
    # DRAM: 9 GB with bf16 DRAM pages); each video starts from an emptied cache
    # (wa_cache_reset), outside the timed loop
    def video(cache):
        cache.append(ks[0], vs[0], prompts[0])
        for m in range(1, NCH):
            cache.retrieve(qs[m], curs[m], KP, kb, vb)
            wa.wa_block_attn(qs[m], kb, vb, ks[m][:NLOC], vs[m][:NLOC], o)
            cache.append(ks[m], vs[m], prompts[m])
        cache.wait_copies()          # the last offloads belong to this video too

    def timed(fmt, clk=None):
        cache = wa.WaCache(H, D, P, PPC, hbm_pages=16, host_pages=96, max_chunks=NCH,
                           prompt_dim=PDIM, dram_format=fmt)
        for _ in range(max(1, args.warmup - 2)):
            cache.reset()
            video(cache)
        torch.cuda.synchronize()
        steps = max(1, min(args.steps, 5))
        total = 0.0
        with (clk if clk is not None else contextlib.nullcontext()):
            for _ in range(steps):
                cache.reset()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                video(cache)
                e1.record()
                torch.cuda.synchronize()
                total += e0.elapsed_time(e1)
        st = cache.stats()
        cache.close()
        return max_over_ranks(total, world) / steps, steps, st

    clk = Clocks(local)
    ms, steps, st = timed("native", clk)
    ms8, _, st8 = timed("fp8")
    ms4, _, st4 = timed("nvfp4")
    flops = (NCH - 1) * attn_flops(NQ, KP * P + NLOC, D, H)
    return {"metric": METRIC, "value": round(world * flops / (ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "ms_per_chunk": round(ms / (NCH - 1), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "cache: 12 chunks x 8 pages x 12,480 tokens through the KV "
                                   "cache manager (HBM tier 16 pages, pinned DRAM tier 96, "
                                   "inclusive, offloads on a copy stream), retrieve top-4 + "
                                   "attention + append per chunk, H=12 d=128 bf16",
                       "value_is": "attention FLOPs of the 11 chunks / whole-loop time "
                                   "(appends, offloads, fetches and promotions included, the "
                                   "last offloads waited for; tier allocation excluded)"},
            "cache_stats_per_video": st,
            "fp8_dram_tier": {"ms_per_step": round(ms8, 3), "ms_per_chunk": round(ms8 / (NCH - 1), 3),
                              "cache_stats_per_video": st8},
            "nvfp4_dram_tier": {"ms_per_step": round(ms4, 3),
                                "ms_per_chunk": round(ms4 / (NCH - 1), 3),
                                "cache_stats_per_video": st4},
            "gpu_launches": steps * (NCH + 2 * (NCH - 1)),   # summaries per append; select + attention
            "clocks": clk.summary()}


def run_one_kernel(args, local):
    """One kernel alone at the workload's shape (inputs drawn directly): the
    attention over a 49,920-token buffer + 4,680 local tokens, the gather of 4
    pages from a 12-page bank, both in one launch (gather_attention), or a page
    codec (FP8 / NVFP4) encoding and decoding 8 pages (307 MB of bf16, larger
    than L2).  Used for profiling captures."""
    import torch

    import sparse_kv_cache_page_gb300 as wa
    from sparse_kv_cache_page_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wa.load()
    g = lambda shape, t: synth.normal(shape, synth.seed_of("one_kernel", t), device=dev,  # noqa: E731
                                      dtype=torch.bfloat16)
    if args.kernel == "attention":
        q, kb, vb = g((NQ, H, D), "q"), g((KP * P, H, D), "kb"), g((KP * P, H, D), "vb")
        kl, vl = g((NLOC, H, D), "kl"), g((NLOC, H, D), "vl")
        o = torch.empty(q.shape, dtype=torch.float32, device=dev)
        fn = lambda: wa.wa_block_attn(q, kb, vb, kl, vl, o)  # noqa: E731
        work, unit = attn_flops(NQ, KP * P + NLOC, D, H) / 1e12, "TFLOP/s"
    elif args.kernel == "gather_attention":
        kp, vp = g((12, P, H, D), "kp"), g((12, P, H, D), "vp")
        idx = torch.tensor([9, 2, 5, 11], dtype=torch.int32, device=dev)
        q, kl, vl = g((NQ, H, D), "q"), g((NLOC, H, D), "kl"), g((NLOC, H, D), "vl")
        kb = torch.empty((KP * P, H, D), dtype=torch.bfloat16, device=dev)
        vb = torch.empty_like(kb)
        o = torch.empty(q.shape, dtype=torch.float32, device=dev)
        fn = lambda: wa.wa_gather_attn(q, kp, vp, idx, kl, vl, o, kb, vb)  # noqa: E731
        work, unit = attn_flops(NQ, KP * P + NLOC, D, H) / 1e12, "TFLOP/s"
    elif args.kernel == "linear":
        L, R = KP * P + NLOC, 256
        q, kb, vb = g((NQ, H, D), "q"), g((KP * P, H, D), "kb"), g((KP * P, H, D), "vb")
        kl, vl = g((NLOC, H, D), "kl"), g((NLOC, H, D), "vl")
        ek = synth.normal((H, L, R), synth.seed_of("one_kernel", "ek"), dev, torch.bfloat16,
                          std=L ** -0.5)
        ev = synth.normal((H, L, R), synth.seed_of("one_kernel", "ev"), dev, torch.bfloat16,
                          std=L ** -0.5)
        o = torch.zeros((NQ, H, D), dtype=torch.float32, device=dev)
        fn = lambda: wa.wa_linear_branch(q, kb, vb, kl, vl, ek, ev, o)  # noqa: E731
        work, unit = (2 * H * L * R * 2 + 2 * L * H * D * 2) / 1e9, "GB/s (E + K,V read)"
    elif args.kernel in ("fp8", "nvfp4"):
        x = g((8 * P, H, D), "pages")
        y = torch.empty_like(x)
        n = 8 * P * H
        if args.kernel == "fp8":
            c = torch.empty((8 * P, H, D), dtype=torch.uint8, device=dev)
            sc = torch.empty((8 * P, H), dtype=torch.float32, device=dev)
            enc = lambda: wa.wa_fp8_encode(x, c, sc)  # noqa: E731
            dec = lambda: wa.wa_fp8_decode(c, sc, y)  # noqa: E731
            packed = n * (D + 4)
        else:
            c = torch.empty((8 * P, H, D // 2), dtype=torch.uint8, device=dev)
            b = torch.empty((8 * P, H, D // 16), dtype=torch.uint8, device=dev)
            r = torch.empty((8 * P, H), dtype=torch.float32, device=dev)
            enc = lambda: wa.wa_nvfp4_encode(x, c, b, r)  # noqa: E731
            dec = lambda: wa.wa_nvfp4_decode(c, b, r, y)  # noqa: E731
            packed = n * (D // 2 + D // 16 + 4)
        out = {"kernel": args.kernel, "steps": args.steps, "warmup": args.warmup,
               "bytes_per_launch": n * D * 2 + packed}
        hbm = peaks()[0]
        # the write-only rate of this GPU on the same 307 MB (a fill of the bf16
        # pages): the bound of a decoder, whose traffic is mostly the bf16 it writes
        fill = lambda: y.fill_(1.0)  # noqa: E731
        for name, fn in (("write_only_fill", fill), ("encode", enc), ("decode", dec)):
            for _ in range(args.warmup):
                fn()
            wa.wa_check()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.steps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            wa.wa_check()
            ms = e0.elapsed_time(e1) / args.steps
            if name == "write_only_fill":
                out[name] = {"ms": round(ms, 4), "GB/s": round(n * D * 2 / (ms * 1e-3) / 1e9, 1),
                             "frac_of_hbm": round(n * D * 2 / (ms * 1e-3) / 1e9 / hbm, 3)}
                continue
            gbs = (n * D * 2 + packed) / (ms * 1e-3) / 1e9
            out[name] = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 3)}
        # the decoder against the time the device takes to write its bf16 alone
        out["decode"]["frac_of_write_bound"] = round(out["write_only_fill"]["ms"] / out["decode"]["ms"], 3)
        return out
    else:
        kp, vp = g((12, P, H, D), "kp"), g((12, P, H, D), "vp")
        idx = torch.tensor([9, 2, 5, 11], dtype=torch.int32, device=dev)
        kb, vb = torch.empty((KP * P, H, D), dtype=torch.bfloat16, device=dev), None
        vb = torch.empty_like(kb)
        fn = lambda: wa.wa_gather_pages(kp, vp, idx, None, kb, vb)  # noqa: E731
        work, unit = 2 * 2 * KP * P * H * D * 2 / 1e9, "GB/s"
    for _ in range(args.warmup):
        fn()
    wa.wa_check()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    wa.wa_check()
    ms = e0.elapsed_time(e1) / args.steps
    return {"kernel": args.kernel, "ms": round(ms, 4), "value": round(work / (ms * 1e-3), 1),
            "unit": unit, "steps": args.steps, "warmup": args.warmup}


def run_denoise(args, world, rank, local):
    """Block-diffusion denoising reuse: a cached 21-frame (32,760-token) KV
    window per layer, re-attended by a 3-frame query block for 4 denoising
    steps, each with fresh queries and fresh local K/V.  One bench step = the
    4 denoising steps of one block."""
    import torch

    import sparse_kv_cache_page_gb300 as wa
    from sparse_kv_cache_page_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wa.load()
    WIN, T = 21 * 1560, 4
    g = lambda shape, t: synth.normal(shape, synth.seed_of("denoise", rank, t), dev,  # noqa: E731
                                      torch.bfloat16)
    kw, vw = g((WIN, H, D), "kw"), g((WIN, H, D), "vw")
    qs = [g((NQ, H, D), ("q", t)) for t in range(T)]
    kls = [g((NLOC, H, D), ("kl", t)) for t in range(T)]
    vls = [g((NLOC, H, D), ("vl", t)) for t in range(T)]
    o = torch.empty((NQ, H, D), dtype=torch.float32, device=dev)

    def step():
        for t in range(T):
            wa.wa_block_attn(qs[t], kw, vw, kls[t], vls[t], o)

    for _ in range(args.warmup):
        step()
    wa.wa_check()
    barrier(world)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
    wa.wa_check()
    ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    flops = T * attn_flops(NQ, WIN + NLOC, D, H)
    return {"metric": METRIC, "value": round(world * flops / (ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "ms_per_denoising_step": round(ms / T, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "denoise: 21-frame window (32,760 tokens) reused for 4 "
                                   "denoising steps, 3-frame query block (4,680) + fresh local "
                                   "KV, H=12 d=128 bf16", "l2": "window 201 MB per tensor > L2"},
            "gpu_launches": T * args.steps, "clocks": clk.summary()}


def run_stress(args, world, rank, local):
    """Minute-long stress: layers run one after another; each layer's 120
    cached pages (K and V, 9.2 GB) live in pinned host memory -- one page store
    shared by all layers, each layer with its own queries and local KV.  Per
    layer: top-4 of 120 pages, the 4 pages copied host -> device by the copy
    engine on a side stream into one of two buffers, attention on the main
    stream.  Retrieval for all layers runs first (the synthetic queries exist up
    front), so layer l+1's copy overlaps layer l's attention."""
    import torch

    import sparse_kv_cache_page_gb300 as wa
    from sparse_kv_cache_page_gb300 import synth
    from sparse_kv_cache_page_gb300.tiered import TieredPipeline, TierLayer

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wa.load()
    NPG, NL = synth.STRESS_PAGES, args.layers
    hk = torch.empty((NPG, P, H, D), dtype=torch.bfloat16, pin_memory=True)
    hv = torch.empty((NPG, P, H, D), dtype=torch.bfloat16, pin_memory=True)
    # the compressed tier: the same pages as FP8 E4M3 codes + per-row scales
    kc = torch.empty((NPG, P, H, D), dtype=torch.uint8, pin_memory=True)
    vc = torch.empty((NPG, P, H, D), dtype=torch.uint8, pin_memory=True)
    ksc = torch.empty((NPG, P, H), dtype=torch.float32, pin_memory=True)
    vsc = torch.empty((NPG, P, H), dtype=torch.float32, pin_memory=True)
    # and as NVFP4: E2M1 codes, E4M3 scales per 16 values, fp32 row scales
    nv = [(torch.empty((NPG, P, H, D // 2), dtype=torch.uint8, pin_memory=True),
           torch.empty((NPG, P, H, D // 16), dtype=torch.uint8, pin_memory=True),
           torch.empty((NPG, P, H), dtype=torch.float32, pin_memory=True)) for _ in range(2)]
    kbar = torch.empty((NPG, H, D), dtype=torch.float32, device=dev)
    for j in range(NPG):
        kj, vj = synth.stress_page(j, dev, rank)
        wa.wa_page_summarize(kj[None], kbar[j:j + 1])
        hk[j].copy_(kj)
        hv[j].copy_(vj)
        wa.wa_fp8_encode(kj, kc[j], ksc[j])
        wa.wa_fp8_encode(vj, vc[j], vsc[j])
        for t, x in enumerate((kj, vj)):
            wa.wa_nvfp4_encode(x, nv[t][0][j], nv[t][1][j], nv[t][2][j])
    torch.cuda.synchronize()
    o = torch.empty((NQ, H, D), dtype=torch.float32, device=dev)
    layers = [TierLayer(*synth.stress_layer(l, dev, rank), kbar, hk, hv, o, kc, ksc, vc, vsc,
                        k_nv=nv[0], v_nv=nv[1])
              for l in range(NL)]
    pipe = TieredPipeline(KP, P, H, D, device=dev)
    torch.cuda.synchronize()

    def timed(mode, reps):
        pipe.run(layers, mode)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            pipe.run(layers, mode)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    for _ in range(max(1, args.warmup - 1)):
        pipe.run(layers)
    wa.wa_check()
    reps = max(1, args.steps // 10)
    with Clocks(local) as clk:
        t_pipe = timed("pipeline", reps)
    t_serial = timed("serial", 1)
    t_direct = timed("direct", reps)
    t_fp8 = timed("fp8", reps)
    t_fp8p = timed("fp8_pipeline", reps)
    t_nv = timed("nvfp4", reps)
    t_nvp = timed("nvfp4_pipeline", reps)
    t_copy = timed("copy", 1)
    t_attn = timed("attn", 1)
    wa.wa_check()
    flops = NL * attn_flops(NQ, KP * P + NLOC, D, H)
    h2d = NL * 2 * KP * P * H * D * 2
    hidden = max(0.0, min(1.0, (t_copy + t_attn - t_pipe) / t_copy)) if t_copy > 0 else None
    return {"metric": METRIC, "value": round(world * flops / (t_pipe * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "n_gpus": world, "steps": reps, "warmup": args.warmup,
            "ms_per_step": round(t_pipe, 3), "ms_per_layer": round(t_pipe / NL, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"stress: {NL} layers, 120 pages/layer in pinned host memory "
                                   "(one 9.2 GB store shared by the layers), top-4 of 120, H=12 "
                                   "d=128 bf16, 4,680 queries + 4,680 local per layer"},
            "serial_ms": round(t_serial, 3), "direct_ms": round(t_direct, 3),
            "fp8_tier_ms": round(t_fp8, 3), "fp8_tier_pipeline_ms": round(t_fp8p, 3),
            "fp8_tier_link_bytes_per_layer": 2 * KP * P * H * (D + 4),
            "nvfp4_tier_ms": round(t_nv, 3), "nvfp4_tier_pipeline_ms": round(t_nvp, 3),
            "nvfp4_tier_link_bytes_per_layer": 2 * KP * P * H * (D // 2 + D // 16 + 4),
            "copy_only_ms": round(t_copy, 3),
            "attn_only_ms": round(t_attn, 3), "h2d_gbs": round(h2d / (t_copy * 1e-3) / 1e9, 1),
            "copy_hidden_frac": hidden, "gpu_launches": NL * 2, "clocks": clk.summary()}


# ----------------------------------------------------------------------------
# CPU oracle arm
# ----------------------------------------------------------------------------

SAMPLE_ROWS_STEP = N_PAGES    # query rows 0, 40, 80, ...: 117 rows, 1/40 of the chunk's queries


class _PageBank:
    """Host copies of page bodies for the oracle, fetched on first use (never
    inside a timed sample: every page a sample reads is fetched in set-up)."""

    def __init__(self, fetch):
        self.fetch = fetch
        self.pages = {}

    def __getitem__(self, j):
        j = int(j)
        if j not in self.pages:
            self.pages[j] = self.fetch(j)
        return self.pages[j]


def oracle_setup(c, fetch_k, fetch_v):
    """Untimed set-up of the oracle sample: the oracle's own summaries of every
    cached page (the retrieval in the sample scores real summaries), the
    queries, local KV and prompts converted once, and the selected pages'
    bodies fetched, so that a timed sample spends its time in the oracle only."""
    import numpy as np

    import oracle as O
    from sparse_kv_cache_page_gb300 import synth

    kb, vb = _PageBank(fetch_k), _PageBank(fetch_v)
    inp = {"k_bank": kb, "v_bank": vb, "q": synth.to_oracle(c.q),
           "kloc": synth.to_oracle(c.k_loc), "vloc": synth.to_oracle(c.v_loc),
           "pcur": synth.to_oracle(c.prompt_cur), "pch": synth.to_oracle(c.prompt_chunks)}
    inp["kbar"] = np.stack([O.page_summarize(kb[j][None])[0] for j in range(N_PAGES)])
    idx, _, chunk = O.select_pages(inp["q"], inp["kbar"], inp["pcur"], inp["pch"], PPC, KP)
    for j in idx:
        vb[j]
    inp["idx"], inp["chunk"] = [int(j) for j in idx], chunk
    inp["rows"] = np.arange(0, NQ, SAMPLE_ROWS_STEP)
    # buffer rows whose gathered bytes the GPU arm checks: every 997th, and the last
    inp["buf_rows"] = np.concatenate([np.arange(0, KP * P, 997), [KP * P - 1]])
    return inp


def oracle_sample(inp):
    """One timed sample of the chunk, by the fp64 oracle as it stands: the
    summary of one page (of 40), the two-stage retrieval over the 40
    summaries, the 4-page gather of K and V, and attention for 117 of the
    4,680 query rows (every head, all 54,600 keys).  Returns the measured
    seconds of each part and the attention output of the sampled rows."""
    import oracle as O

    t0 = time.perf_counter()
    O.page_summarize(inp["k_bank"][0][None])
    t1 = time.perf_counter()
    idx, _, chunk = O.select_pages(inp["q"], inp["kbar"], inp["pcur"], inp["pch"], PPC, KP)
    t2 = time.perf_counter()
    kbuf = O.gather_pages(inp["k_bank"], idx)
    vbuf = O.gather_pages(inp["v_bank"], idx)
    t3 = time.perf_counter()
    o, _ = O.block_attn(inp["q"], kbuf, vbuf, inp["kloc"], inp["vloc"], rows=inp["rows"])
    t4 = time.perf_counter()
    brows = inp["buf_rows"]
    return {"summarize": t1 - t0, "select": t2 - t1, "gather": t3 - t2, "attention": t4 - t3,
            "idx": [int(j) for j in idx], "chunk": chunk, "o": o,
            "kbuf_rows": kbuf[brows], "vbuf_rows": vbuf[brows]}


def oracle_sample_flops(inp):
    return attn_flops(len(inp["rows"]), KP * P + NLOC, D, H)


def oracle_baseline(samples, inp, wall_s, cpu_s):
    """The cpu_baseline record from measured samples (no scaling in `value`)."""
    n_rows = len(inp["rows"])
    sample_ms = [1e3 * sum(x[k] for k in ("summarize", "select", "gather", "attention"))
                 for x in samples]
    ms = statistics.median(sample_ms)
    part = {k: statistics.median(1e3 * x[k] for x in samples)
            for k in ("summarize", "select", "gather", "attention")}
    est = N_PAGES * part["summarize"] + part["select"] + part["gather"] + \
        (NQ / n_rows) * part["attention"]
    return {"value": round(oracle_sample_flops(inp) / (ms * 1e-3) / 1e12, 6), "unit": "TFLOP/s",
            "sample_ms": round(ms, 1), "cores": len(os.sched_getaffinity(0)),
            "cpu_util": round(cpu_s / max(wall_s, 1e-9), 2), "kind": "oracle",
            "sample": f"fp64 numpy oracle, measured per sample: 1 page summary (of {N_PAGES}), "
                      f"two-stage retrieval over {N_PAGES} oracle summaries, {KP}-page gather "
                      f"(K and V), attention of {n_rows} query rows (every {SAMPLE_ROWS_STEP}th "
                      f"of {NQ}) x {H} heads over {KP * P + NLOC} keys; value = the sampled "
                      f"rows' attention FLOPs / sample time",
            "samples": len(samples),
            "parts_ms": {k: round(v, 1) for k, v in part.items()},
            "extrapolated_chunk_ms": round(est, 1),
            "extrapolated_is": f"an estimate, not a measurement: {N_PAGES} x summary + retrieval "
                               f"+ gather + {NQ / n_rows:.0f} x sampled attention"}


def cpu_baseline_gpu_arm(c, kp, vp, o_dev, idx_dev, chunk_dev, kbuf_dev=None, vbuf_dev=None,
                        reps=3):
    """The oracle timed on the host cores on the GPU arm's own inputs; also
    checks the benchmarked chunk's indices, sampled rows of its gathered
    buffer and sampled output rows against it."""
    import numpy as np
    import torch

    from sparse_kv_cache_page_gb300 import synth

    inp = oracle_setup(c, lambda j: synth.to_oracle(kp[j]), lambda j: synth.to_oracle(vp[j]))
    oracle_sample(inp)                      # warm-up (first touch of the fp64 buffers)
    w0, c0 = time.perf_counter(), time.process_time()
    samples = [oracle_sample(inp) for _ in range(reps)]
    wall, cpu = time.perf_counter() - w0, time.process_time() - c0
    rec = oracle_baseline(samples, inp, wall, cpu)
    rows = torch.from_numpy(inp["rows"]).to(o_dev.device)
    err = np.abs(o_dev[rows].double().cpu().numpy() - samples[0]["o"])
    parity = {"indices_match": idx_dev.cpu().tolist() == inp["idx"],
              "chunk_match": int(chunk_dev.item()) == inp["chunk"],
              "idx": inp["idx"], "chunk": inp["chunk"],
              "sampled_rows": len(inp["rows"]),
              "attn_max_abs_err": float(err.max()), "attn_mean_abs_err": float(err.mean()),
              "tolerance": "indices and buffer bytes bit-exact; attention max 1e-2, mean 1e-3"}
    if kbuf_dev is not None:
        br = torch.from_numpy(inp["buf_rows"]).to(kbuf_dev.device)
        parity["buffer_rows_match"] = bool(
            np.array_equal(synth.to_oracle(kbuf_dev[br]), samples[0]["kbuf_rows"])
            and np.array_equal(synth.to_oracle(vbuf_dev[br]), samples[0]["vbuf_rows"]))
        parity["buffer_rows_checked"] = len(inp["buf_rows"])
    return rec, parity


def headline_config(world):
    return {"workload": WORKLOAD,
            "l2": "inputs larger than L2 (3.07 GB page bank streamed per step)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "value_is": "attention matmul FLOPs of the chunk / whole-step time"}


def run_reference(args, world, rank):
    """The oracle arm: each step is one measured oracle sample of the chunk
    (oracle_sample) on host cores; ms_per_step is that measured time."""
    from sparse_kv_cache_page_gb300 import synth
    if rank != 0:
        return None
    c = synth.worldattention_case(device="cpu", recall_chunk=3, lazy_pages=True)
    drawn = {}

    def page(j):
        if j not in drawn:
            drawn[j] = c.extra["page"](j, "cpu")
        return drawn[j]

    inp = oracle_setup(c, lambda j: synth.to_oracle(page(j)[0]),
                       lambda j: synth.to_oracle(page(j)[1]))
    for _ in range(args.warmup):
        oracle_sample(inp)
    w0, c0 = time.perf_counter(), time.process_time()
    samples = [oracle_sample(inp) for _ in range(args.steps)]
    wall, cpu = time.perf_counter() - w0, time.process_time() - c0
    rec = oracle_baseline(samples, inp, wall, cpu)
    ms = 1e3 * wall / args.steps
    value = round(oracle_sample_flops(inp) / (ms * 1e-3) / 1e12, 6)
    rec["value"] = value
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), WorldAttention shapes; drawn on the host)",
        "config": headline_config(world),
        "cpu_baseline": rec,
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true",
                    help="skip the PyTorch attention context timing")
    ap.add_argument("--kernel", default="all",
                    choices=["all", "attention", "gather_attention", "gather", "linear", "fp8",
                             "nvfp4"],
                    help="time one kernel alone on its own inputs (for profiling)")
    ap.add_argument("--workload", default="worldattention",
                    choices=["worldattention", "denoise", "hybrid", "hsa", "per_head", "cache",
                             "stress"],
                    help="worldattention: the headline one-layer chunk; denoise: 4 denoising "
                         "steps over a cached 21-frame window; hybrid: + Linformer branch; "
                         "hsa: sparse + Linformer branches in place of dense attention; "
                         "per_head: a page set per head; cache: 12-chunk generation loop "
                         "through the KV cache manager; "
                         "stress: 30 layers with pages in pinned host memory")
    ap.add_argument("--layers", type=int, default=30, help="stress workload: layers")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_init(args)
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    elif args.kernel != "all":
        line = run_one_kernel(args, local)
    elif args.workload == "denoise":
        line = run_denoise(args, world, rank, local)
    elif args.workload == "hybrid":
        line = run_gpu(args, world, rank, local, hybrid=True)
    elif args.workload == "hsa":
        line = run_hsa(args, world, rank, local)
    elif args.workload == "per_head":
        line = run_gpu(args, world, rank, local, per_head=True)
    elif args.workload == "cache":
        line = run_cache(args, world, rank, local)
    elif args.workload == "stress":
        line = run_stress(args, world, rank, local)
    else:
        line = run_gpu(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
