"""Layer pipeline over the DRAM tier of the page cache.

WorldAttention (review page), HKV section, tiers L1/L2 (Fig. 2): GPU HBM holds
only the retrieved pages plus the prompt and page indices, while the pages of
chunks not in use live in CPU DRAM.  Inferix (summary page), KV Cache Manager:
offloading to main memory, with selected blocks loaded back before attention.

Here each layer's page bodies sit in pinned host memory and its page
summaries in HBM.  For a run of layers: retrieval for every layer on the main
stream, one device->host copy of all page indices, then per layer a
copy-engine fetch of the K_p selected pages (wa_gather_pages from pinned host
memory) on a side stream into one of two device buffers, and attention on the
main stream once that layer's copy has landed.  The fetch of layer l+1 thus
overlaps the attention of layer l; a buffer is refilled only after the
attention that read it two layers earlier has finished.

Every step runs in libwa; this module only orders calls on streams.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from . import (wa_block_attn, wa_gather_pages, wa_gather_pages_fp8, wa_gather_pages_nvfp4,
               wa_select_pages)


@dataclass
class TierLayer:
    q: torch.Tensor            # [n_q][H][d] device
    k_loc: torch.Tensor        # [n_loc][H][d] device
    v_loc: torch.Tensor
    kbar: torch.Tensor         # [n_pages][H][d] fp32 device (summaries of the host pages)
    k_host: torch.Tensor       # [n_pages][P][H][d] pinned host
    v_host: torch.Tensor
    out: torch.Tensor          # [n_q][H][d] device, fp32 or the input dtype
    # compressed copy of the page bodies (FP8 E4M3 codes [n_pages][P][H][d] and
    # scales [n_pages][P][H], pinned host), used by the "fp8" mode
    k_codes: torch.Tensor | None = None
    k_scales: torch.Tensor | None = None
    v_codes: torch.Tensor | None = None
    v_scales: torch.Tensor | None = None
    # NVFP4 copy (E2M1 codes [n_pages][P][H][d/2], E4M3 block scales
    # [n_pages][P][H][d/16], fp32 row scales [n_pages][P][H], pinned host), used
    # by the "nvfp4" modes
    k_nv: tuple | None = None
    v_nv: tuple | None = None


class TieredPipeline:
    """Double-buffered host->device page fetch overlapped with attention."""

    def __init__(self, k_p: int, page_tokens: int, n_heads: int, head_dim: int,
                 dtype=torch.bfloat16, device="cuda"):
        self.k_p = k_p
        shape = (k_p * page_tokens, n_heads, head_dim)
        self.bufs = [(torch.empty(shape, dtype=dtype, device=device),
                      torch.empty(shape, dtype=dtype, device=device)) for _ in range(2)]
        self.side = torch.cuda.Stream(device=device)
        self.device = device
        self.k_p, self.page_tokens, self.n_heads, self.head_dim = k_p, page_tokens, n_heads, head_dim
        self.stage = None     # FP8 staging pages, allocated on first "fp8_pipeline" run
        self.stage4 = None    # NVFP4 staging pages, allocated on first "nvfp4_pipeline" run

    def _staging(self):
        if self.stage is None:
            P, H, d = self.page_tokens, self.n_heads, self.head_dim
            mk = lambda *shape, dt: torch.empty(shape, dtype=dt, device=self.device)  # noqa: E731
            self.stage = [dict(kc=mk(self.k_p, P, H, d, dt=torch.uint8),
                               vc=mk(self.k_p, P, H, d, dt=torch.uint8),
                               ks=mk(self.k_p, P, H, dt=torch.float32),
                               vs=mk(self.k_p, P, H, dt=torch.float32)) for _ in range(2)]
            self.ident = torch.arange(self.k_p, dtype=torch.int32, device=self.device)
        return self.stage

    def _staging4(self):
        if self.stage4 is None:
            P, H, d = self.page_tokens, self.n_heads, self.head_dim
            mk = lambda *shape, dt: torch.empty(shape, dtype=dt, device=self.device)  # noqa: E731
            self.stage4 = [{t: (mk(self.k_p, P, H, d // 2, dt=torch.uint8),
                                mk(self.k_p, P, H, d // 16, dt=torch.uint8),
                                mk(self.k_p, P, H, dt=torch.float32)) for t in ("k", "v")}
                           for _ in range(2)]
            self.ident = torch.arange(self.k_p, dtype=torch.int32, device=self.device)
        return self.stage4

    def _fetch_nvfp4(self, ly, idx_host, st):
        """Copy-engine fetch of k_p NVFP4 pages into a staging slot: codes, block
        scales and row scales each viewed as one row of 2-byte elements per page
        (16-byte rows need page_tokens * n_heads % 4 == 0)."""
        page = lambda t: t.view(t.shape[0], 1, 1, -1).view(torch.bfloat16)  # noqa: E731
        for a in range(3):
            kb, vb = page(st["k"][a]), page(st["v"][a])
            wa_gather_pages(page(ly.k_nv[a]), page(ly.v_nv[a]), None, idx_host,
                            kb.view(self.k_p, 1, -1), vb.view(self.k_p, 1, -1), stream=self.side)

    def _fetch_fp8(self, ly, idx_host, st):
        """Copy-engine fetch of k_p FP8 pages (codes viewed as 2-byte elements,
        scales as one-float rows) into a staging slot."""
        P, H, d = self.page_tokens, self.n_heads, self.head_dim
        bf = lambda t: t.view(torch.bfloat16)  # noqa: E731
        wa_gather_pages(bf(ly.k_codes), bf(ly.v_codes), None, idx_host, bf(st["kc"]), bf(st["vc"]),
                        stream=self.side)
        # a page's scales as one row of P*H floats (16-byte rows need P*H % 4 == 0)
        wa_gather_pages(ly.k_scales.view(-1, 1, 1, P * H), ly.v_scales.view(-1, 1, 1, P * H), None,
                        idx_host, st["ks"].view(-1, 1, P * H), st["vs"].view(-1, 1, P * H),
                        stream=self.side)

    def run(self, layers, mode: str = "pipeline", on_layer=None):
        """Run all layers.  mode: "pipeline" (copy-engine fetches on a side
        stream overlap attention), "serial" (each layer's copy, then its
        attention, on one stream), "direct" (the gather kernel reads the pinned
        pages over the CPU-GPU link on the side stream, indices stay on the
        device, no host round trip), "copy" / "attn" (one half only, for
        timing), "fp8" (as "direct", but the pages cross the link as FP8 codes
        and scales and are decoded to bf16 on the device: the compressed DRAM
        tier), "fp8_pipeline" (the FP8 pages fetched by the copy engine on the
        side stream into a staging slot and decoded there, overlapping the
        previous layer's attention), "nvfp4" / "nvfp4_pipeline" (the same with the
        NVFP4 copy: E2M1 codes and two levels of scales).  ``on_layer(l, k_buf,
        v_buf)``, if given, is called once layer l's attention is enqueued on
        the current stream and before the buffers it read may be refilled: work
        it enqueues on that stream sees the buffers as the attention did.
        Returns the page indices [n_layers][k_p] (int32; pinned host memory, or
        device memory in the "direct", "fp8" and "nvfp4" modes)."""
        main = torch.cuda.current_stream(self.device)
        n = len(layers)
        idx = torch.empty((n, self.k_p), dtype=torch.int32, device=self.device)
        for l, ly in enumerate(layers):
            wa_select_pages(ly.q, ly.kbar, None, None, 1, self.k_p, idx[l])
        if mode in ("direct", "fp8", "nvfp4"):
            return self._run_direct(layers, idx, main, codec=mode, on_layer=on_layer)
        idx_h = torch.empty((n, self.k_p), dtype=torch.int32, pin_memory=True)
        idx_h.copy_(idx, non_blocking=True)
        main.synchronize()                         # indices reach the host once
        ev_copy = [torch.cuda.Event() for _ in range(n)]
        ev_attn = [torch.cuda.Event() for _ in range(n)]
        if mode in ("fp8_pipeline", "nvfp4_pipeline"):
            # side stream: fetch layer l's compressed pages into a staging slot,
            # then (once layer l-2's attention has read the bf16 buffer) decode
            # them; the main stream only runs attention
            nv = mode == "nvfp4_pipeline"
            stage = self._staging4() if nv else self._staging()
            for l, ly in enumerate(layers):
                kb, vb = self.bufs[l % 2]
                st = stage[l % 2]
                with torch.cuda.stream(self.side):
                    (self._fetch_nvfp4 if nv else self._fetch_fp8)(ly, idx_h[l], st)
                    if l >= 2:
                        self.side.wait_event(ev_attn[l - 2])
                    if nv:
                        wa_gather_pages_nvfp4(*st["k"], self.ident, kb, stream=self.side)
                        wa_gather_pages_nvfp4(*st["v"], self.ident, vb, stream=self.side)
                    else:
                        wa_gather_pages_fp8(st["kc"], st["ks"], self.ident, kb, stream=self.side)
                        wa_gather_pages_fp8(st["vc"], st["vs"], self.ident, vb, stream=self.side)
                    ev_copy[l].record(self.side)
                main.wait_event(ev_copy[l])
                wa_block_attn(ly.q, kb, vb, ly.k_loc, ly.v_loc, ly.out)
                if on_layer is not None:
                    on_layer(l, kb, vb)
                ev_attn[l].record(main)
            main.wait_stream(self.side)
            return idx_h
        for l, ly in enumerate(layers):
            kb, vb = self.bufs[l % 2]
            if mode == "serial":
                wa_gather_pages(ly.k_host, ly.v_host, None, idx_h[l], kb, vb)
            elif mode != "attn":
                with torch.cuda.stream(self.side):
                    if l >= 2:
                        self.side.wait_event(ev_attn[l - 2])
                    wa_gather_pages(ly.k_host, ly.v_host, None, idx_h[l], kb, vb,
                                    stream=self.side)
                    ev_copy[l].record(self.side)
            if mode != "copy":
                if mode == "pipeline":
                    main.wait_event(ev_copy[l])
                wa_block_attn(ly.q, kb, vb, ly.k_loc, ly.v_loc, ly.out)
                if on_layer is not None:
                    on_layer(l, kb, vb)
                ev_attn[l].record(main)
        main.wait_stream(self.side)
        return idx_h

    def _run_direct(self, layers, idx, main, codec="direct", on_layer=None):
        ev_sel = torch.cuda.Event()
        ev_sel.record(main)
        n = len(layers)
        ev_copy = [torch.cuda.Event() for _ in range(n)]
        ev_attn = [torch.cuda.Event() for _ in range(n)]
        for l, ly in enumerate(layers):
            kb, vb = self.bufs[l % 2]
            with torch.cuda.stream(self.side):
                self.side.wait_event(ev_sel if l < 2 else ev_attn[l - 2])
                if codec == "fp8":
                    wa_gather_pages_fp8(ly.k_codes, ly.k_scales, idx[l], kb, stream=self.side)
                    wa_gather_pages_fp8(ly.v_codes, ly.v_scales, idx[l], vb, stream=self.side)
                elif codec == "nvfp4":
                    wa_gather_pages_nvfp4(*ly.k_nv, idx[l], kb, stream=self.side)
                    wa_gather_pages_nvfp4(*ly.v_nv, idx[l], vb, stream=self.side)
                else:
                    wa_gather_pages(ly.k_host, ly.v_host, idx[l], None, kb, vb, stream=self.side)
                ev_copy[l].record(self.side)
            main.wait_event(ev_copy[l])
            wa_block_attn(ly.q, kb, vb, ly.k_loc, ly.v_loc, ly.out)
            if on_layer is not None:
                on_layer(l, kb, vb)
            ev_attn[l].record(main)
        main.wait_stream(self.side)
        return idx
