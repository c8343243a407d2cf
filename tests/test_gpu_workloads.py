"""GPU checks of the multi-call workloads against the fp64 oracle:
block-diffusion denoising reuse of a cached window (Inferix summary page, §3
Technical Approach, generation loop; KV Cache Manager, range access) and the
DRAM-tier layer pipeline (WorldAttention review page, HKV tiers L1/L2)."""

import numpy as np
import pytest
import torch

import oracle as O
import sparse_kv_cache_page_gb300 as wa
from sparse_kv_cache_page_gb300 import synth
from sparse_kv_cache_page_gb300.tiered import TieredPipeline, TierLayer
from tests._util import assert_attn_close, np_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_denoising_reuse_of_a_21_frame_window():
    """A 32,760-token window (21 frames of 1,560) is re-attended by a 3-frame
    query block in 4 denoising steps with fresh queries and local KV; the
    window is read, never written, and each step matches the oracle."""
    H, WIN, NQ = 12, 21 * 1560, 4680
    g = lambda shape, t: synth.normal(shape, synth.seed_of("denoise_t", t), DEV, torch.bfloat16)  # noqa: E731
    kw, vw = g((WIN, H, 128), "kw"), g((WIN, H, 128), "vw")
    kw0, vw0 = kw.clone(), vw.clone()
    rows = np.array([0, 1, 999, 2047, 4095, 4600, 4679])
    okw, ovw = np_of(kw), np_of(vw)
    for t in range(4):
        q, kl, vl = g((NQ, H, 128), ("q", t)), g((NQ, H, 128), ("kl", t)), g((NQ, H, 128), ("vl", t))
        o = torch.empty((NQ, H, 128), dtype=torch.float32, device=DEV)
        wa.wa_block_attn(q, kw, vw, kl, vl, o)
        wa.wa_check()
        ref, _ = O.block_attn(np_of(q), okw, ovw, np_of(kl), np_of(vl), rows=rows)
        assert_attn_close(o[torch.from_numpy(rows).to(DEV)], ref, torch.bfloat16, f"step {t}")
    assert torch.equal(kw, kw0) and torch.equal(vw, vw0)


@pytest.mark.parametrize("mode", ["pipeline", "serial", "direct", "fp8", "fp8_pipeline", "nvfp4",
                                  "nvfp4_pipeline"])
def test_tiered_layer_pipeline(mode):
    """Three layers, 12 pages of 700 tokens each in pinned host memory, top-4
    per layer; the double-buffered side-stream fetch must give every layer the
    pages the oracle picks (bit-exact) and the oracle's attention.  The fp8
    modes fetch the FP8 copy of the pages and the nvfp4 modes the NVFP4 copy
    (compressed DRAM tier): the reference attention then runs over the
    oracle's decoded pages."""
    H, P, NPG, NQ, NLOC, NL = 2, 700, 12, 300, 90, 3
    fp8, nv = mode.startswith("fp8"), mode.startswith("nvfp4")
    layers, refs = [], []
    for l in range(NL):
        c = synth.make_chunk_case(f"tier{l}", n_heads=H, head_dim=128, page_tokens=P,
                                  n_pages=NPG, pages_per_chunk=1, n_chunks=0, prompt_dim=0,
                                  k_p=4, n_q=NQ, n_loc=NLOC, dtype=torch.bfloat16,
                                  plant_pages=[l, 5 + l], plant_strength=0.3)
        kbar = torch.empty((NPG, H, 128), dtype=torch.float32, device=DEV)
        wa.wa_page_summarize(c.k_pages.to(DEV), kbar)
        out = torch.empty((NQ, H, 128), dtype=torch.float32, device=DEV)
        codes = []
        for pages in (c.k_pages, c.v_pages):
            pc = torch.empty((NPG, P, H, 128), dtype=torch.uint8).pin_memory()
            ps = torch.empty((NPG, P, H), dtype=torch.float32).pin_memory()
            wa.wa_fp8_encode(pages.to(DEV).reshape(NPG * P, H, 128), pc, ps)
            codes += [pc, ps]
        nvc = []
        for pages in (c.k_pages, c.v_pages):
            arrs = (torch.empty((NPG, P, H, 64), dtype=torch.uint8).pin_memory(),
                    torch.empty((NPG, P, H, 8), dtype=torch.uint8).pin_memory(),
                    torch.empty((NPG, P, H), dtype=torch.float32).pin_memory())
            wa.wa_nvfp4_encode(pages.to(DEV).reshape(NPG * P, H, 128), *arrs)
            nvc.append(arrs)
        wa.wa_check()
        layers.append(TierLayer(c.q.to(DEV), c.k_loc.to(DEV), c.v_loc.to(DEV), kbar,
                                c.k_pages.pin_memory(), c.v_pages.pin_memory(), out, *codes,
                                k_nv=nvc[0], v_nv=nvc[1]))
        okp, ovp = np_of(c.k_pages), np_of(c.v_pages)
        idx, _, _ = O.select_pages(np_of(c.q), O.page_summarize(okp), None, None, 1, 4)
        if fp8:
            def dec(pg):
                cc, ss = O.fp8_encode_rows(pg.reshape(NPG * P, H, 128))
                return O.bf16_bits(O.fp8_decode_rows(cc, ss)).reshape(NPG, P, H, 128)
            okp, ovp = dec(okp), dec(ovp)
        if nv:
            def dec4(pg):
                return O.bf16_bits(O.nvfp4_decode_rows(*O.nvfp4_encode_rows(
                    pg.reshape(NPG * P, H, 128)))).reshape(NPG, P, H, 128)
            okp, ovp = dec4(okp), dec4(ovp)
        ref, _ = O.block_attn(np_of(c.q), O.gather_pages(okp, idx), O.gather_pages(ovp, idx),
                              np_of(c.k_loc), np_of(c.v_loc))
        refs.append((idx, ref))
    pipe = TieredPipeline(4, P, H, 128)
    idx_h = pipe.run(layers, mode)
    torch.cuda.synchronize()
    wa.wa_check()
    for l in range(NL):
        assert idx_h[l].cpu().tolist() == refs[l][0].tolist()
        assert {l, 5 + l} <= set(refs[l][0].tolist())
        assert_attn_close(layers[l].out, refs[l][1], torch.bfloat16, f"layer {l}")
