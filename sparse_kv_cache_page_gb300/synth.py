"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path (via the binding) and the CPU oracle
are fed from it.  Values are i.i.d. N(0, 1) fp32 from a torch generator seeded
per (workload, layer, tensor name), then rounded to bf16 by round-to-nearest-
even where the workload is bf16.  Small cases are drawn on the CPU; full-size
cases may be drawn on the GPU (same recipe, torch's CUDA generator) so that a
3 GB page bank does not take a minute of host time.

Geometry (WorldAttention review page, HKV section): a frame is 1,560 tokens,
a page is 8 frames, K_p = 4, so the active KV is 4 x 8 x 1,560 = 49,920 tokens.
"""

from __future__ import annotations

import zlib
from dataclasses import dataclass, field

import numpy as np
import torch

SEED_BASE = 20261202

TOKENS_PER_FRAME = 1560
FRAMES_PER_PAGE = 8
PAGE_TOKENS = TOKENS_PER_FRAME * FRAMES_PER_PAGE  # 12,480
K_P = 4
ACTIVE_TOKENS = K_P * PAGE_TOKENS  # 49,920


def seed_of(*parts) -> int:
    """Stable 63-bit seed from the base seed and a tuple of names/ints."""
    h = zlib.crc32(repr((SEED_BASE,) + tuple(parts)).encode())
    return (SEED_BASE * 1_000_003 + h) & ((1 << 63) - 1)


def normal(shape, seed: int, device="cpu", dtype=torch.float32, std: float = 1.0) -> torch.Tensor:
    """i.i.d. N(0, std^2) drawn in fp32, then cast (RNE) to ``dtype``."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, device=dev, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def to_oracle(t: torch.Tensor) -> np.ndarray:
    """Host numpy view for the oracle: bf16 as uint16 bit patterns, fp32 as is."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float32, torch.float64, torch.int32, torch.int64):
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")


@dataclass
class ChunkCase:
    """Inputs of one chunk step: KV page bank, prompts, queries, local KV."""
    name: str
    n_heads: int
    head_dim: int
    page_tokens: int
    n_pages: int
    pages_per_chunk: int
    n_chunks: int          # past chunks with a prompt embedding (0: no prompt stage)
    prompt_dim: int
    k_p: int
    n_q: int
    n_loc: int
    dtype: torch.dtype
    k_pages: torch.Tensor = None   # [n_pages][P][H][d]
    v_pages: torch.Tensor = None
    q: torch.Tensor = None         # [n_q][H][d]
    k_loc: torch.Tensor = None     # [n_loc][H][d]
    v_loc: torch.Tensor = None
    prompt_cur: torch.Tensor = None     # [prompt_dim] fp32
    prompt_chunks: torch.Tensor = None  # [n_chunks][prompt_dim] fp32
    extra: dict = field(default_factory=dict)


def make_chunk_case(name: str, *, n_heads: int, head_dim: int, page_tokens: int, n_pages: int,
                    pages_per_chunk: int, n_chunks: int, prompt_dim: int, k_p: int, n_q: int,
                    n_loc: int, dtype=torch.bfloat16, device="cpu", layer: int = 0,
                    plant_pages=None, plant_strength: float = 0.0,
                    recall_chunk: int | None = None, std: float = 1.0,
                    lazy_pages: bool = False) -> ChunkCase:
    """Draw one chunk case.  Optional structure (input construction only):

    * ``plant_pages`` / ``plant_strength``: a per-head direction u_h ~ N(0,1)
      is added, times the strength, to every key of the listed pages and to
      every query, so those pages are the relevant ones.
    * ``recall_chunk``: the current prompt embedding is that past chunk's
      embedding plus half-scale noise (the "throw the red ball again" recall).
    * ``lazy_pages``: leave the page bank undrawn; ``case.extra["page"](j)``
      draws page j on demand.
    """
    H, d = n_heads, head_dim
    c = ChunkCase(name, H, d, page_tokens, n_pages, pages_per_chunk, n_chunks, prompt_dim, k_p,
                  n_q, n_loc, dtype)
    s = lambda t: seed_of(name, layer, t)  # noqa: E731
    u = normal((H, d), s("plant_dir"), device) if plant_pages else None

    def page(j, dev=device):
        """(K, V) of page j, [P][H][d]; the same values whether drawn eagerly
        with the bank or later on their own."""
        kj = normal((page_tokens, H, d), s(("k_page", j)), dev, std=std)
        if plant_pages and j in plant_pages:
            kj += plant_strength * u.to(dev)
        vj = normal((page_tokens, H, d), s(("v_page", j)), dev, dtype, std=std)
        return kj.to(dtype), vj

    c.extra["page"] = page
    if not lazy_pages:
        kp = torch.empty((n_pages, page_tokens, H, d), dtype=dtype, device=device)
        vp = torch.empty_like(kp)
        for j in range(n_pages):
            kp[j], vp[j] = page(j)
        c.k_pages, c.v_pages = kp, vp
    q = normal((n_q, H, d), s("q"), device, std=std)
    if plant_pages:
        q += plant_strength * u
    c.q = q.to(dtype)
    c.k_loc = normal((n_loc, H, d), s("k_loc"), device, dtype, std=std)
    c.v_loc = normal((n_loc, H, d), s("v_loc"), device, dtype, std=std)
    if n_chunks > 0:
        c.prompt_chunks = normal((n_chunks, prompt_dim), s("prompt_chunks"), device)
        cur = normal((prompt_dim,), s("prompt_cur"), device)
        if recall_chunk is not None:
            cur = c.prompt_chunks[recall_chunk] + 0.5 * cur
        c.prompt_cur = cur
    return c


def tiny_fp32_case(**kw) -> ChunkCase:
    """Tiny fp32 oracle check: 1 head, d_k = 64, frame = 16 tokens, page = 2
    frames, 8 pages in 2 chunks, prompt embeddings of dim 32, K_p = 2, a query
    chunk of 1 frame plus its local KV of 1 frame."""
    args = dict(n_heads=1, head_dim=64, page_tokens=32, n_pages=8, pages_per_chunk=4,
                n_chunks=2, prompt_dim=32, k_p=2, n_q=16, n_loc=16, dtype=torch.float32)
    args.update(kw)
    return make_chunk_case("tiny_fp32", **args)


def worldattention_case(device="cpu", **kw) -> ChunkCase:
    """One layer at the WorldAttention shape: 12 heads, d_k = 128, bf16,
    40 cached pages of 12,480 tokens in 5 chunks of 8 pages, prompt embeddings
    of dim 4096, K_p = 4 (49,920 tokens), 4,680 query tokens + 4,680 local."""
    args = dict(n_heads=12, head_dim=128, page_tokens=PAGE_TOKENS, n_pages=40, pages_per_chunk=8,
                n_chunks=5, prompt_dim=4096, k_p=K_P, n_q=3 * TOKENS_PER_FRAME,
                n_loc=3 * TOKENS_PER_FRAME, dtype=torch.bfloat16)
    args.update(kw)
    return make_chunk_case("worldattention_1layer", device=device, **args)


def peaked_queries(k_src: torch.Tensor, n_q: int, seed: int, gain: float = 8.0) -> tuple:
    """Queries that each point at one key: q_i = gain * k_{pi(i)} with pi a
    seeded random choice of source rows.  Returns (q, pi)."""
    g = torch.Generator().manual_seed(int(seed))
    pi = torch.randint(0, k_src.shape[0], (n_q,), generator=g)
    q = (gain * k_src[pi.to(k_src.device)].float()).to(k_src.dtype)
    return q, pi


# Minute-long stress workload: layers one after another, 120 cached pages per
# layer whose bodies live in pinned host memory (one page store shared by the
# layers), each layer with its own queries and local KV.
STRESS_PAGES = 120
STRESS_LAYERS = 30


def stress_page(j: int, device="cpu", rank: int = 0, n_heads: int = 12, head_dim: int = 128,
                page_tokens: int = PAGE_TOKENS):
    """(K, V) of page j of the stress workload's page store, [P][H][d] bf16."""
    s = lambda t: seed_of("stress", rank, t)  # noqa: E731
    shape = (page_tokens, n_heads, head_dim)
    return (normal(shape, s(("k", j)), device, torch.bfloat16),
            normal(shape, s(("v", j)), device, torch.bfloat16))


def stress_layer(l: int, device="cpu", rank: int = 0, n_heads: int = 12, head_dim: int = 128,
                 n_q: int = 3 * TOKENS_PER_FRAME, n_loc: int = 3 * TOKENS_PER_FRAME):
    """(Q, K_loc, V_loc) of layer l of the stress workload, [tokens][H][d] bf16."""
    s = lambda t: seed_of("stress", rank, t)  # noqa: E731
    return (normal((n_q, n_heads, head_dim), s(("q", l)), device, torch.bfloat16),
            normal((n_loc, n_heads, head_dim), s(("kl", l)), device, torch.bfloat16),
            normal((n_loc, n_heads, head_dim), s(("vl", l)), device, torch.bfloat16))
