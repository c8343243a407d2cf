"""fp64 CPU oracle for the page-retrieval sparse-attention path of one chunk.

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product path.  Shares no
code with the CUDA library: it reads plain numpy arrays and does every step in
float64 with numpy, in the order the pages state the method.

Sources (page title, then section / equation / figure on that page):

* [WA]  "WorldAttention: An Efficient Attention Architecture for Interactive
  Video World Models" (review page).  HKV section (paper §3.1 HKV): pages of
  8 frames x 1,560 tokens, prompt-stage top-1 chunk by cosine similarity,
  page-stage score alpha_{m,j} = Qbar^T Kbar_{m,j} / sqrt(d_k), top-K_p with
  K_p = 4.  HSA section (paper §3.2 HSA): Linformer-style per-head E_K, E_V in
  R^{L x r}; per-head gate fusion.  "How It Works" steps 3-5 (worked example:
  4 x 8 x 1560 = 49,920 active tokens).  Custom-kernels prong (Fig. 1):
  retrieved pages reorganised into one contiguous buffer.
* [IX]  "Inferix: A Block-Diffusion based Next-Generation Inference Engine for
  World Simulation" (summary page).  §3 Technical Approach, generation loop
  Step 3: Attention(Q_t, [K_cache (+) K_t], [V_cache (+) V_t]), bidirectional
  inside the block, no mask.
* [EIN] einsum tutorial page, "Step 7: reading the attention string":
  logits = einsum('bhqd,bhkd->bhqk', q, k).

Readings taken where the pages are silent or garbled (each also listed in the
design notes):

* One page set per layer, shared by all heads: the page score sums the
  per-head dot products, alpha_j = sum_h Qbar_h . Kbar_{j,h} / sqrt(d_k).
* Qbar is the mean over the chunk's query tokens; Kbar_j the mean over all
  tokens of page j (means, not sums).
* Prompt stage: candidates are the pages of the top-1 chunk; with no prompt
  embeddings every page is a candidate.  A zero-norm vector has cosine 0.
  Exact ties go to the lowest chunk index.
* Top-K_p ties go to the lowest page index; the selected indices are returned
  in ascending page order (temporal order), and the gathered buffer holds the
  pages in that order, page-major.
* The Linformer equation is missing on the page; read as Linformer:
  K'_h = E_K^(h)T K_h, V'_h = E_V^(h)T V_h, O_lin = softmax(Q_h K'_h^T s) V'_h,
  with E rows aligned to [gathered buffer ; local KV].
* The gate equation is missing on the page; fused output is
  O = w_attn[h] * O_attn + w_lin[h] * O_lin, default weights 1 and 1.

Array conventions: token-major [tokens][H][d]; pages [n_pages][P][H][d];
bf16 values are passed as np.uint16 bit patterns and decoded exactly.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "as_f64",
    "decode_bf16",
    "page_summarize",
    "mean_query",
    "cosine",
    "prompt_top1",
    "page_scores",
    "topk_pages",
    "candidate_pages",
    "select_pages",
    "gather_pages",
    "attention_rows",
    "block_attn",
    "linformer_project",
    "linear_branch",
    "fuse_branches",
]


# ----------------------------------------------------------------------------
# exact decoding
# ----------------------------------------------------------------------------

def decode_bf16(u16: np.ndarray) -> np.ndarray:
    """Exact bf16 -> fp64: a bf16 is the top half of an IEEE fp32 word."""
    u16 = np.ascontiguousarray(u16, dtype=np.uint16)
    f32 = (u16.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return f32.astype(np.float64)


def as_f64(a: np.ndarray) -> np.ndarray:
    """Decode an input array to fp64: uint16 means bf16 bit patterns."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return decode_bf16(a)
    if a.dtype in (np.float32, np.float64):
        return a.astype(np.float64)
    raise TypeError(f"unsupported oracle input dtype {a.dtype}")


# ----------------------------------------------------------------------------
# [WA] HKV: page summaries and the mean query
# ----------------------------------------------------------------------------

def page_summarize(k_pages: np.ndarray) -> np.ndarray:
    """Kbar[j, h, :] = (1/P) sum_t K[j, t, h, :]  ([WA] HKV, page mean key).

    k_pages: [n_pages][P][H][d] (bf16 bits or float).  Returns fp64 [n_pages][H][d].
    """
    k = as_f64(k_pages)
    n_pages, p_tok = k.shape[0], k.shape[1]
    out = np.empty((n_pages,) + k.shape[2:], dtype=np.float64)
    for j in range(n_pages):
        out[j] = k[j].sum(axis=0) / p_tok
    return out


def mean_query(q: np.ndarray) -> np.ndarray:
    """Qbar[h, :] = (1/n_q) sum_i Q[i, h, :]  ([WA] HKV, the chunk's mean query)."""
    qq = as_f64(q)
    return qq.sum(axis=0) / qq.shape[0]


# ----------------------------------------------------------------------------
# [WA] HKV: two-stage retrieval
# ----------------------------------------------------------------------------

def cosine(a: np.ndarray, b: np.ndarray) -> float:
    """cos(a, b) = a.b / (|a| |b|); 0 when either norm is 0 (reading)."""
    a = as_f64(a)
    b = as_f64(b)
    na = math.sqrt(float(np.dot(a, a)))
    nb = math.sqrt(float(np.dot(b, b)))
    if na == 0.0 or nb == 0.0:
        return 0.0
    return float(np.dot(a, b)) / (na * nb)


def prompt_top1(prompt_cur: np.ndarray, prompt_chunks: np.ndarray) -> int:
    """Prompt stage ([WA] HKV, stage 1): the past chunk whose prompt embedding
    has the largest cosine similarity with the current prompt embedding.
    Exact ties go to the lowest chunk index."""
    best_m, best_c = -1, -math.inf
    for m in range(prompt_chunks.shape[0]):
        c = cosine(prompt_cur, prompt_chunks[m])
        if c > best_c:  # strict: the first (lowest) index wins a tie
            best_m, best_c = m, c
    return best_m


def page_scores(qbar: np.ndarray, kbar: np.ndarray, pages, head_dim: int) -> np.ndarray:
    """alpha_j = Qbar^T Kbar_j / sqrt(d_k) for each page j in ``pages``
    ([WA] HKV, stage 2), summed over heads (one page set per layer)."""
    qb = as_f64(qbar)
    kb = as_f64(kbar)
    return np.array([float((qb * kb[j]).sum()) / math.sqrt(head_dim) for j in pages],
                    dtype=np.float64)


def topk_pages(alpha: np.ndarray, pages, k_p: int):
    """Top-K_p pages by alpha; ties to the lowest page index; the result is
    sorted ascending by page index.  Returns (idx, alpha_of_idx)."""
    pages = list(pages)
    if k_p > len(pages):
        raise ValueError("k_p exceeds the number of candidate pages")
    order = sorted(range(len(pages)), key=lambda i: (-alpha[i], pages[i]))
    chosen = sorted(order[:k_p], key=lambda i: pages[i])
    idx = np.array([pages[i] for i in chosen], dtype=np.int32)
    sc = np.array([alpha[i] for i in chosen], dtype=np.float64)
    return idx, sc


def candidate_pages(n_pages: int, chunk: int, pages_per_chunk: int):
    """Pages of chunk m are m*ppc .. (m+1)*ppc-1; chunk -1 means all pages."""
    if chunk < 0:
        return list(range(n_pages))
    return list(range(chunk * pages_per_chunk, (chunk + 1) * pages_per_chunk))


def select_pages(q, kbar, prompt_cur, prompt_chunks, pages_per_chunk: int, k_p: int):
    """Both retrieval stages for one chunk.  With no prompt embeddings
    (prompt_chunks is None or has 0 rows) the prompt stage is skipped and all
    pages are candidates.  Returns (idx, alpha_of_idx, chunk)."""
    kb = as_f64(kbar)
    n_pages, _, d = kb.shape
    qbar = mean_query(q)
    if prompt_chunks is None or len(prompt_chunks) == 0:
        chunk = -1
    else:
        chunk = prompt_top1(prompt_cur, prompt_chunks)
    cand = candidate_pages(n_pages, chunk, pages_per_chunk)
    alpha = page_scores(qbar, kb, cand, d)
    idx, sc = topk_pages(alpha, cand, k_p)
    return idx, sc, chunk


# ----------------------------------------------------------------------------
# [WA] custom-kernels prong: contiguous buffer of the retrieved pages
# ----------------------------------------------------------------------------

def gather_pages(pages: np.ndarray, idx) -> np.ndarray:
    """buf[s*P + t] = pages[idx[s]][t]: a byte copy, page-major, in idx order."""
    parts = [np.asarray(pages[int(j)]) for j in idx]
    return np.concatenate(parts, axis=0)


# ----------------------------------------------------------------------------
# [IX] Step 3 / [EIN] Step 7: softmax attention, textbook form
# ----------------------------------------------------------------------------

def attention_rows(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """Dense attention for a block of query rows of one head, materialised:

        S = scale * q k^T          (the 'bhqd,bhkd->bhqk' contraction)
        P = exp(S - rowmax) / rowsum
        O = P v,   LSE = log sum_k exp(S)

    q_rows [n][d], k/v [L][d] as fp64.  Returns (O [n][d], LSE [n], P [n][L])."""
    s = scale * (q_rows @ k.T)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    p = e / l
    o = p @ v
    lse = (m + np.log(l))[:, 0]
    return o, lse, p


def block_attn(q, k_main, v_main, k_loc, v_loc, scale: float | None = None,
               rows=None, heads=None):
    """Attention of the chunk's queries over [K_main ; K_loc], [V_main ; V_loc]
    ([IX] Step 3: cached KV (+) the block's own KV; no mask).

    q [n_q][H][d]; k_main/v_main [n_main][H][d]; k_loc/v_loc [n_loc][H][d]
    (either segment may have 0 rows).  scale None or <= 0 means 1/sqrt(d).
    ``rows``/``heads`` restrict the computation to a sample of query rows and
    heads.  Returns (O [len(rows)][len(heads)][d], LSE [len(heads)][len(rows)]).
    """
    qq = as_f64(q)
    n_q, n_h, d = qq.shape
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(d)
    segs_k = [as_f64(x) for x in (k_main, k_loc) if x is not None and len(x) > 0]
    segs_v = [as_f64(x) for x in (v_main, v_loc) if x is not None and len(x) > 0]
    kk = np.concatenate(segs_k, axis=0)
    vv = np.concatenate(segs_v, axis=0)
    rows = np.arange(n_q) if rows is None else np.asarray(rows)
    heads = np.arange(n_h) if heads is None else np.asarray(heads)
    o = np.empty((len(rows), len(heads), d), dtype=np.float64)
    lse = np.empty((len(heads), len(rows)), dtype=np.float64)
    for hi, h in enumerate(heads):
        oh, lh, _ = attention_rows(qq[rows, h, :], kk[:, h, :], vv[:, h, :], scale)
        o[:, hi, :] = oh
        lse[hi, :] = lh
    return o, lse


# ----------------------------------------------------------------------------
# [WA] HSA: Linformer-style low-rank branch and the gate fusion
# ----------------------------------------------------------------------------

def linformer_project(kv_cat: np.ndarray, e: np.ndarray) -> np.ndarray:
    """X'_h = E^(h)T X_h for each head: kv_cat [L][H][d], e [H][L][r] -> [H][r][d]."""
    x = np.asarray(kv_cat)
    n_h = x.shape[1]
    # one head at a time keeps the fp64 copies small at full size
    return np.stack([as_f64(e[h]).T @ as_f64(x[:, h, :]) for h in range(n_h)], axis=0)


def linear_branch(q, k_cat, v_cat, e_k, e_v, scale: float | None = None, rows=None):
    """O_lin = softmax(Q_h K'_h^T * scale) V'_h per head, with K' and V' the
    rank-r projections of [buffer ; local] ([WA] HSA, linear branch).
    Returns O_lin [len(rows)][H][d] in fp64."""
    qq = as_f64(q)
    n_q, n_h, d = qq.shape
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(d)
    kp = linformer_project(k_cat, e_k)
    vp = linformer_project(v_cat, e_v)
    rows = np.arange(n_q) if rows is None else np.asarray(rows)
    out = np.empty((len(rows), n_h, d), dtype=np.float64)
    for h in range(n_h):
        oh, _, _ = attention_rows(qq[rows, h, :], kp[h], vp[h], scale)
        out[:, h, :] = oh
    return out


def fuse_branches(o_attn: np.ndarray, o_lin: np.ndarray, w_attn=None, w_lin=None):
    """O = w_attn[h] * O_attn + w_lin[h] * O_lin ([WA] HSA, per-head gate);
    missing weights are 1 (the two branches summed with equal weight)."""
    n_h = o_attn.shape[1]
    wa = np.ones(n_h) if w_attn is None else np.asarray(w_attn, dtype=np.float64)
    wl = np.ones(n_h) if w_lin is None else np.asarray(w_lin, dtype=np.float64)
    return o_attn * wa[None, :, None] + o_lin * wl[None, :, None]
