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
* Per-head page selection (the per-head variant of the page stage): the
  prompt stage is shared; head h scores pages on its own slice,
  alpha_{j,h} = Qbar_h . Kbar_{j,h} / sqrt(d_k), keeps its own top-K_p (same
  tie rule, ascending), and the buffer keeps the token-major layout with head
  h's slice taken from head h's pages.
* Compressed DRAM tier (the pages name FP8 / FP4 storage only in passing):
  each (token, head) row of d values is stored as FP8 E4M3 codes with one
  fp32 scale, s = amax(|row|) / 448 and code = E4M3 round-to-nearest-even of
  x / s (both divisions in IEEE fp32); decoding multiplies the code's value by
  s in fp32 and rounds to bf16 for the attention buffer.  A row of zeros has
  s = 0 and codes 0.
  The NVFP4 form of the tier (FP4 E2M1 values with E4M3 scales per 16-element
  block, the format the pages' "FP4" storage points to) keeps per row an fp32
  scale g = amax(|row|) / 2688 (2688 = 6 * 448), per block of 16 an E4M3
  scale sb = E4M3 RNE of amax(|block|) / (6 g), and per element the E2M1
  round-to-nearest-even (saturating at 6) of x / (sb * g); every product and
  quotient is one IEEE fp32 operation, in that order.  Decoding multiplies the
  E2M1 value by sb * g in fp32 and rounds to bf16.  Codes pack two elements per
  byte, the even element in the low nibble.
* HSA sparse branch ([WA] HSA section and its appendix notes): key blocks of
  B_inter = 128 tokens over the retrieved buffer and B_intra = 64 over the
  chunk's own tokens (a ragged last block keeps its own size); query blocks of
  B_intra = 64.  The pooled attention map of head h is the softmax over key
  blocks of scale * Qbar_qb . Kbar_kb (block means), one row per query block;
  the head's block mass is that map averaged over query blocks.  Selection is
  per head (the same block set for every query of the head): blocks ordered by
  mass (ties to the lower block index), the minimal prefix whose cumulative
  mass reaches tau_h.  The Gini-to-threshold formula is missing on the page;
  read as tau_h = 1 - G_h with G_h the Gini coefficient of the head's block
  mass (a uniform head keeps every block, a peaked head few), unless the
  caller passes tau_h.  The branch output is softmax attention restricted to
  the selected blocks' tokens.

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
    "block_bounds",
    "block_means",
    "key_blocks",
    "pooled_mass",
    "gini",
    "sparse_select",
    "sparse_attn",
    "page_scores_per_head",
    "select_pages_per_head",
    "gather_pages_per_head",
    "e4m3_values",
    "e4m3_round",
    "fp8_encode_rows",
    "fp8_decode_rows",
    "e2m1_values",
    "e2m1_round",
    "nvfp4_encode_rows",
    "nvfp4_decode_rows",
    "bf16_bits",
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


# ----------------------------------------------------------------------------
# [WA] HSA: sparse branch (pooled block map, Gini-adaptive block selection,
# attention restricted to the selected blocks)
# ----------------------------------------------------------------------------

def block_bounds(n: int, block: int):
    """Rows [start, end) of the blocks of ``block`` rows over n rows; the last
    block is ragged when block does not divide n."""
    return [(s, min(n, s + block)) for s in range(0, n, block)]


def block_means(x, block: int) -> np.ndarray:
    """Mean of each block of rows: x [n][H][d] -> [n_blocks][H][d] (fp64),
    a ragged last block divided by its own row count."""
    xx = as_f64(x)
    return np.stack([xx[a:b].sum(axis=0) / (b - a) for a, b in block_bounds(len(xx), block)],
                    axis=0)


def key_blocks(n_main: int, n_loc: int, b_inter: int = 128, b_intra: int = 64):
    """Key blocks in index order: the retrieved buffer in blocks of B_inter,
    then the chunk's own tokens in blocks of B_intra.  Each entry is
    (segment, start, end) with segment 0 = buffer, 1 = local."""
    out = [(0, a, b) for a, b in block_bounds(n_main, b_inter)]
    out += [(1, a, b) for a, b in block_bounds(n_loc, b_intra)]
    return out


def pooled_mass(q, k_main, k_loc, scale: float | None = None, b_q: int = 64,
                b_inter: int = 128, b_intra: int = 64) -> np.ndarray:
    """Block mass of each head: mass[h][kb] = mean over query blocks qb of
    softmax_kb(scale * Qbar_qb,h . Kbar_kb,h), the pooled attention map of the
    HSA sparse branch.  Returns [H][n_kb] (each row sums to 1)."""
    qq = as_f64(q)
    d = qq.shape[2]
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(d)
    qbar = block_means(qq, b_q)
    parts = []
    if k_main is not None and len(k_main) > 0:
        parts.append(block_means(k_main, b_inter))
    if k_loc is not None and len(k_loc) > 0:
        parts.append(block_means(k_loc, b_intra))
    kbar = np.concatenate(parts, axis=0)
    n_h = qq.shape[1]
    mass = np.empty((n_h, kbar.shape[0]), dtype=np.float64)
    for h in range(n_h):
        _, _, a = attention_rows(qbar[:, h, :], kbar[:, h, :], kbar[:, h, :], scale)
        mass[h] = a.mean(axis=0)
    return mass


def gini(m) -> float:
    """Gini coefficient of a non-negative vector (sorted-rank form):
    G = sum_i (2 i - n - 1) x_(i) / (n sum x), x_(1) <= ... <= x_(n)."""
    x = np.sort(np.asarray(m, dtype=np.float64))
    n = len(x)
    tot = x.sum()
    if n == 0 or tot == 0.0:
        return 0.0
    i = np.arange(1, n + 1, dtype=np.float64)
    return float(((2.0 * i - n - 1.0) * x).sum() / (n * tot))


def sparse_select(mass: np.ndarray, tau=None):
    """Per head: G_h = gini(mass[h]); tau_h = 1 - G_h unless given; blocks in
    order of mass (descending, ties to the lower index); the minimal prefix
    whose cumulative mass reaches tau_h (at least one block).  Returns
    (list of ascending block-index arrays per head, G [H], tau [H])."""
    n_h, n_kb = mass.shape
    sel, g_all, t_all = [], np.empty(n_h), np.empty(n_h)
    for h in range(n_h):
        g = gini(mass[h])
        t = (1.0 - g) if tau is None else float(tau[h])
        order = sorted(range(n_kb), key=lambda b: (-mass[h][b], b))
        acc, k = 0.0, 0
        for b in order:
            acc += mass[h][b]
            k += 1
            if acc >= t:
                break
        sel.append(np.array(sorted(order[:k]), dtype=np.int32))
        g_all[h], t_all[h] = g, t
    return sel, g_all, t_all


def sparse_attn(q, k_main, v_main, k_loc, v_loc, sel, scale: float | None = None,
                rows=None, b_inter: int = 128, b_intra: int = 64):
    """Attention of the chunk's queries restricted, per head, to the tokens of
    the selected key blocks (ascending block order).  sel: per-head arrays of
    block indices into key_blocks(n_main, n_loc).  Returns O [len(rows)][H][d]."""
    qq = as_f64(q)
    n_q, n_h, d = qq.shape
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(d)
    n_main = 0 if k_main is None else len(k_main)
    n_loc = 0 if k_loc is None else len(k_loc)
    blocks = key_blocks(n_main, n_loc, b_inter, b_intra)
    rows = np.arange(n_q) if rows is None else np.asarray(rows)
    out = np.empty((len(rows), n_h, d), dtype=np.float64)
    for h in range(n_h):
        ks, vs = [], []
        for b in sel[h]:
            seg, a, e = blocks[int(b)]
            src_k, src_v = (k_main, v_main) if seg == 0 else (k_loc, v_loc)
            ks.append(as_f64(src_k[a:e, h, :]))
            vs.append(as_f64(src_v[a:e, h, :]))
        oh, _, _ = attention_rows(qq[rows, h, :], np.concatenate(ks), np.concatenate(vs), scale)
        out[:, h, :] = oh
    return out


# ----------------------------------------------------------------------------
# [WA] HKV page stage, one page set per head
# ----------------------------------------------------------------------------

def page_scores_per_head(qbar: np.ndarray, kbar: np.ndarray, pages, head_dim: int) -> np.ndarray:
    """alpha[h][c] = Qbar_h . Kbar_{j_c,h} / sqrt(d_k) for the candidates j_c."""
    qb = as_f64(qbar)
    kb = as_f64(kbar)
    return np.array([[float(np.dot(qb[h], kb[j, h])) / math.sqrt(head_dim) for j in pages]
                     for h in range(qb.shape[0])], dtype=np.float64)


def select_pages_per_head(q, kbar, prompt_cur, prompt_chunks, pages_per_chunk: int, k_p: int):
    """Shared prompt stage, then each head's top-K_p candidates by its own
    score (ties to the lowest page index, ascending).  Returns (idx [H][k_p],
    alpha_of_idx [H][k_p], chunk)."""
    kb = as_f64(kbar)
    n_pages, n_h, d = kb.shape
    qbar = mean_query(q)
    if prompt_chunks is None or len(prompt_chunks) == 0:
        chunk = -1
    else:
        chunk = prompt_top1(prompt_cur, prompt_chunks)
    cand = candidate_pages(n_pages, chunk, pages_per_chunk)
    alpha = page_scores_per_head(qbar, kb, cand, d)
    idx = np.empty((n_h, k_p), dtype=np.int32)
    sc = np.empty((n_h, k_p), dtype=np.float64)
    for h in range(n_h):
        idx[h], sc[h] = topk_pages(alpha[h], cand, k_p)
    return idx, sc, chunk


def gather_pages_per_head(pages: np.ndarray, idx) -> np.ndarray:
    """buf[s*P + t][h] = pages[idx[h][s]][t][h]: a byte copy per head slice."""
    pg = np.asarray(pages)
    idx = np.asarray(idx)
    n_h, k_p = idx.shape
    p_tok = pg.shape[1]
    out = np.empty((k_p * p_tok,) + pg.shape[2:], dtype=pg.dtype)
    for h in range(n_h):
        for s_ in range(k_p):
            out[s_ * p_tok:(s_ + 1) * p_tok, h] = pg[int(idx[h, s_]), :, h]
    return out


# ----------------------------------------------------------------------------
# Compressed DRAM tier: FP8 E4M3 page codec with one fp32 scale per row
# ----------------------------------------------------------------------------

def e4m3_values() -> np.ndarray:
    """Value of each of the 256 E4M3 codes (sign bit, 4 exponent bits with
    bias 7, 3 mantissa bits; exponent 0 is subnormal; S.1111.111 is NaN; no
    infinities).  Returns float64 [256]."""
    out = np.empty(256, dtype=np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            out[c] = np.nan
        elif e == 0:
            out[c] = sign * (m / 8.0) * 2.0 ** -6
        else:
            out[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


def e4m3_round(q: np.ndarray) -> np.ndarray:
    """E4M3 code of each fp32 value by round-to-nearest, ties to the even code
    (mantissa LSB 0), the sign kept (also for a zero result); values in
    (448, 464) round to 448, larger ones are rejected.  Returns uint8 codes."""
    q = np.asarray(q, dtype=np.float64)
    vals = e4m3_values()
    pos = np.arange(0, 0x7F)                      # codes 0x00 .. 0x7E, increasing values
    pv = vals[pos]
    a = np.abs(q)
    if np.any(a >= 464.0):                       # 464 would round past the largest finite
        raise ValueError("value outside the E4M3 range")
    hi = np.searchsorted(pv, a, side="left")      # first value >= a
    hi = np.minimum(hi, len(pv) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - pv[lo], pv[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((pos[hi] & 1) == 0) & (hi != lo))
    code = np.where(take_hi, pos[hi], pos[lo]).astype(np.uint8)
    code = np.where(pv[hi] == a, pos[hi], code).astype(np.uint8)
    sign = np.signbit(q).astype(np.uint8) << 7    # IEEE: the sign survives a zero result
    return code | sign


def fp8_encode_rows(x):
    """x [n][H][d] (bf16 bits or float) -> (codes uint8 [n][H][d], scales
    float32 [n][H]): s = fp32(amax / 448), codes = E4M3 RNE of fp32(x / s)."""
    xx = as_f64(x).astype(np.float32)             # exact: bf16 values are fp32 values
    amax = np.abs(xx).max(axis=2)
    s = (amax / np.float32(448.0)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = (xx / safe[:, :, None]).astype(np.float32)
    codes = e4m3_round(q)
    codes[s == 0] = 0
    return codes, s


def fp8_decode_rows(codes, scales) -> np.ndarray:
    """fp32(value(code) * s) per element: [n][H][d] float32."""
    v = e4m3_values()[np.asarray(codes)].astype(np.float32)
    return (v * np.asarray(scales, dtype=np.float32)[:, :, None]).astype(np.float32)


def bf16_bits(x) -> np.ndarray:
    """bf16 bit patterns of fp32 values, round to nearest even (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = u + 0x7FFF + ((u >> 16) & 1)
    return (rounded >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------
# Compressed DRAM tier, NVFP4 form: E2M1 codes, E4M3 scales per 16 elements,
# one fp32 scale per row
# ----------------------------------------------------------------------------

E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_values() -> np.ndarray:
    """Value of each of the 16 E2M1 codes: sign bit 3, then 2 exponent bits
    (bias 1) and 1 mantissa bit; exponent 0 is subnormal (0 and 0.5).  Built
    from the field definitions, returns float64 [16]."""
    out = np.empty(16, dtype=np.float64)
    for c in range(16):
        sign = -1.0 if c & 0x8 else 1.0
        e = (c >> 1) & 0x3
        m = c & 0x1
        mag = (m / 2.0) if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
        out[c] = sign * mag
    return out


def e2m1_round(q: np.ndarray) -> np.ndarray:
    """E2M1 code (0..15) of each fp32 value: round to nearest, ties to the even
    code (mantissa bit 0), magnitudes above 6 saturate to 6, the sign kept (also
    for a zero result).  Returns uint8 codes."""
    q = np.asarray(q, dtype=np.float64)
    mags = np.array(E2M1_MAGNITUDES)
    a = np.minimum(np.abs(q), 6.0)
    hi = np.minimum(np.searchsorted(mags, a, side="left"), 7)   # first magnitude >= a
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - mags[lo], mags[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(a == mags[hi], hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    neg = (q < 0) | ((q == 0) & np.signbit(q))
    return (code | np.where(neg, 8, 0)).astype(np.uint8)


def nvfp4_encode_rows(x):
    """x [n][H][d] (bf16 bits or float, d a multiple of 16) -> (codes uint8
    [n][H][d/2], two per byte with the even element low; block scales uint8
    (E4M3 codes) [n][H][d/16]; row scales float32 [n][H])."""
    xx = as_f64(x).astype(np.float32)                     # exact for bf16 inputs
    n, h, d = xx.shape
    f32 = np.float32
    g = (np.abs(xx).max(axis=2) / f32(2688.0)).astype(f32)          # row scale
    blocks = xx.reshape(n, h, d // 16, 16)
    bamax = np.abs(blocks).max(axis=3)
    den = (g * f32(6.0)).astype(f32)
    safe_den = np.where(den > 0, den, f32(1.0)).astype(f32)
    sb_val = (bamax / safe_den[:, :, None]).astype(f32)
    sb = e4m3_round(np.where(den[:, :, None] > 0, sb_val, f32(0.0)))
    es = (e4m3_values()[sb].astype(f32) * g[:, :, None]).astype(f32)  # element scale per block
    safe_es = np.where(es > 0, es, f32(1.0)).astype(f32)
    q = (blocks / safe_es[:, :, :, None]).astype(f32)
    c = e2m1_round(q)
    c[np.broadcast_to((es <= 0)[:, :, :, None], c.shape)] = 0
    c = c.reshape(n, h, d)
    codes = (c[:, :, 0::2] | (c[:, :, 1::2] << 4)).astype(np.uint8)
    return codes, sb.astype(np.uint8), g


def nvfp4_decode_rows(codes, bscales, rscales) -> np.ndarray:
    """fp32( value(code) * fp32(value(sb) * g) ) per element: [n][H][d] float32."""
    codes = np.asarray(codes, dtype=np.uint8)
    n, h, half = codes.shape
    d = 2 * half
    c = np.empty((n, h, d), dtype=np.uint8)
    c[:, :, 0::2] = codes & 0x0F
    c[:, :, 1::2] = codes >> 4
    f32 = np.float32
    es = (e4m3_values()[np.asarray(bscales)].astype(f32)
          * np.asarray(rscales, dtype=f32)[:, :, None]).astype(f32)
    v = e2m1_values()[c].astype(f32).reshape(n, h, d // 16, 16)
    return (v * es[:, :, :, None]).astype(f32).reshape(n, h, d)
